"""Host-side logic of bench.py: replica aggregation over ranks (gloo, two
processes on the CPU), the algorithmic byte count of the step, and the
reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [3.0, 5.0][rank]                       # rank 1 is the slow one
    t = bench.max_over_ranks(elapsed, dist, "cpu")
    q.put((rank, t, bench.whole_job_gbs(1_000_000_000, 10, world, t)))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    assert [o[1] for o in out] == [5.0, 5.0]
    # 2 ranks x 10 steps x 1 GB in 5 ms
    assert out[0][2] == pytest.approx(2 * 10 * 1.0 / 0.005)


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.whole_job_gbs(10**9, 1, 1, 1000.0) == pytest.approx(1.0)


def test_step_bytes_match_the_step_definition():
    seq = bench.step_linears(28, True)
    assert len(seq) == 113
    weights = sum(l.N * l.K // 2 for _, l in seq)
    assert weights == 3_535_142_912
    total = sum(bench.algorithmic_bytes(l, 1) for _, l in seq)
    assert total == 3_556_995_072
    # one W4A8 row of the single-GEMV workload: 0.5 B per weight (1792 B at K = 3584)
    assert bench.algorithmic_bytes(bench.wl.workload("w4a8_single").linears[0], 1) == 937_984


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--ref-budget-s", "1"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_kernel_digest_does_not_depend_on_the_checkout_path(monkeypatch):
    """The profile summaries name the kernel sources by digest; the same
    sources in another directory (the GPU host's copy) give the same digest."""
    from bit_quantized_decode_gb300 import build
    here = build.kernel_digest()
    elsewhere = "/some/other/checkout/include"
    monkeypatch.setattr(build, "NVCC_FLAGS", [elsewhere if f == build.INCLUDE else f for f in build.NVCC_FLAGS])
    monkeypatch.setattr(build, "INCLUDE", elsewhere)
    assert build.kernel_digest() == here


def test_suite_gemv_selection():
    assert bench.suite_selected("", "lm_head", "lm_head_q6g32")
    assert bench.suite_selected("gemma_q4_0", "gemma_q4_0", "qkv")
    assert not bench.suite_selected("gemma_q4_0", "lm_head", "lm_head")
    assert bench.suite_selected("gemma_q4_0:down, lm_head:lm_head_q6g32", "lm_head", "lm_head_q6g32")
    assert not bench.suite_selected("lm_head:lm_head_q6g32", "lm_head", "lm_head_i8g32")


def test_suite_token_count_options():
    args = bench.parse_args(["--suite", "--suite-gemv-ms", "1,9,16", "--suite-ms", ""])
    assert args.suite and args.suite_gemv_ms == "1,9,16" and args.suite_ms == ""
    assert bench.parse_args([]).suite_gemv_ms == "1"      # single GEMVs at one token by default
