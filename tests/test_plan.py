"""The launch planner (w4_plan) on the host, without a GPU.

The expected grids, shared-memory sizes, stages and K splits are those of the
launches measured on a GB300 (ncu launch lists and -Xptxas/launch attributes of
the 7B decode step): the one-token DP4A GEMV at 115,712 B (98,176 B at
K = 18944) on 152 blocks, and the tensor-core GEMV at 114,920 B with clusters
of 4 for QKV and O and of 8 for down (its splits keep at least four K blocks,
so it fills both block slots of every SM), and 106,728 B for gate/up, whose K
is not split (no buffer for the other splits' sums).  The launch path takes its decisions through the same
functions, so these checks cover the host side of every GEMV launch.
"""
import math

import pytest

from bit_quantized_decode_gb300 import workloads as wl

# cudaDevAttrMultiProcessorCount, MaxSharedMemoryPerMultiprocessor,
# ReservedSharedMemoryPerBlock and MaxSharedMemoryPerBlockOptin of a GB300
GB300 = {"sms": 152, "smem_per_sm": 233472, "smem_reserved": 1024, "smem_optin": 232448}
HALF = GB300["smem_per_sm"] // 2 - GB300["smem_reserved"]


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_decode_gb300 import _lib, build
    build.build()
    _lib.load()
    yield _lib
    for k in _lib.TUNE_KEYS:
        _lib.set_tuning(k, 0)


def plan(lib, fmt, M, N, K, **kw):
    return lib.w4_plan(fmt, M, N, K, GB300, **kw)


def test_one_token_step_is_one_fused_launch_per_linear(lib):
    for lin in wl.qwen7b_layer():
        p = plan(lib, "w4", 1, lin.N, lin.K)
        assert p["path"] == "fused" and p["quantize_launches"] == 0
        assert p["grid"] == 152 and p["threads"] == 256 and p["k_splits"] == 1
        # two blocks per SM: the next linear's block is resident beside this one
        assert p["smem_bytes"] == (98176 if lin.K == 18944 else HALF)
        assert p["stages"] >= 2
    assert plan(lib, "w4", 1, 152064, 3584)["smem_bytes"] == HALF


def test_long_gemvs_take_both_block_slots(lib):
    # at least 64 tiles per SM and two blocks' worth of shared memory per SM:
    # the lm_heads at one and two tokens run on 2 x 152 blocks (measured faster
    # alone; two tokens then take the two-per-SM budget instead of the whole
    # SM); the layer linears keep one block per SM for the next linear's
    # prefetch, and three or more tokens keep the whole-SM ring
    for fmt, N, K in (("w4", 152064, 3584), ("i8g32", 262144, 1536), ("q6g32", 262144, 1536)):
        for M in (1, 2):
            p = plan(lib, fmt, M, N, K)
            assert p["grid"] == 304 and p["smem_bytes"] <= HALF
    for fmt in ("i8g32", "q6g32"):
        assert plan(lib, fmt, 3, 262144, 1536)["grid"] == 152
    # two tokens: two blocks per SM wherever the fused prologue fits half an
    # SM; the K = 18944 down projection keeps the fused prologue on the whole
    # SM (measured: the 7B step 1.25 ms so, 1.35 ms with down on the separate
    # quantizer and two blocks per SM, 1.37 ms with every linear on the whole SM)
    for lin in wl.qwen7b_layer():
        p = plan(lib, "w4", 2, lin.N, lin.K)
        assert p["path"] == "fused"
        if lin.K == 18944:
            assert p["grid"] == 152 and p["smem_bytes"] > HALF
        else:
            assert p["grid"] == 304 and p["smem_bytes"] <= HALF
    assert plan(lib, "w4", 1, 37888, 3584)["grid"] == 152
    lib.set_tuning("grid_blocks", 100)
    try:
        assert plan(lib, "w4", 1, 152064, 3584)["grid"] == 100  # the tuned cap wins
    finally:
        lib.set_tuning("grid_blocks", 0)


@pytest.mark.parametrize("name,grid,splits", [("qkv", 144, 4), ("o", 112, 4), ("gate_up", 296, 1), ("down", 224, 8)])
def test_sixteen_tokens_run_on_the_tensor_cores(lib, name, grid, splits):
    lin = {l.name: l for l in wl.qwen7b_layer()}[name]
    p = plan(lib, "w4", 16, lin.N, lin.K)
    assert p["path"] == "tensor_cores" and p["quantize_launches"] == 1
    smem = 114920 if splits > 1 else 106728
    assert (p["grid"], p["k_splits"], p["threads"], p["smem_bytes"], p["stages"]) == (grid, splits, 320, smem, 2)


def test_lm_head_and_largest_k_on_the_tensor_cores(lib):
    p = plan(lib, "w4", 16, 152064, 3584)
    assert (p["grid"], p["k_splits"]) == (1188, 1)
    p = plan(lib, "w4", 8, 128, 131072)          # eight splits of 16384 K
    assert (p["grid"], p["k_splits"]) == (8, 8)


def test_token_threshold_and_formats(lib):
    # measured: two tokens are faster on DP4A (1.39 against 1.43 ms per 7B step),
    # three and four on the tensor cores (1.46 / 1.49 against 1.80 / 2.05 ms)
    assert plan(lib, "w4", 2, 4608, 3584)["path"] == "fused"
    for M in (3, 4, 5, 6, 7):
        assert plan(lib, "w4", M, 4608, 3584)["path"] == "tensor_cores"
    for fmt in ("q4_0", "i8g32", "q6g32"):        # the tensor-core path is per-row INT4 only
        assert plan(lib, fmt, 16, 2560, 1536)["path"] != "tensor_cores"
    lib.set_tuning("tc_min_m", 17)
    try:
        p = plan(lib, "w4", 16, 3584, 18944)      # 16 x 18944 codes do not fit the fused prologue
        assert p["path"] in ("codes_smem", "codes_global") and p["quantize_launches"] == 1
    finally:
        lib.set_tuning("tc_min_m", 0)


def test_gemv_on_codes_and_gated_rows(lib):
    p = plan(lib, "w4", 1, 4608, 3584, linear=False)
    assert p["path"] in ("codes_smem", "codes_global") and p["quantize_launches"] == 0
    # a gated call of I outputs reads 8 ceil(I / 4) weight rows: gate/up of the 7B layer
    p = plan(lib, "w4", 16, 18944, 3584, glu=True)
    assert (p["grid"], p["k_splits"]) == (296, 1)
    assert plan(lib, "w4", 1, 18944, 3584, glu=True, norm=True)["path"] == "fused"


def test_norm_limits_the_fused_prologue(lib):
    # the norm keeps x in registers: at most four tokens in the fused prologue
    assert plan(lib, "q4_0", 4, 2560, 1536, norm=True)["path"] == "fused"
    p = plan(lib, "q4_0", 8, 2560, 1536, norm=True)
    assert p["path"] != "fused" and p["quantize_launches"] == 1


def test_group_formats_past_eight_tokens(lib):
    """Q4_0 / I8G32 / Q6G32 with more than eight tokens run as two GEMV
    launches of the eight-token kernel (tokens 0-7, then the rest), each
    planned as the eight-token call.  W4_TUNE_GROUP_LAUNCH_TOKENS = t makes
    launches of at most t tokens.  Per-row INT4 stays one launch (the tensor
    cores take any M)."""
    keys = ("path", "quantize_launches", "grid", "threads", "smem_bytes", "stages", "k_splits")
    for fmt, N, K in (("q4_0", 12288, 1536), ("q4_0", 1536, 6144), ("i8g32", 262144, 1536),
                      ("q6g32", 262144, 1536), ("q4_0", 77, 96), ("i8g32", 2560, 1536)):
        for linear in (True, False):
            p8 = plan(lib, fmt, 8, N, K, linear=linear)
            assert p8["gemv_launches"] == 1
            for M in (9, 10, 12, 13, 16):
                p = plan(lib, fmt, M, N, K, linear=linear)
                assert p["gemv_launches"] == 2, (fmt, M, N, K, linear)
                assert {k: p[k] for k in keys} == {k: p8[k] for k in keys}, (fmt, M, N, K, linear)
    assert plan(lib, "q4_0", 12, 2560, 1536, norm=True)["gemv_launches"] == 2
    assert plan(lib, "q4_0", 10, 2000, 1536, glu=True)["gemv_launches"] == 2
    for M in (1, 2, 4, 8):
        assert plan(lib, "i8g32", M, 262144, 1536)["gemv_launches"] == 1
    for M in (1, 9, 16):
        assert plan(lib, "w4", M, 4608, 3584)["gemv_launches"] == 1
    assert plan(lib, "q4_0", 0, 2560, 1536)["gemv_launches"] == 0
    assert plan(lib, "q4_0", 12, 0, 1536)["gemv_launches"] == 0
    lib.set_tuning("group_launch_tokens", 4)
    try:
        assert plan(lib, "q4_0", 16, 77, 96)["gemv_launches"] == 4
        assert plan(lib, "q6g32", 9, 262144, 1536)["gemv_launches"] == 3
        assert plan(lib, "q4_0", 4, 77, 96)["gemv_launches"] == 1
        assert plan(lib, "w4", 16, 77, 96)["gemv_launches"] == 1
    finally:
        lib.set_tuning("group_launch_tokens", 16)
    try:
        assert plan(lib, "i8g32", 16, 262144, 1536)["gemv_launches"] == 1
    finally:
        lib.set_tuning("group_launch_tokens", 0)


def test_empty_calls_and_tuning(lib):
    assert plan(lib, "w4", 0, 4608, 3584)["path"] == "none"
    p = plan(lib, "w4", 1, 0, 3584)
    assert p["path"] == "none" and p["quantize_launches"] == 1     # the linear still writes qx, sx
    assert plan(lib, "w4", 1, 0, 3584, linear=False)["quantize_launches"] == 0
    assert plan(lib, "w4", 1, 9, 3584)["grid"] == 2                # two 8-row tiles
    lib.set_tuning("grid_blocks", 76)
    try:
        assert plan(lib, "w4", 1, 4608, 3584)["grid"] == 76
    finally:
        lib.set_tuning("grid_blocks", 0)


def test_argument_errors(lib):
    from bit_quantized_decode_gb300 import _lib
    with pytest.raises(_lib.W4Error) as e:
        plan(lib, "i8g32", 1, 64, 1536, glu=True)
    assert e.value.status == 1
    with pytest.raises(_lib.W4Error) as e:
        plan(lib, "w4", 1, 64, 1536, linear=False, norm=True)
    assert e.value.status == 1
    with pytest.raises(_lib.W4Error) as e:
        lib.w4_plan("w4", 1, 64, 1536, dict(GB300, sms=0))
    assert e.value.status == 1
    for M, K in ((17, 1536), (1, 1537), (1, 131072 + 32)):
        with pytest.raises(_lib.W4Error) as e:
            plan(lib, "w4", M, 64, K)
        assert e.value.status == 2


def test_invariants_over_a_shape_sweep(lib):
    for M in (1, 2, 3, 4, 5, 8, 12, 16):
        for K in (32, 96, 1536, 3584, 6144, 16384, 16416, 18944, 40960, 131072):
            for N in (1, 8, 77, 300, 4608, 37888):
                p = plan(lib, "w4", M, N, K)
                if p["path"] == "tensor_cores":
                    ks = p["k_splits"]
                    C = K // 32
                    assert 1 <= ks <= 8 and ks <= C
                    assert math.ceil(C / ks) * 32 <= 16384        # every split's sums stay exact
                    assert ks & (ks - 1) == 0 or ks == math.ceil(K / 16384) or ks == C
                    assert p["grid"] == math.ceil(N / 128) * ks
                    assert p["smem_bytes"] <= HALF                  # two blocks per SM
                else:
                    assert p["path"] in ("fused", "codes_smem", "codes_global")
                    ks = p["k_splits"]                                # DP4A: clusters of ks blocks
                    assert ks in (1, 2, 4) and (ks == 1 or (M <= 2 and K // 32 // ks >= 16))
                    T = math.ceil(N / 8)
                    # two of the GEMV's own blocks per SM: two tokens, or one token and
                    # at least 64 tiles per SM, when two blocks fit an SM
                    two = ks == 1 and (M == 2 or (M == 1 and T >= 64 * 152)) and p["smem_bytes"] <= HALF
                    assert p["grid"] == min((304 if two else 152) // ks, T) * ks
                    assert 2 <= p["stages"] and p["smem_bytes"] <= GB300["smem_optin"]


def test_describe_device_without_a_gpu_is_an_error(lib):
    import torch

    from bit_quantized_decode_gb300 import _lib
    if torch.cuda.is_available():
        d = lib.w4_describe_device()
        assert d["sms"] > 0 and d["smem_optin"] > 0
    else:
        with pytest.raises(_lib.W4Error) as e:
            lib.w4_describe_device()
        assert e.value.status == 4


def test_k_splits_only_when_forced(lib):
    """DP4A GEMVs split K over a cluster only when W4_TUNE_K_SPLITS asks for it
    (a split measured slower on every shape tried, the few-tile GEMVs
    included), for one or two tokens and where every split keeps at least 16
    chunks; the grid is then a cluster per tile range."""
    for fmt, N, K in (("w4", 512, 3584), ("q4_0", 1536, 6144), ("q4_0", 2560, 1536), ("w4", 152064, 3584)):
        assert plan(lib, fmt, 1, N, K)["k_splits"] == 1
    lib.set_tuning("k_splits", 4)
    try:
        p = plan(lib, "w4", 1, 512, 3584)
        assert (p["k_splits"], p["grid"]) == (4, 38 * 4)
        assert plan(lib, "w4", 2, 4608, 3584)["k_splits"] == 4
        assert plan(lib, "q4_0", 3, 1536, 6144)["k_splits"] == 1     # three tokens' DP4A kernel: no split
        assert plan(lib, "w4", 1, 8, 64)["k_splits"] == 1            # two chunks: nothing to split
    finally:
        lib.set_tuning("k_splits", 0)
    assert lib.load().w4_set_tuning(5, 3) == 1                      # splits: 0, 1, 2, 4 or 8
