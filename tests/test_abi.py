"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point include/w4a8.h declares, and rejects bad arguments on the
host before touching the GPU.  The product never imports the oracle."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a8.h")
PKG = os.path.join(ROOT, "bit_quantized_decode_gb300")


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_decode_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w4_repack", "a8_quantize", "w4a8_gemv", "q4_0_gemv", "i8g32_gemv", "w4a8_linear",
                     "q4_0_repack", "i8g32_repack", "w4_quantize_rows", "q4_0_quantize", "i8g32_quantize"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_the_header():
    from bit_quantized_decode_gb300 import _lib
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_library_is_built_for_sm_103a():
    """The build command targets compute_103a/sm_103a only."""
    from bit_quantized_decode_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-prec-div=true" in build.NVCC_FLAGS and "-ftz=false" in build.NVCC_FLAGS


def test_tuning_roundtrip_and_checks(lib):
    from bit_quantized_decode_gb300 import _lib
    for key in _lib.TUNE_KEYS:
        assert _lib.get_tuning(key) == 0
    _lib.set_tuning("max_stages", 4)
    assert _lib.get_tuning("max_stages") == 4
    _lib.set_tuning("max_stages", 0)
    assert lib.w4_set_tuning(0, 3) == 1          # blocks_per_sm must be 0, 1 or 2
    assert lib.w4_set_tuning(1, 1) == 1          # a ring needs two stages
    assert lib.w4_set_tuning(7, 0) == 1          # unknown key
    assert lib.w4_get_tuning(7) == -1
    assert lib.w4_set_tuning(6, 17) == 1         # tokens per group-format launch: at most 16
    _lib.set_tuning("group_launch_tokens", 16)
    assert _lib.get_tuning("group_launch_tokens") == 16
    _lib.set_tuning("group_launch_tokens", 0)
    assert lib.w4_set_tuning(4, 5000) == 1       # chain L2 lookahead: at most 4096 KB
    _lib.set_tuning("chain_prefetch_kb", 32)
    assert _lib.get_tuning("chain_prefetch_kb") == 32
    _lib.set_tuning("chain_prefetch_kb", 0)


def test_status_strings(lib):
    from bit_quantized_decode_gb300 import _lib
    for code, name in _lib.STATUS.items():
        assert _lib.status_str(code) == name
    assert _lib.version() == 1


def test_repacked_sizes(lib):
    from bit_quantized_decode_gb300 import _lib
    # 8-row tiles, 0.5 B per weight; Q4_0 adds 2 B per 32; i8g32 1 B + 2 B per 32
    assert _lib.w4_repacked_bytes(4608, 3584) == 4608 * 3584 // 2
    assert _lib.w4_repacked_bytes(13, 64) == 16 * 64 // 2
    assert _lib.q4_0_repacked_bytes(2560, 1536) == 2560 * 1536 * 18 // 32
    assert _lib.i8g32_repacked_bytes(262144, 1536) == 262144 * 1536 * 34 // 32
    assert _lib.w4_repacked_bytes(8, 48) == 0          # K % 32 != 0
    assert _lib.w4_repacked_bytes(-1, 64) == 0


FAKE = ctypes.c_void_p(0x1000)       # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x1004)        # 4-byte but not 16-byte aligned


def test_gemv_argument_checks_return_before_launch(lib):
    # M > 16
    assert lib.w4a8_gemv(FAKE, FAKE, None, FAKE, FAKE, 17, 8, 64, FAKE, None) == 2
    # K not a multiple of 32, K <= 0, K too large
    assert lib.w4a8_gemv(FAKE, FAKE, None, FAKE, FAKE, 1, 8, 48, FAKE, None) == 2
    assert lib.w4a8_gemv(FAKE, FAKE, None, FAKE, FAKE, 1, 8, 0, FAKE, None) == 1
    assert lib.w4a8_gemv(FAKE, FAKE, None, FAKE, FAKE, 1, 8, 131072 + 32, FAKE, None) == 2
    # negative sizes, null pointers
    assert lib.w4a8_gemv(FAKE, FAKE, None, FAKE, FAKE, -1, 8, 64, FAKE, None) == 1
    assert lib.w4a8_gemv(FAKE, FAKE, None, FAKE, FAKE, 1, -8, 64, FAKE, None) == 1
    assert lib.w4a8_gemv(None, FAKE, None, FAKE, FAKE, 1, 8, 64, FAKE, None) == 1
    assert lib.w4a8_gemv(FAKE, None, None, FAKE, FAKE, 1, 8, 64, FAKE, None) == 1
    assert lib.q4_0_gemv(FAKE, None, None, FAKE, 1, 8, 64, FAKE, None) == 1
    # misaligned weights / activations
    assert lib.w4a8_gemv(ODD, FAKE, None, FAKE, FAKE, 1, 8, 64, FAKE, None) == 3
    assert lib.i8g32_gemv(FAKE, None, ODD, FAKE, 1, 8, 64, FAKE, None) == 3
    # empty calls succeed without a launch
    assert lib.w4a8_gemv(None, None, None, None, None, 0, 8, 64, None, None) == 0
    assert lib.q4_0_gemv(None, None, None, None, 1, 0, 64, None, None) == 0


def test_linear_and_quantize_argument_checks(lib):
    assert lib.w4a8_linear(FAKE, FAKE, None, FAKE, 1, 8, 64, FAKE, FAKE, FAKE, 4, None) == 1   # unknown flag
    assert lib.w4a8_linear(FAKE, FAKE, None, None, 1, 8, 64, FAKE, FAKE, FAKE, 0, None) == 1   # no x
    assert lib.q4_0_linear(FAKE, None, ODD, 1, 8, 64, FAKE, FAKE, FAKE, 0, None) == 3
    assert lib.w4a8_linear(None, None, None, None, 0, 8, 64, None, None, None, 0, None) == 0
    assert lib.a8_quantize(FAKE, 1, 33, FAKE, FAKE, None) == 2
    assert lib.a8_quantize(None, 1, 64, FAKE, FAKE, None) == 1
    assert lib.a8_quantize(FAKE, 0, 64, FAKE, FAKE, None) == 0
    assert lib.w4_quantize_rows(FAKE, 4, 12, FAKE, FAKE, None) == 2
    assert lib.q4_0_quantize(FAKE, 4, 48, FAKE, None) == 2
    assert lib.i8g32_quantize(ODD, 4, 64, FAKE, FAKE, None) == 3


def test_repack_argument_checks(lib):
    from bit_quantized_decode_gb300 import _lib
    pp, keep = _lib._ptr_array([None])
    rows, keep2 = _lib._int_array([8])
    assert lib.w4_repack(pp, rows, 1, 64, FAKE, 1 << 20, None) == 1          # null shard
    pp2 = (ctypes.c_void_p * 1)(0x1000)
    ppc = ctypes.cast(pp2, _lib._PP)
    assert lib.w4_repack(ppc, rows, 1, 64, FAKE, 16, None) == 2              # output too small
    assert lib.w4_repack(ppc, rows, 0, 64, FAKE, 1 << 20, None) == 1         # no shards
    assert lib.w4_repack(ppc, rows, 9, 64, FAKE, 1 << 20, None) == 1         # too many shards
    assert lib.w4_repack(ppc, rows, 1, 64, ODD, 1 << 20, None) == 3
    neg, keep3 = _lib._int_array([-1])
    assert lib.w4_repack(ppc, neg, 1, 64, FAKE, 1 << 20, None) == 1
    assert lib.i8g32_repack(ppc, None, rows, 1, 64, FAKE, 1 << 20, None) == 1


def test_chain_argument_checks(lib):
    from bit_quantized_decode_gb300 import _lib
    d = (_lib.LinearDesc * 2)()
    for i in range(2):
        d[i] = _lib.LinearDesc(0x1000, 0x1000, None, 0x1000, 0x1000, None, None, 8, 64)
    ws = FAKE
    assert lib.w4_chain_workspace_bytes() >= 8
    assert lib.w4a8_linear_chain(d, 0, 1, ws, 256, None) == 0                    # empty chain
    assert lib.w4a8_linear_chain(d, 2, 0, ws, 256, None) == 0                    # no tokens
    assert lib.w4a8_linear_chain(d, 129, 1, ws, 256, None) == 2                  # chain too long
    assert lib.w4a8_linear_chain(d, 2, 17, ws, 256, None) == 2                   # M > 16
    assert lib.w4a8_linear_chain(d, 2, 1, None, 256, None) == 1                  # no workspace
    assert lib.w4a8_linear_chain(d, 2, 1, ws, 8, None) == 2                      # workspace too small
    assert lib.w4a8_linear_chain(d, 2, 1, ODD, 256, None) == 3                   # misaligned workspace
    d[1] = _lib.LinearDesc(0x1000, 0x1000, None, 0x1000, 0x1000, None, None, 8, 48)
    assert lib.w4a8_linear_chain(d, 2, 1, ws, 256, None) == 2                    # K % 32 != 0
    d[1] = _lib.LinearDesc(0x1000, None, None, 0x1000, 0x1000, None, None, 8, 64)
    assert lib.w4a8_linear_chain(d, 2, 1, ws, 256, None) == 1                    # no s_w
    d[1] = _lib.LinearDesc(0x1004, 0x1000, None, 0x1000, 0x1000, None, None, 8, 64)
    assert lib.w4a8_linear_chain(d, 2, 1, ws, 256, None) == 3                    # misaligned weights


def test_product_never_imports_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|from\s+\.\.?\s*import\s+oracle)|liboracle|oracle/",
                     re.M)
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f


def test_fusion_and_weight_only_argument_checks(lib):
    """The fused-operator and weight-only entry points reject bad arguments on
    the host, before any device query or launch."""
    from bit_quantized_decode_gb300 import _lib
    F = _lib.Fusion
    by = ctypes.byref
    args = (FAKE, FAKE, None, FAKE, 1, 8, 64, FAKE, FAKE, FAKE)
    bad_glu = F(None, 0.0, 3, None)
    assert lib.w4a8_linear_fused(*args, by(bad_glu), 0, None) == 1               # unknown GLU kind
    glu = F(None, 0.0, 1, None)
    assert lib.i8g32_linear_fused(FAKE, None, FAKE, 1, 8, 64, FAKE, FAKE, FAKE, by(glu), 0, None) == 2
    assert lib.q6g32_linear_fused(FAKE, None, FAKE, 1, 8, 64, FAKE, FAKE, FAKE, by(glu), 0, None) == 2
    no_eps = F(0x1000, 0.0, 0, None)
    assert lib.w4a8_linear_fused(*args, by(no_eps), 0, None) == 1                # RMSNorm needs eps > 0
    inf_eps = F(0x1000, float("inf"), 0, None)
    assert lib.w4a8_linear_fused(*args, by(inf_eps), 0, None) == 1
    odd_norm = F(0x1004, 1e-6, 0, None)
    assert lib.w4a8_linear_fused(*args, by(odd_norm), 0, None) == 3             # norm weight 16-B aligned
    odd_res = F(None, 0.0, 0, 0x1002)
    assert lib.w4a8_linear_fused(*args, by(odd_res), 0, None) == 3
    assert lib.w4a8_linear_fused(*args, by(glu), 2, None) == 1                   # unknown flag
    assert lib.w4a8_linear_fused(None, None, None, None, 0, 8, 64, None, None, None, None, 0, None) == 0
    # normalize + quantize, and the separate operators
    assert lib.rms_a8_quantize(FAKE, FAKE, 0.0, 1, 64, FAKE, FAKE, 0, None) == 1
    assert lib.rms_a8_quantize(FAKE, ODD, 1e-6, 1, 64, FAKE, FAKE, 0, None) == 3
    assert lib.rms_a8_quantize(FAKE, FAKE, 1e-6, 0, 64, None, None, 0, None) == 0
    assert lib.w4_rmsnorm(FAKE, FAKE, 1e-6, 1, 48, FAKE, 0, None) == 2
    assert lib.w4_rmsnorm(FAKE, FAKE, 1e-6, 1, 64, None, 0, None) == 1
    assert lib.w4_glu(FAKE, 0, 1, 8, FAKE, 0, None) == 1
    assert lib.w4_glu(FAKE, 1, 17, 8, FAKE, 0, None) == 2
    assert lib.w4_glu(None, 2, 1, 0, None, 0, None) == 0
    assert lib.w4_add(FAKE, FAKE, -1, FAKE, 0, None) == 1
    assert lib.w4_add(None, None, 0, None, 0, None) == 0
    # paired gate/up layout sizes and checks
    assert lib.w4_glu_repacked_bytes(3, 64) == 8 * 64 // 2
    assert lib.w4_glu_repacked_bytes(8, 64) == 16 * 64 // 2
    assert lib.q4_0_glu_repacked_bytes(5, 64) == 16 * 64 * 18 // 32
    assert lib.w4_glu_repacked_bytes(8, 48) == 0
    assert lib.w4_repack_glu(FAKE, None, 8, 64, FAKE, 1 << 20, None) == 1
    assert lib.w4_repack_glu(FAKE, FAKE, 8, 64, FAKE, 16, None) == 2
    assert lib.w4_repack_glu(FAKE, FAKE, 8, 64, ODD, 1 << 20, None) == 3
    assert lib.w4_repack_glu(FAKE, FAKE, 0, 64, None, 0, None) == 0
    # weight-only paths on float activations
    assert lib.w4a32_gemv(FAKE, FAKE, None, FAKE, 5, 8, 64, FAKE, 0, None) == 2  # at most four tokens
    assert lib.w8a32_gemv(FAKE, None, None, FAKE, 1, 8, 64, FAKE, 0, None) == 1
    assert lib.w8a32_gemv(FAKE, FAKE, None, ODD, 1, 8, 64, FAKE, 0, None) == 3
    assert lib.w4a32_gemv(None, None, None, None, 1, 0, 64, None, 0, None) == 0
    assert lib.w8_repacked_bytes(13, 64) == 16 * 64
    assert lib.w8_quantize_rows(FAKE, 4, 6, FAKE, FAKE, None) == 2
    assert lib.w8_quantize_rows(ODD, 4, 64, FAKE, FAKE, None) == 3


def test_noalloc_chain_checks_run_before_any_device_work(lib):
    """A bad descriptor is rejected before the scratch is looked up or
    cleared: without a GPU a CUDA call would fail with W4_ERR_CUDA (4), so
    the argument statuses here show that nothing reached the device."""
    from bit_quantized_decode_gb300 import _lib
    d = (_lib.LinearDesc * 2)()
    for i in range(2):
        d[i] = _lib.LinearDesc(0x1000, 0x1000, None, 0x1000, 0x1000, None, None, 8, 64)
    assert lib.w4a8_linear_chain_noalloc(d, 0, 1, None) == 0                   # empty chain
    assert lib.w4a8_linear_chain_noalloc(d, 129, 1, None) == 2
    d[1] = _lib.LinearDesc(0x1000, 0x1000, None, 0x1000, 0x1000, None, None, 8, 48)
    assert lib.w4a8_linear_chain_noalloc(d, 2, 1, None) == 2                   # K % 32 != 0
    d[1] = _lib.LinearDesc(0x1000, None, None, 0x1000, 0x1000, None, None, 8, 64)
    assert lib.w4a8_linear_chain_noalloc(d, 2, 1, None) == 1                   # no s_w
    d[1] = _lib.LinearDesc(0x1004, 0x1000, None, 0x1000, 0x1000, None, None, 8, 64)
    assert lib.w4a8_linear_chain_noalloc(d, 2, 1, None) == 3                   # misaligned weights


def test_workspace_query_and_error_word_alias(lib):
    for M, N, K in ((1, 512, 3584), (16, 152064, 3584), (4, 8, 32)):
        assert lib.w4_workspace_bytes(M, N, K) == 0
    assert hasattr(lib, "w4_last_device_error")
    assert lib.w4_last_device_error(None) == 1          # null output pointer, checked before any device call


def test_hbm_read_argument_checks(lib):
    assert lib.w4_hbm_read(FAKE, 1 << 20, None, None) == 1     # no sink
    assert lib.w4_hbm_read(None, 64, FAKE, None) == 1          # no buffer
    assert lib.w4_hbm_read(FAKE, 40, FAKE, None) == 2          # not a multiple of 16 bytes
    assert lib.w4_hbm_read(ODD, 64, FAKE, None) == 3
    assert lib.w4_hbm_read(FAKE, 64, ctypes.c_void_p(0x1002), None) == 3


def test_wait_selftest_argument_checks(lib):
    # checked on the host before any device work: no GPU is needed for these
    assert lib.w4_selftest_wait_timeout(2, 1000, None) == 1         # cluster is 0 or 1
    assert lib.w4_selftest_wait_timeout(0, 0, None) == 1            # a limit of at least 1 us
    assert lib.w4_selftest_wait_timeout(1, 1000001, None) == 1      # and at most one second


def test_host_quantizer_argument_checks(lib):
    assert lib.w4_quantize_rows_host(FAKE, 4, 12, FAKE, FAKE) == 2
    assert lib.w4_quantize_rows_host(FAKE, -1, 64, FAKE, FAKE) == 1
    assert lib.w4_quantize_rows_host(None, 4, 64, FAKE, FAKE) == 1
    assert lib.w4_quantize_rows_host(None, 0, 64, None, None) == 0
    assert lib.q4_0_quantize_host(FAKE, 4, 48, FAKE) == 2
    assert lib.q4_0_quantize_host(FAKE, 4, 64, None) == 1
    assert lib.i8g32_quantize_host(FAKE, 4, 0, FAKE, FAKE) == 1
    assert lib.i8g32_quantize_host(FAKE, 4, 64, FAKE, None) == 1
