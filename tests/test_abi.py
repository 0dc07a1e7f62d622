"""The C-ABI library builds, loads, exports every declared symbol and validates
arguments on the host (no GPU needed: nothing here launches a kernel)."""

import ctypes

import pytest

from gemm_trellis_tile_gb300 import build, escha
from gemm_trellis_tile_gb300 import workloads as WL


@pytest.fixture(scope="module")
def lib():
    build.build()
    return escha.load()


def test_every_declared_function_is_exported(lib):
    names = escha.declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
        assert n in escha._SIGS, "binding lacks " + n


def test_status_strings(lib):
    for code in range(6):
        assert lib.escha_status_string(code)
    assert lib.escha_status_string(5) == b"device wait timed out"
    assert lib.escha_version() >= 100


def test_null_arguments_rejected_before_any_cuda_call(lib):
    h = ctypes.c_void_p()
    assert lib.escha_linear_create(None, None, None, None, None, None, None, 6, None) == 1
    assert lib.escha_linear_create(ctypes.byref(h), None, None, None, None, None, None, 6, None) == 1
    assert lib.escha_linear_gemv(None, None, None, 1, None) == 1
    assert lib.escha_linear_decode(None, None, None) == 1
    assert lib.escha_linear_destroy(None) == 1
    assert lib.escha_mlp_gemv(None, None, None, 1, None) == 1
    assert lib.escha_linear_set_rounding(None, 1) == 1
    assert lib.escha_moe_set_rounding(None, 0) == 1
    for s in (0, 1, 2, -1, 7):
        assert lib.escha_linear_gemv_stage(None, s, None, None, 1, None) == 1
        assert lib.escha_mlp_gemv_stage(None, s, None, None, 1, None) == 1
        assert lib.escha_linear_moe_gemv_stage(None, s, None, None, None, None, 1, 8, None) == 1
    assert lib.escha_mlp_create(ctypes.byref(h), None, None, None) == 1
    assert lib.escha_mlp_set_input_norm(None, None, ctypes.c_float(1e-6), 1) == 1
    assert lib.escha_moe_set_shared_expert(None, None, None, None, 2, None, None, None, None,
                                           None, None) == 1
    assert lib.escha_linear_check(None, None) == 1
    assert lib.escha_profile_enable(None, 0, 1) == 1
    assert lib.escha_selftest_wait_timeout(0, None) == 1
    assert lib.escha_selftest_wait_timeout(2000000, None) == 1
    fake = ctypes.c_void_p(0x10000)
    assert lib.escha_trellis_encode(None, 16, 16, 2, 0, fake, None, None) == 1
    assert lib.escha_trellis_encode(fake, 16, 16, 2, 0, None, None, None) == 1
    assert lib.escha_trellis_encode(fake, 0, 16, 2, 0, fake, None, None) == 1
    assert lib.escha_trellis_encode(fake, 24, 16, 2, 0, fake, None, None) == 2   # not whole tiles
    assert lib.escha_trellis_encode(fake, 16, 16, 5, 0, fake, None, None) == 2   # bits
    assert lib.escha_trellis_encode(fake, 16, 16, 2, 3, fake, None, None) == 1   # rounding
    assert lib.escha_linear_gemm_fp8(None, fake, fake, 1, None) == 1
    assert lib.escha_linear_gemm_fp8(fake, fake, fake, 0, None) == 1
    assert lib.escha_linear_gemm_fp8_codes(fake, None, fake, fake, 1, None) == 1
    assert lib.escha_linear_gemm_fp8_codes(fake, fake, fake, fake, 0, None) == 1
    assert lib.escha_linear_gemm_fp8_codes(fake, fake, ctypes.c_void_p(0x10002), fake, 1, None) == 1
    assert lib.escha_quantize_e4m3_rows(None, fake, fake, 1, 128, None) == 1
    assert lib.escha_quantize_e4m3_rows(fake, fake, fake, 0, 128, None) == 1
    for k in (0, 64, 200, 65536 + 128):                  # K: multiple of 128, at most 65536
        assert lib.escha_quantize_e4m3_rows(fake, fake, fake, 1, k, None) == 1, k
    odd = ctypes.c_void_p(0x10008)
    assert lib.escha_quantize_e4m3_rows(fake, odd, fake, 1, 128, None) == 1    # alignment


def test_bad_config_rejected_on_host(lib):
    """Config vectors are parsed on the host: wrong lengths and values never reach CUDA."""
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: config is checked first
    cfg_t = ctypes.c_int32 * 9

    def create(vals, n=None):
        arr = cfg_t(*(list(vals) + [0] * (9 - len(vals))))
        return lib.escha_linear_create(ctypes.byref(h), fake, fake, fake, None, None,
                                       ctypes.cast(arr, ctypes.c_void_p), n or len(vals), None)
    assert create([16, 2, 1, 1, 512, 512], 5) == 1          # bad length
    assert create([16, 5, 1, 1, 512, 512]) == 2             # bits outside {2,3,4}
    assert create([16, 2, 0, 1, 512, 512]) == 2             # cb != 1
    assert create([8, 2, 1, 1, 512, 512]) == 2              # tile != 16
    assert create([16, 2, 1, 1, 500, 512]) == 2             # in not a multiple of 128
    assert create([16, 2, 1, 1, 512, 0]) == 1               # empty output
    assert create([16, 32, 3, 1, 1, 512, 512, 512, 512]) == 2  # K does not match bits
    assert create([16, 2, 2, 1, 2, 512, 512, 512, 512]) == 2   # num_experts != 1
    assert create([16, 2, 2, 1, 1, 512, 512, 640, 512]) == 2   # padding unsupported
    misaligned = ctypes.c_void_p(0x10008)
    arr = cfg_t(16, 2, 1, 1, 512, 512)
    assert lib.escha_linear_create(ctypes.byref(h), misaligned, fake, fake, None, None,
                                   ctypes.cast(arr, ctypes.c_void_p), 6, None) == 1


def test_moe_halves_create_rejects_bad_arguments_on_host(lib):
    """escha_moe_create_halves: sizes, null tables and misaligned tables are
    rejected before any CUDA call (table entries live on the device and are
    checked there)."""
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)

    def create(E=4, hidden=256, inter=256, tabs=(fake, fake, fake), bits=(fake, fake, fake)):
        return lib.escha_moe_create_halves(ctypes.byref(h), E, hidden, inter, *tabs, *bits,
                                           fake, None, fake, None, fake, None, fake, None,
                                           fake, None, None)
    assert lib.escha_moe_create_halves(None, 4, 256, 256, *([fake] * 6), *([fake] * 10), None) == 1
    assert create(E=0) == 1
    assert create(E=5000) == 2
    assert create(inter=200) == 2
    assert create(hidden=320) == 2
    assert create(tabs=(fake, None, fake)) == 1
    assert create(bits=(fake, fake, None)) == 1
    assert create(tabs=(fake, odd, fake)) == 1        # pointer table not 8-byte aligned
    assert create(bits=(fake, ctypes.c_void_p(0x10002), fake)) == 1


def test_valid_config_without_gpu_fails_as_cuda_error(lib):
    """No GPU here: a well-formed create reaches the device query and reports a CUDA error."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x10000)
    arr = (ctypes.c_int32 * 6)(16, 2, 1, 1, 512, 512)
    assert lib.escha_linear_create(ctypes.byref(h), fake, fake, fake, None, None,
                                   ctypes.cast(arr, ctypes.c_void_p), 6, None) == 3
    assert lib.escha_selftest_wait_timeout(1000, None) == 3
    assert lib.escha_trellis_encode(fake, 16, 16, 2, 0, fake, None, None) == 3


def test_byte_accounting_matches_printed_layer_sizes():
    """EXLR8 page: 256 experts of 37,748,736 weights cost 2.42/3.62/4.83 GB at K2/3/4,
    and the home manifest (64 experts K4 + 192 K3) 3.93 GB per layer."""
    w = WL.moe_expert_weights(6144, 2048)
    assert w == 37748736
    for bits, gb in ((2, 2.42), (3, 3.62), (4, 4.83)):
        total = 256 * sum(WL.code_bytes(i, o, bits) for i, o in ((6144, 2048), (6144, 2048), (2048, 6144)))
        assert abs(total / 1e9 - gb) < 0.006
    home = sum(WL.code_bytes(i, o, b) * n for b, n in ((4, 64), (3, 192))
               for i, o in ((6144, 2048), (6144, 2048), (2048, 6144)))
    assert abs(home / 1e9 - 3.93) < 0.006
    assert WL.code_bytes(16, 16, 2) == 64 and WL.code_bytes(16, 16, 3) == 96
