"""The allocation-free entry point escha_linear_gemv_noalloc, through the C ABI.

It serves callers that must not allocate device memory (runtimes that own all
device memory in a pool reserved up front, or code running where a cudaMalloc
would synchronise the device or is not allowed).  These tests check that it
gives the same output as the handle-based escha_linear_gemv, within the
tolerance the other tests use, on two calls in a row with different layers
(so stale scratch from the first call cannot leak into the second), and that a
layer too large for its fixed scratch is refused before anything is launched.

This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from tests.helpers import (REL_L2_TOL, cuda_layer, make_linear_handle, oracle_linear,
                           worst_rel_l2)

torch = pytest.importorskip("torch")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, d, layer, x, y):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.escha_linear_gemv_noalloc(
        _p(d["code"]), _p(d["rin"]), _p(d["rout"]), _p(d["s_in"]), _p(d["s_out"]),
        layer["in_features"], layer["out_features"], layer["bits"], _p(x), _p(y), x.shape[0],
        stream)


def test_noalloc_rejects_bad_arguments_on_host():
    """Null pointers and out-of-range sizes are refused before any CUDA call."""
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    lib = escha.load()
    fake = ctypes.c_void_p(0x10000)
    assert lib.escha_linear_gemv_noalloc(None, fake, fake, None, None, 512, 512, 2,
                                         fake, fake, 1, None) == 1
    assert lib.escha_linear_gemv_noalloc(fake, fake, fake, None, None, 512, 512, 2,
                                         fake, fake, 17, None) == 1
    assert lib.escha_linear_gemv_noalloc(fake, fake, fake, None, None, 500, 512, 2,
                                         fake, fake, 1, None) == 2
    assert lib.escha_linear_gemv_noalloc(fake, fake, fake, None, None, 512, 512, 5,
                                         fake, fake, 1, None) == 2


@pytest.mark.gpu
def test_noalloc_matches_gemv_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    lib = escha.load()
    rng = np.random.default_rng(4242)
    cases = [(S.make_linear(rng, 1024, 1280, 3), 5), (S.make_linear(rng, 5120, 10240, 2), 16)]
    for layer, m in cases:
        d = cuda_layer(layer)
        x_np = S.make_activations(rng, m, layer["in_features"])
        x = torch.from_numpy(x_np).cuda()
        y = torch.empty((m, layer["out_features"]), dtype=torch.float16, device="cuda")
        assert _noalloc(lib, d, layer, x, y) == 0
        torch.cuda.synchronize()
        lin, _ = make_linear_handle(layer)
        y_ref = lin.gemv(x).cpu().numpy()
        got = y.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert worst_rel_l2(got, y_ref) <= REL_L2_TOL
        assert worst_rel_l2(got, oracle_linear(layer, x_np)) <= REL_L2_TOL
        lin.close()


@pytest.mark.gpu
def test_noalloc_refuses_layers_larger_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    lib = escha.load()
    # Real (small) buffers, declared shape far too large: refused on the host
    # from the size computation, before any launch reads the buffers.
    buf = torch.zeros(4096, dtype=torch.int16, device="cuda")
    out_features = 1 << 18
    assert ((4 * (128 + out_features) + 64 * 128 + 64 * out_features)
            > escha_scratch_bytes())
    st = lib.escha_linear_gemv_noalloc(_p(buf), _p(buf), _p(buf), None, None, 128, out_features,
                                       2, _p(buf), _p(buf), 1, None)
    assert st == 2
    # the entry point still works afterwards
    rng = np.random.default_rng(7)
    layer = S.make_linear(rng, 256, 384, 4)
    d = cuda_layer(layer)
    x_np = S.make_activations(rng, 2, 256)
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty((2, 384), dtype=torch.float16, device="cuda")
    assert _noalloc(lib, d, layer, x, y) == 0
    assert worst_rel_l2(y.cpu().numpy(), oracle_linear(layer, x_np)) <= REL_L2_TOL


_SYNC_DEBUG_NOALLOC = r"""
import ctypes, hashlib, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
from gemm_trellis_tile_gb300 import escha, synthetic as S
lib = escha.load()
rng = np.random.default_rng(77)
layer = S.make_linear(rng, 512, 768, 3)
d = {k: torch.from_numpy(layer[k]).cuda() for k in ("code", "rin", "rout", "s_in", "s_out")}
p = lambda t: ctypes.c_void_p(t.data_ptr())
out = b""
for m in (3, 16):
    x = torch.from_numpy(S.make_activations(rng, m, 512)).cuda()
    y = torch.empty((m, 768), dtype=torch.float16, device="cuda")
    st = lib.escha_linear_gemv_noalloc(p(d["code"]), p(d["rin"]), p(d["rout"]), p(d["s_in"]),
                                       p(d["s_out"]), 512, 768, 3, p(x), p(y), m,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st
    out += y.cpu().numpy().tobytes()
print(hashlib.sha256(out).hexdigest())
"""


@pytest.mark.gpu
def test_noalloc_sync_debug_mode_gives_the_same_results():
    """With ESCHA_SYNC_DEBUG=1 the entry point synchronises and reads its error
    word after each call; the results are the same bits as without it."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for flag in ("0", "1"):
        env = dict(os.environ, ESCHA_SYNC_DEBUG=flag)
        r = subprocess.run([sys.executable, "-c", _SYNC_DEBUG_NOALLOC, root], env=env,
                           capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip().splitlines()[-1])
    assert outs[0] == outs[1]


def escha_scratch_bytes():
    import re
    from gemm_trellis_tile_gb300 import escha
    text = open(escha.HEADER_PATH).read()
    m = re.search(r"#define ESCHA_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    return int(m.group(1)) * int(m.group(2)) * int(m.group(3))
