"""Gated MLP with its input RMSNorm fused into the input rotations, through
the C ABI, against the CPU oracle: down(silu(gate(n)) * up(n)) with
n = rms_norm(x), the norm weight stored as escha stores it (w - 1), or
without the offset.  Outputs within relative L2 2e-3 of the fp64 oracle."""

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from oracle import escha_oracle as O
from tests.helpers import REL_L2_TOL, oracle_layer_dict, worst_rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()


def _mlp(seed, hidden, inter, bits=(2, 3, 3)):
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(seed)
    spec = S.make_mlp(rng, hidden, inter, *bits)
    layers = [escha.Linear.from_arrays(spec[k]) for k in ("gate", "up", "down")]
    return rng, spec, escha.MLP(*layers), layers


def _oracle(spec, x):
    return O.mlp_forward(x, oracle_layer_dict(spec["gate"]), oracle_layer_dict(spec["up"]),
                         oracle_layer_dict(spec["down"]))


@pytest.mark.parametrize("m,offset", [(1, True), (3, True), (16, True), (5, False)])
def test_mlp_input_norm_matches_oracle(m, offset):
    rng, spec, mlp, _ = _mlp(6000 + m, 384, 640)
    w = S.make_norm_weight(rng, 384)
    eps = 1e-6
    mlp.set_input_norm(torch.from_numpy(w).cuda(), eps, offset)
    x = S.make_activations(rng, m, 384) * np.float16(3.0)
    y = mlp.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    assert mlp.check() == 0
    ref = _oracle(spec, O.rms_norm(x, w, eps, stored_minus_one=offset))
    assert worst_rel_l2(y, ref) <= REL_L2_TOL


def test_mlp_input_norm_removed_restores_the_plain_mlp():
    rng, spec, mlp, _ = _mlp(6100, 256, 512)
    x = torch.from_numpy(S.make_activations(rng, 2, 256)).cuda()
    plain = mlp.gemv(x)
    mlp.set_input_norm(torch.from_numpy(S.make_norm_weight(rng, 256)).cuda())
    normed = mlp.gemv(x)
    mlp.set_input_norm(None)
    again = mlp.gemv(x)
    torch.cuda.synchronize()
    assert torch.equal(plain, again)
    assert not torch.equal(plain, normed)


def test_mlp_input_norm_full_width_stages_compose():
    """5120 -> 2048 -> 5120 (the 27B MLP's hidden width), M = 4: the staged
    call equals the full call bit for bit and matches the oracle."""
    from gemm_trellis_tile_gb300 import escha
    rng, spec, mlp, _ = _mlp(6200, 5120, 2048)
    w = S.make_norm_weight(rng, 5120)
    mlp.set_input_norm(torch.from_numpy(w).cuda(), 1e-6, True)
    x = S.make_activations(rng, 4, 5120)
    xt = torch.from_numpy(x).cuda()
    full = mlp.gemv(xt)
    staged = torch.empty_like(full)
    for s in range(escha.MLP.STAGES):
        mlp.gemv(xt, staged, stage=s)
    torch.cuda.synchronize()
    assert torch.equal(full, staged)
    ref = _oracle(spec, O.rms_norm(x, w, 1e-6))
    assert worst_rel_l2(full.cpu().numpy(), ref) <= REL_L2_TOL
