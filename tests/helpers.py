"""Shared test helpers: move synthetic inputs to the GPU and compute oracle references."""

import numpy as np

from oracle import escha_oracle as O

REL_L2_TOL = 2e-3   # layer outputs vs the fp64 oracle


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def worst_rel_l2(a, b):
    """The larger of the whole-output relative L2 error and the worst single
    token's (row's): a wrong token or block cannot hide in the whole-output norm."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = rel_l2(a, b)
    if a.ndim == 2 and a.shape[0] > 1:
        err = max(err, max(rel_l2(a[r], b[r]) for r in range(a.shape[0])))
    return err


def cuda_layer(layer):
    import torch
    d = {}
    for k in ("code", "rin", "rout", "s_in", "s_out"):
        d[k] = torch.from_numpy(layer[k]).cuda()
    d["config"] = torch.from_numpy(layer["config"])
    return d


def make_linear_handle(layer, config_on_device=False):
    from gemm_trellis_tile_gb300 import escha
    d = cuda_layer(layer)
    cfg = d["config"].cuda() if config_on_device else d["config"]
    return escha.Linear(d["code"], d["rin"], d["rout"], d["s_in"], d["s_out"], cfg), d


def oracle_scales(layer):
    return O.fold_scales(layer["rin"], layer["s_in"]), O.fold_scales(layer["rout"], layer["s_out"])


def oracle_linear(layer, x, w=None, rounding="fp16"):
    if w is None:
        w = O.decode_matrix(layer["code"], layer["bits"], rounding=rounding)
    su, sv = oracle_scales(layer)
    return O.linear_forward(x, w, su, sv)


def oracle_layer_dict(layer, w=None, rounding="fp16"):
    if w is None:
        w = O.decode_matrix(layer["code"], layer["bits"], rounding=rounding)
    su, sv = oracle_scales(layer)
    return dict(w=w, su=su, sv=sv)
