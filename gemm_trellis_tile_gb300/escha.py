"""Python binding of libescha (include/escha.h): argument marshalling only.

Every computation runs in the CUDA library; this module converts torch
tensors to device pointers and status codes to exceptions.  There is no CPU
fallback: if libescha.so is missing, loading fails loudly.

The raw C entry points are exposed under their C names (escha_linear_create,
escha_linear_gemv, ...) taking integer pointers; the classes Linear and MLP
wrap them for torch CUDA tensors.
"""

import ctypes
import os
import re

import numpy as np

from . import build as _build

ESCHA_OK = 0
STATUS_NAMES = {0: "ESCHA_OK", 1: "ESCHA_ERR_INVALID_ARG", 2: "ESCHA_ERR_UNSUPPORTED",
                3: "ESCHA_ERR_CUDA", 4: "ESCHA_ERR_OOM", 5: "ESCHA_ERR_TIMEOUT"}
KIND_LINEAR, KIND_MLP, KIND_MOE = 0, 1, 2

HEADER_PATH = os.path.join(os.path.dirname(_build.HERE), "include", "escha.h")


class EschaError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (what, STATUS_NAMES.get(status, "?"), status))


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
ROUNDING = {"fp16": 0, "e4m3": 1}   # ESCHA_ROUND_FP16, ESCHA_ROUND_E4M3

_SIGS = {
    "escha_status_string": (ctypes.c_char_p, [_I]),
    "escha_version": (_I, []),
    "escha_last_error_string": (ctypes.c_char_p, []),
    "escha_linear_create": (_I, [ctypes.POINTER(_P), _P, _P, _P, _P, _P, _P, _I, _P]),
    "escha_linear_destroy": (_I, [_P]),
    "escha_linear_shape": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "escha_linear_decode": (_I, [_P, _P, _P]),
    "escha_linear_gemv": (_I, [_P, _P, _P, _I, _P]),
    "escha_linear_gemv_stage": (_I, [_P, _I, _P, _P, _I, _P]),
    "escha_linear_gemm": (_I, [_P, _P, _P, _I, _P]),
    "escha_linear_reserve": (_I, [_P, _I]),
    "escha_mlp_create": (_I, [ctypes.POINTER(_P), _P, _P, _P]),
    "escha_mlp_destroy": (_I, [_P]),
    "escha_mlp_gemv": (_I, [_P, _P, _P, _I, _P]),
    "escha_mlp_gemv_stage": (_I, [_P, _I, _P, _P, _I, _P]),
    "escha_moe_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _P, _P, _P, _P,
                              _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "escha_moe_create_halves": (_I, [ctypes.POINTER(_P), _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                     _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "escha_moe_destroy": (_I, [_P]),
    "escha_moe_set_shared_expert": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P]),
    "escha_linear_moe_gemv": (_I, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "escha_linear_moe_gemv_stage": (_I, [_P, _I, _P, _P, _P, _P, _I, _I, _P]),
    "escha_linear_set_rounding": (_I, [_P, _I]),
    "escha_moe_set_rounding": (_I, [_P, _I]),
    "escha_linear_check": (_I, [_P, _P]),
    "escha_moe_check": (_I, [_P, _P]),
    "escha_mlp_check": (_I, [_P, _P]),
    "escha_mlp_set_input_norm": (_I, [_P, _P, ctypes.c_float, _I]),
    "escha_profile_enable": (_I, [_P, _I, _I]),
    "escha_profile_collect": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I)]),
    "escha_selftest_wait_timeout": (_I, [_I, _P]),
    "escha_trellis_encode": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "escha_linear_gemv_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _P]),
    "escha_linear_gemm_fp8": (_I, [_P, _P, _P, _I, _P]),
    "escha_quantize_e4m3_rows": (_I, [_P, _P, _P, _I, _I, _P]),
    "escha_linear_gemm_fp8_codes": (_I, [_P, _P, _P, _P, _I, _P]),
}


def lib_path():
    return _build.LIB_PATH


def load():
    """Load libescha.so (built in-tree by gemm_trellis_tile_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError("libescha.so is not built (%s); run gemm_trellis_tile_gb300.build.build()"
                           % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def declared_functions():
    """Names of the functions declared in include/escha.h."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(escha_[a-z0-9_]+)\s*\(", text)))


def check(status, what):
    if status != ESCHA_OK:
        detail = load().escha_last_error_string().decode() if status == 3 else ""
        raise EschaError(status, what + (" [%s]" % detail if detail else ""))


def __getattr__(name):
    # raw C entry points under their own names
    if name.startswith("escha_") and name in _SIGS:
        return getattr(load(), name)
    raise AttributeError(name)


# ---------------------------------------------------------------- torch wrappers

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, shape=None):
    """Validate a device tensor argument."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError("expected dtype %s, got %s" % (dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("expected shape %s, got %s" % (tuple(shape), tuple(t.shape)))
    return t


def _rows(t, width, what):
    """Row count of a [M, width] tensor; the kernels read whole rows of `width`
    elements, so any other shape is refused before it reaches them."""
    if t.dim() != 2 or t.shape[1] != width:
        raise ValueError("%s must be [M, %d], got %s" % (what, width, tuple(t.shape)))
    return t.shape[0]


def _out(y, m, width, device):
    """The caller's fp16 output [m, width], or a new one."""
    torch = _torch()
    if y is None:
        return torch.empty((m, width), dtype=torch.float16, device=device)
    return _dev(y, torch.float16, (m, width))


def _collect(handle, kind):
    ms = ctypes.c_double()
    n = _I()
    check(load().escha_profile_collect(handle, kind, ctypes.byref(ms), ctypes.byref(n)),
          "escha_profile_collect")
    return ms.value, n.value


class Linear:
    """Dense trellis-coded linear layer on the current CUDA device.

    Tensors: code int16 [in/16, out/16, 16*bits]; rin, rout fp16; s_in, s_out
    fp32 (optional); config int32 [6] or [9] (host or device tensor).  code must
    stay alive as long as the layer (it is borrowed, not copied).
    """

    def __init__(self, code, rin, rout, s_in=None, s_out=None, config=None, stream=None):
        torch = _torch()
        lib = load()
        if config is None:
            kt, nt, w = code.shape
            config = torch.tensor([16, w // 16, 1, 1, kt * 16, nt * 16], dtype=torch.int32)
        self._keep = (code, rin, rout, s_in, s_out, config)
        h = ctypes.c_void_p()
        cfg_ptr = ctypes.c_void_p(config.data_ptr())
        check(lib.escha_linear_create(ctypes.byref(h), _ptr(code), _ptr(rin), _ptr(rout), _ptr(s_in),
                                      _ptr(s_out), cfg_ptr, int(config.numel()), _stream(stream)),
              "escha_linear_create")
        self.handle = h
        a, b, c = _I(), _I(), _I()
        check(lib.escha_linear_shape(h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
              "escha_linear_shape")
        self.in_features, self.out_features, self.bits = a.value, b.value, c.value

    @classmethod
    def from_arrays(cls, layer, device="cuda"):
        """Build from host numpy arrays (code, rin, rout, s_in, s_out, config)."""
        torch = _torch()
        t = {k: torch.from_numpy(layer[k]).to(device) for k in ("code", "rin", "rout", "s_in", "s_out")}
        return cls(t["code"], t["rin"], t["rout"], t["s_in"], t["s_out"],
                   torch.from_numpy(layer["config"]))

    STAGES = 3

    def gemv(self, x, y=None, stream=None, stage=None):
        torch = _torch()
        _dev(x, torch.float16)
        m = _rows(x, self.in_features, "x")
        y = _out(y, m, self.out_features, x.device)
        if stage is None:
            check(load().escha_linear_gemv(self.handle, _ptr(x), _ptr(y), m, _stream(stream)),
                  "escha_linear_gemv")
        else:
            check(load().escha_linear_gemv_stage(self.handle, int(stage), _ptr(x), _ptr(y), m,
                                                 _stream(stream)), "escha_linear_gemv_stage")
        return y

    def gemm(self, x, y=None, stream=None):
        torch = _torch()
        _dev(x, torch.float16)
        m = _rows(x, self.in_features, "x")
        y = _out(y, m, self.out_features, x.device)
        check(load().escha_linear_gemm(self.handle, _ptr(x), _ptr(y), m, _stream(stream)),
              "escha_linear_gemm")
        return y

    def gemm_fp8(self, x, y=None, stream=None):
        """Prefill on FP8 tensor cores (E4M3-rounded handles): activations
        quantised per token to E4M3 (escha_linear_gemm_fp8)."""
        torch = _torch()
        _dev(x, torch.float16)
        m = _rows(x, self.in_features, "x")
        y = _out(y, m, self.out_features, x.device)
        check(load().escha_linear_gemm_fp8(self.handle, _ptr(x), _ptr(y), m, _stream(stream)),
              "escha_linear_gemm_fp8")
        return y

    def gemm_fp8_codes(self, q, d, y=None, stream=None):
        """The FP8 prefill's contraction on given E4M3 codes q (uint8 [M, in]) and
        per-row scales d (fp32 [M]) (escha_linear_gemm_fp8_codes)."""
        torch = _torch()
        _dev(q, torch.uint8)
        m = _rows(q, self.in_features, "q")
        _dev(d, torch.float32, (m,))
        y = _out(y, m, self.out_features, q.device)
        check(load().escha_linear_gemm_fp8_codes(self.handle, _ptr(q), _ptr(d), _ptr(y), m,
                                                 _stream(stream)), "escha_linear_gemm_fp8_codes")
        return y

    def reserve(self, max_m):
        check(load().escha_linear_reserve(self.handle, int(max_m)), "escha_linear_reserve")

    def set_rounding(self, rounding):
        """"fp16" (default) or "e4m3" (codebook values rounded to FP8 E4M3)."""
        check(load().escha_linear_set_rounding(self.handle, ROUNDING[rounding]),
              "escha_linear_set_rounding")

    def decode(self, stream=None):
        torch = _torch()
        w = torch.empty((self.in_features, self.out_features), dtype=torch.float16, device="cuda")
        check(load().escha_linear_decode(self.handle, _ptr(w), _stream(stream)), "escha_linear_decode")
        return w

    def check(self, stream=None):
        return load().escha_linear_check(self.handle, _stream(stream))

    def profile(self, on=True):
        check(load().escha_profile_enable(self.handle, KIND_LINEAR, int(on)), "escha_profile_enable")

    def collect(self):
        return _collect(self.handle, KIND_LINEAR)

    def close(self):
        if getattr(self, "handle", None):
            load().escha_linear_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MLP:
    """Gated MLP down(silu(gate x) * up x) over three Linear layers (borrowed)."""

    def __init__(self, gate, up, down):
        self._layers = (gate, up, down)
        h = ctypes.c_void_p()
        check(load().escha_mlp_create(ctypes.byref(h), gate.handle, up.handle, down.handle),
              "escha_mlp_create")
        self.handle = h
        self.hidden = gate.in_features

    STAGES = 5

    def gemv(self, x, y=None, stream=None, stage=None):
        torch = _torch()
        _dev(x, torch.float16)
        m = _rows(x, self.hidden, "x")
        y = _out(y, m, self.hidden, x.device)
        if stage is None:
            check(load().escha_mlp_gemv(self.handle, _ptr(x), _ptr(y), m, _stream(stream)),
                  "escha_mlp_gemv")
        else:
            check(load().escha_mlp_gemv_stage(self.handle, int(stage), _ptr(x), _ptr(y), m,
                                              _stream(stream)), "escha_mlp_gemv_stage")
        return y

    def set_input_norm(self, norm_w, eps=1e-6, stored_minus_one=True):
        """Input RMSNorm (weight as stored: fp16 CUDA tensor [in], or None to remove)."""
        torch = _torch()
        if norm_w is not None:
            _dev(norm_w, torch.float16, (self.hidden,))
        check(load().escha_mlp_set_input_norm(self.handle, _ptr(norm_w), float(eps),
                                              int(bool(stored_minus_one))),
              "escha_mlp_set_input_norm")
        self._norm = norm_w

    def check(self, stream=None):
        """The MLP's own device error flag (its launches), then the layers'."""
        st = load().escha_mlp_check(self.handle, _stream(stream))
        return st if st != 0 else max(layer.check(stream) for layer in self._layers)

    def profile(self, on=True):
        check(load().escha_profile_enable(self.handle, KIND_MLP, int(on)), "escha_profile_enable")

    def collect(self):
        return _collect(self.handle, KIND_MLP)

    def close(self):
        if getattr(self, "handle", None):
            load().escha_mlp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoE:
    """Routed-expert layer with one shared hidden-side rotation.

    gate_codes / up_codes / down_codes: lists of E int16 CUDA tensors (they may
    alias one another for experts that are never routed); bits: E widths.
    Side vectors are CUDA tensors: rin_hidden, rout_hidden fp16 [hidden];
    s_in_hidden, s_out_hidden fp32 [hidden]; rout_gate, rout_up, rin_down fp16
    [E, inter]; s_out_gate, s_out_up, s_in_down fp32 [E, inter].
    """

    def __init__(self, hidden, inter, gate_codes, up_codes, down_codes, bits, rin_hidden,
                 s_in_hidden, rout_gate, s_out_gate, rout_up, s_out_up, rin_down, s_in_down,
                 rout_hidden, s_out_hidden, stream=None):
        E = len(bits)
        self._keep = (gate_codes, up_codes, down_codes, rin_hidden, s_in_hidden, rout_gate,
                      s_out_gate, rout_up, s_out_up, rin_down, s_in_down, rout_hidden, s_out_hidden)
        ptrs = ctypes.c_void_p * E
        g = ptrs(*[t.data_ptr() for t in gate_codes])
        u = ptrs(*[t.data_ptr() for t in up_codes])
        d = ptrs(*[t.data_ptr() for t in down_codes])
        b = (ctypes.c_int32 * E)(*[int(v) for v in bits])
        self._tables = (g, u, d, b)
        h = ctypes.c_void_p()
        check(load().escha_moe_create(
            ctypes.byref(h), E, hidden, inter, ctypes.cast(g, _P), ctypes.cast(u, _P),
            ctypes.cast(d, _P), ctypes.cast(b, _P), _ptr(rin_hidden), _ptr(s_in_hidden),
            _ptr(rout_gate), _ptr(s_out_gate), _ptr(rout_up), _ptr(s_out_up), _ptr(rin_down),
            _ptr(s_in_down), _ptr(rout_hidden), _ptr(s_out_hidden), _stream(stream)),
            "escha_moe_create")
        self.handle = h
        self.hidden = hidden

    @classmethod
    def from_arrays(cls, spec, expert_codes, device="cuda"):
        """Build from host arrays: spec holds the side vectors and widths (see
        synthetic.make_moe_spec); expert_codes maps expert id -> (gate, up, down)
        int16 arrays.  Experts without codes point at one zero-filled stand-in
        buffer (never read unless routed to)."""
        torch = _torch()
        E, hidden, inter = spec["num_experts"], spec["hidden"], spec["inter"]
        dev = {e: tuple(torch.from_numpy(c).to(device) for c in codes)
               for e, codes in expert_codes.items()}
        stand_in = torch.zeros(hidden * inter // 2, dtype=torch.int16, device=device)
        gates = [dev[e][0] if e in dev else stand_in for e in range(E)]
        ups = [dev[e][1] if e in dev else stand_in for e in range(E)]
        downs = [dev[e][2] if e in dev else stand_in for e in range(E)]
        t = {k: torch.from_numpy(spec[k]).to(device) for k in (
            "rin_hidden", "s_in_hidden", "rout_gate", "s_out_gate", "rout_up", "s_out_up",
            "rin_down", "s_in_down", "rout_hidden", "s_out_hidden")}
        obj = cls(hidden, inter, gates, ups, downs, spec["bits"], t["rin_hidden"],
                  t["s_in_hidden"], t["rout_gate"], t["s_out_gate"], t["rout_up"], t["s_out_up"],
                  t["rin_down"], t["s_in_down"], t["rout_hidden"], t["s_out_hidden"])
        obj._keep_dev = (dev, stand_in, t)
        return obj

    STAGES = 5

    def gemv(self, x, expert_ids, expert_w, y=None, stream=None, stage=None):
        torch = _torch()
        _dev(x, torch.float16)
        m = _rows(x, self.hidden, "x")
        _dev(expert_ids, torch.int32)
        if expert_ids.dim() != 2 or expert_ids.shape[0] != m:
            raise ValueError("expert_ids must be [M, topk] with M = %d, got %s"
                             % (m, tuple(expert_ids.shape)))
        topk = expert_ids.shape[1]
        _dev(expert_w, torch.float32, (m, topk))
        y = _out(y, m, self.hidden, x.device)
        if stage is None:
            check(load().escha_linear_moe_gemv(self.handle, _ptr(x), _ptr(expert_ids),
                                               _ptr(expert_w), _ptr(y), m, topk, _stream(stream)),
                  "escha_linear_moe_gemv")
        else:
            check(load().escha_linear_moe_gemv_stage(self.handle, int(stage), _ptr(x),
                                                     _ptr(expert_ids), _ptr(expert_w), _ptr(y), m,
                                                     topk, _stream(stream)),
                  "escha_linear_moe_gemv_stage")
        return y

    def set_shared_expert(self, gate_code, up_code, down_code, bits, rout_gate, s_out_gate,
                          rout_up, s_out_up, rin_down, s_in_down):
        """Shared expert (CUDA tensors; codes borrowed), or gate_code=None to remove it."""
        if gate_code is None:
            check(load().escha_moe_set_shared_expert(self.handle, None, None, None, 0, None, None,
                                                     None, None, None, None),
                  "escha_moe_set_shared_expert")
            self._shared = None
            return
        self._shared = (gate_code, up_code, down_code)
        check(load().escha_moe_set_shared_expert(
            self.handle, _ptr(gate_code), _ptr(up_code), _ptr(down_code), int(bits),
            _ptr(rout_gate), _ptr(s_out_gate), _ptr(rout_up), _ptr(s_out_up), _ptr(rin_down),
            _ptr(s_in_down)), "escha_moe_set_shared_expert")

    def check(self, stream=None):
        return load().escha_moe_check(self.handle, _stream(stream))

    def set_rounding(self, rounding):
        """"fp16" (default) or "e4m3" (codebook values rounded to FP8 E4M3)."""
        check(load().escha_moe_set_rounding(self.handle, ROUNDING[rounding]),
              "escha_moe_set_rounding")

    def profile(self, on=True):
        check(load().escha_profile_enable(self.handle, KIND_MOE, int(on)), "escha_profile_enable")

    def collect(self):
        return _collect(self.handle, KIND_MOE)

    def close(self):
        if getattr(self, "handle", None):
            load().escha_moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoEHalves(MoE):
    """Routed-expert layer stored by halves of 128 intermediate channels, with
    per-half widths for gate/up and per-expert widths for down
    (escha_moe_create_halves).

    gate_half, up_half, down_half: int64 CUDA tensors [E, H] of device
    pointers (H = inter / 128); gate_bits, up_bits: int32 CUDA tensors [E, H];
    down_bits: int32 CUDA tensor [E].  The tables are borrowed and re-read by
    every call, so writing new pointers or widths into them (between calls)
    changes the layer.  Side vectors as for MoE.
    """

    def __init__(self, hidden, inter, gate_half, up_half, down_half, gate_bits, up_bits,
                 down_bits, rin_hidden, s_in_hidden, rout_gate, s_out_gate, rout_up, s_out_up,
                 rin_down, s_in_down, rout_hidden, s_out_hidden, stream=None):
        torch = _torch()
        E = gate_bits.shape[0]
        H = inter // 128
        for t in (gate_half, up_half, down_half):
            _dev(t, torch.int64, (E, H))
        _dev(gate_bits, torch.int32, (E, H))
        _dev(up_bits, torch.int32, (E, H))
        _dev(down_bits, torch.int32, (E,))
        self._keep = (gate_half, up_half, down_half, gate_bits, up_bits, down_bits, rin_hidden,
                      s_in_hidden, rout_gate, s_out_gate, rout_up, s_out_up, rin_down, s_in_down,
                      rout_hidden, s_out_hidden)
        h = ctypes.c_void_p()
        check(load().escha_moe_create_halves(
            ctypes.byref(h), E, hidden, inter, _ptr(gate_half), _ptr(up_half), _ptr(down_half),
            _ptr(gate_bits), _ptr(up_bits), _ptr(down_bits), _ptr(rin_hidden), _ptr(s_in_hidden),
            _ptr(rout_gate), _ptr(s_out_gate), _ptr(rout_up), _ptr(s_out_up), _ptr(rin_down),
            _ptr(s_in_down), _ptr(rout_hidden), _ptr(s_out_hidden), _stream(stream)),
            "escha_moe_create_halves")
        self.handle = h
        self.hidden = hidden
        self.tables = dict(gate_half=gate_half, up_half=up_half, down_half=down_half,
                           gate_bits=gate_bits, up_bits=up_bits, down_bits=down_bits)

    @classmethod
    def from_arrays(cls, spec, expert_codes, device="cuda"):
        """Build from host arrays: spec from synthetic.make_moe_half_spec;
        expert_codes maps expert id -> (gate halves, up halves, down halves),
        lists of int16 arrays.  Entries of experts without codes point at one
        zero-filled stand-in half (never read unless routed to)."""
        torch = _torch()
        E, hidden, inter, H = spec["num_experts"], spec["hidden"], spec["inter"], spec["halves"]
        dev = {e: tuple([torch.from_numpy(c).to(device) for c in part] for part in codes)
               for e, codes in expert_codes.items()}
        stand_in = torch.zeros(hidden * 64, dtype=torch.int16, device=device)
        tabs = []
        for part in range(3):
            ptrs = [[(dev[e][part][h] if e in dev else stand_in).data_ptr() for h in range(H)]
                    for e in range(E)]
            tabs.append(torch.tensor(ptrs, dtype=torch.int64, device=device))
        bits = [torch.from_numpy(np.ascontiguousarray(spec[k])).to(device)
                for k in ("gate_bits", "up_bits", "down_bits")]
        t = {k: torch.from_numpy(spec[k]).to(device) for k in (
            "rin_hidden", "s_in_hidden", "rout_gate", "s_out_gate", "rout_up", "s_out_up",
            "rin_down", "s_in_down", "rout_hidden", "s_out_hidden")}
        obj = cls(hidden, inter, tabs[0], tabs[1], tabs[2], bits[0], bits[1], bits[2],
                  t["rin_hidden"], t["s_in_hidden"], t["rout_gate"], t["s_out_gate"], t["rout_up"],
                  t["s_out_up"], t["rin_down"], t["s_in_down"], t["rout_hidden"],
                  t["s_out_hidden"])
        obj._keep_dev = (dev, stand_in, t)
        return obj


def selftest_wait_timeout(limit_us=10000, stream=None):
    """Run the bounded-wait self test; returns the status code (5 = timed out as designed)."""
    return load().escha_selftest_wait_timeout(int(limit_us), _stream(stream))


def quantize_e4m3_rows(xh, stream=None):
    """Per-token E4M3 codes and scales of fp16 activations xh [M, K] (CUDA):
    returns (q uint8 [M, K] E4M3 bit patterns, d fp32 [M]); xh ~ q * d."""
    torch = _torch()
    _dev(xh, torch.float16)
    if xh.dim() != 2:
        raise ValueError("xh must be [M, K], got %s" % (tuple(xh.shape),))
    m, k = xh.shape
    q = torch.empty((m, k), dtype=torch.uint8, device=xh.device)
    d = torch.empty((m,), dtype=torch.float32, device=xh.device)
    check(load().escha_quantize_e4m3_rows(_ptr(xh), _ptr(q), _ptr(d), int(m), int(k),
                                          _stream(stream)), "escha_quantize_e4m3_rows")
    return q, d


def trellis_encode(w, bits, rounding="fp16", sq_err=False, stream=None):
    """Code int16 [in/16, out/16, 16*bits] of W_inner w (fp32 [in, out], CUDA).

    Viterbi search per 16x16 tile with a tail-biting path (escha_trellis_encode).
    With sq_err=True also returns each tile's squared error, fp32 [in/16, out/16].
    """
    torch = _torch()
    _dev(w, torch.float32)
    if w.dim() != 2:
        raise ValueError("w must be [in, out], got %s" % (tuple(w.shape),))
    k, n = w.shape
    code = torch.empty((k // 16, n // 16, 16 * bits), dtype=torch.int16, device=w.device)
    err = torch.empty((k // 16, n // 16), dtype=torch.float32, device=w.device) if sq_err else None
    check(load().escha_trellis_encode(_ptr(w), int(k), int(n), int(bits), ROUNDING[rounding],
                                      _ptr(code), _ptr(err), _stream(stream)),
          "escha_trellis_encode")
    return (code, err) if sq_err else code
