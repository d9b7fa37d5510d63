"""ctypes wrapper around the CPU oracle (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import
this package.  The CUDA library never does, and nothing here imports the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

from . import build as _build

ORC_TALKER, ORC_CODEC = 0, 1
INVALID_POS = 0xFFFFFFFF

_dp = C.POINTER(C.c_double)
_fp = C.POINTER(C.c_float)


class OrcConfig(C.Structure):
    _fields_ = [("kind", C.c_int), ("layers", C.c_int), ("hidden", C.c_int),
                ("q_heads", C.c_int), ("kv_heads", C.c_int), ("head_dim", C.c_int),
                ("inter", C.c_int), ("norm_eps", C.c_float), ("rope_theta", C.c_double),
                ("weight_bf16", C.c_int), ("max_pos", C.c_int), ("ring", C.c_int),
                ("window", C.c_int), ("streams", C.c_int)]


_LAYER_FIELDS = ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown",
                 "in_norm", "q_norm", "k_norm", "post_norm",
                 "in_proj", "out_proj", "lin1", "lin2",
                 "ln1_w", "ln1_b", "ln2_w", "ln2_b", "ls1", "ls2")


class OrcLayer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _LAYER_FIELDS]


_libs: Dict[str, C.CDLL] = {}


def lib(precision: str = "f32") -> C.CDLL:
    if precision not in _libs:
        path = _build.lib_path(precision)
        if not os.path.exists(path) or _build._stale(path):
            _build.build()
        L = C.CDLL(path)
        L.orc_bf16_to_f32.restype = C.c_float
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_matvec_f32.argtypes = [_fp, C.c_int, C.c_int, _dp, _dp]
        L.orc_matvec_bf16.argtypes = [C.POINTER(C.c_uint16), C.c_int, C.c_int, _dp, _dp]
        L.orc_rms_norm.argtypes = [_dp, _fp, C.c_int, C.c_double, _dp]
        L.orc_matvec_bias.argtypes = [_fp, C.c_int, C.c_int, _dp, _fp, C.c_int, _dp]
        L.orc_layer_norm.argtypes = [_dp, _fp, _fp, C.c_int, C.c_double, _dp]
        L.orc_rope_table.argtypes = [C.c_int, C.c_double, C.c_int, _dp, _dp]
        L.orc_mrope_table.argtypes = [C.c_int, C.c_double, C.POINTER(C.c_int),
                                      C.POINTER(C.c_int), _dp, _dp]
        L.orc_rope_rotate_half.argtypes = [_dp, C.c_int, _dp, _dp]
        L.orc_rope_interleaved.argtypes = [_dp, C.c_int, _dp, _dp]
        L.orc_silu.restype = C.c_double
        L.orc_silu.argtypes = [C.c_double]
        L.orc_gelu.restype = C.c_double
        L.orc_gelu.argtypes = [C.c_double]
        L.orc_gqa_attention.argtypes = [_dp, _dp, _dp, C.c_int, C.c_int, C.c_int, C.c_int, _dp]
        L.orc_ring_attention.argtypes = [_dp, _dp, _dp, C.POINTER(C.c_uint32), C.c_int,
                                         C.c_int, C.c_uint32, C.c_int, C.c_int, _dp]
        L.orc_create.restype = C.c_void_p
        L.orc_create.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcLayer), _fp]
        L.orc_prefill_kv.argtypes = [C.c_void_p, C.c_int, _fp, _fp, C.c_int]
        L.orc_step.argtypes = [C.c_void_p, C.c_int, _fp, C.POINTER(C.c_int), _dp, _dp]
        L.orc_prefill.argtypes = [C.c_void_p, C.c_int, C.c_int, _fp, _dp]
        _ip = C.POINTER(C.c_int)
        L.orc_set_mrope.argtypes = [C.c_void_p, _ip]
        L.orc_step_mrope.argtypes = [C.c_void_p, C.c_int, _fp, _ip, _ip, _dp, _dp]
        L.orc_prefill_mrope.argtypes = [C.c_void_p, C.c_int, C.c_int, _fp, _ip, _dp]
        L.orc_flow_step.argtypes = [C.c_void_p, _fp, _fp, _dp]
        L.orc_set_head.argtypes = [C.c_void_p, _fp, _fp, _fp]
        L.orc_eos.argtypes = [C.c_void_p, C.c_int]
        L.orc_eos.restype = C.c_double
        L.orc_reset.argtypes = [C.c_void_p, C.c_int]
        L.orc_len.argtypes = [C.c_void_p, C.c_int]
        L.orc_read_kv.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, _dp, _dp]
        L.orc_destroy.argtypes = [C.c_void_p]
        L.orc_set_threads.argtypes = [C.c_int]
        L.orc_get_threads.restype = C.c_int
        _libs[precision] = L
    return _libs[precision]


def _d(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(C.POINTER(ct))


# ---------------------------------------------------------------------------- primitives

def bf16_to_f32(bits: int, precision: str = "f32") -> float:
    return float(lib(precision).orc_bf16_to_f32(int(bits)))


def matvec(W: np.ndarray, x, precision: str = "f32") -> np.ndarray:
    """y = W x, W row-major [N][K] float32 or uint16 (bf16 bits)."""
    W = np.ascontiguousarray(W)
    N, K = W.shape
    x = _d(x)
    y = np.empty(N, np.float64)
    if W.dtype == np.uint16:
        lib(precision).orc_matvec_bf16(_ptr(W, C.c_uint16), N, K, _ptr(x, C.c_double),
                                       _ptr(y, C.c_double))
    else:
        W = np.ascontiguousarray(W, dtype=np.float32)
        lib(precision).orc_matvec_f32(_ptr(W, C.c_float), N, K, _ptr(x, C.c_double),
                                      _ptr(y, C.c_double))
    return y


def matvec_bias(W: np.ndarray, x, b, act: int = 0, precision: str = "f32") -> np.ndarray:
    """MV_BIAS (the flow head's linear): b[n] + sum_k W[n,k] x[k], accumulated from the bias in
    ascending k, then SiLU when act == 1.  W float32 [N][K]."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    N, K = W.shape
    x = _d(x)
    y = np.empty(N, np.float64)
    lib(precision).orc_matvec_bias(_ptr(W, C.c_float), N, K, _ptr(x, C.c_double),
                                   _ptr(b, C.c_float), int(act), _ptr(y, C.c_double))
    return y


def rms_norm(x, w, eps: float, precision: str = "f32") -> np.ndarray:
    x = _d(x)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = np.empty_like(x)
    lib(precision).orc_rms_norm(_ptr(x, C.c_double), _ptr(w, C.c_float), x.size, eps,
                                _ptr(y, C.c_double))
    return y


def layer_norm(x, w, b, eps: float, precision: str = "f32") -> np.ndarray:
    x = _d(x)
    w = np.ascontiguousarray(w, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    y = np.empty_like(x)
    lib(precision).orc_layer_norm(_ptr(x, C.c_double), _ptr(w, C.c_float), _ptr(b, C.c_float),
                                  x.size, eps, _ptr(y, C.c_double))
    return y


def rope_table(d: int, theta: float, pos: int, precision: str = "f32"):
    c = np.empty(d // 2, np.float64)
    s = np.empty(d // 2, np.float64)
    lib(precision).orc_rope_table(d, theta, pos, _ptr(c, C.c_double), _ptr(s, C.c_double))
    return c, s


def mrope_table(d: int, theta: float, pos3: Sequence[int], assign: Sequence[int],
                precision: str = "f32"):
    p = np.ascontiguousarray(pos3, dtype=np.int32)
    a = np.ascontiguousarray(assign, dtype=np.int32)
    c = np.empty(d // 2, np.float64)
    s = np.empty(d // 2, np.float64)
    lib(precision).orc_mrope_table(d, theta, _ptr(p, C.c_int), _ptr(a, C.c_int),
                                   _ptr(c, C.c_double), _ptr(s, C.c_double))
    return c, s


def rope_rotate_half(x, c, s, precision: str = "f32") -> np.ndarray:
    x = _d(x).copy()
    c, s = _d(c), _d(s)
    lib(precision).orc_rope_rotate_half(_ptr(x, C.c_double), x.size, _ptr(c, C.c_double),
                                        _ptr(s, C.c_double))
    return x


def rope_interleaved(x, c, s, precision: str = "f32") -> np.ndarray:
    x = _d(x).copy()
    c, s = _d(c), _d(s)
    lib(precision).orc_rope_interleaved(_ptr(x, C.c_double), x.size, _ptr(c, C.c_double),
                                        _ptr(s, C.c_double))
    return x


def silu(g: float, precision: str = "f32") -> float:
    return lib(precision).orc_silu(float(g))


def gelu(v: float, precision: str = "f32") -> float:
    return lib(precision).orc_gelu(float(v))


def gqa_attention(q, kc, vc, precision: str = "f32") -> np.ndarray:
    """q [H][d]; kc, vc [L][G][d] position-major -> out [H][d]."""
    q = _d(q)
    kc = _d(kc)
    vc = _d(vc)
    H, d = q.shape
    L, G, _ = kc.shape
    out = np.empty((H, d), np.float64)
    lib(precision).orc_gqa_attention(_ptr(q, C.c_double), _ptr(kc, C.c_double),
                                     _ptr(vc, C.c_double), L, H, G, d, _ptr(out, C.c_double))
    return out


class OrcFlow(C.Structure):
    _fields_ = [("dim", C.c_int), ("latent", C.c_int), ("cond", C.c_int), ("blocks", C.c_int),
                ("ln_eps", C.c_double),
                ("ip_w", C.c_void_p), ("ip_b", C.c_void_p), ("cond_w", C.c_void_p),
                ("cond_b", C.c_void_p), ("t_const", C.c_void_p),
                ("ada_w", C.c_void_p), ("ada_b", C.c_void_p), ("ln_w", C.c_void_p),
                ("ln_b", C.c_void_p), ("m0_w", C.c_void_p), ("m0_b", C.c_void_p),
                ("m2_w", C.c_void_p), ("m2_b", C.c_void_p),
                ("fada_w", C.c_void_p), ("fada_b", C.c_void_p), ("f_w", C.c_void_p),
                ("f_b", C.c_void_p)]


def flow_step(shape, weights: Dict[str, np.ndarray], cond, noise,
              precision: str = "f32") -> np.ndarray:
    """One LSD step of the flow head (`shape`: dim, latent, cond, blocks, ln_eps; `weights` as
    workloads.generate_flow draws them) for one conditioning row and one noise row."""
    keep = []

    def arr(a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        keep.append(a)
        return a.ctypes.data

    def per_block(name):
        ptrs = (C.c_void_p * max(1, shape.blocks))(*[arr(weights[f"{name}{i}"])
                                                     for i in range(shape.blocks)])
        keep.append(ptrs)
        return C.cast(ptrs, C.c_void_p).value

    f = OrcFlow(dim=shape.dim, latent=shape.latent, cond=shape.cond, blocks=shape.blocks,
                ln_eps=shape.ln_eps,
                ip_w=arr(weights["ip_w"]), ip_b=arr(weights["ip_b"]),
                cond_w=arr(weights["cond_w"]), cond_b=arr(weights["cond_b"]),
                t_const=arr(weights["t_const"]),
                ada_w=per_block("ada_w"), ada_b=per_block("ada_b"), ln_w=per_block("ln_w"),
                ln_b=per_block("ln_b"), m0_w=per_block("m0_w"), m0_b=per_block("m0_b"),
                m2_w=per_block("m2_w"), m2_b=per_block("m2_b"),
                fada_w=arr(weights["fada_w"]), fada_b=arr(weights["fada_b"]),
                f_w=arr(weights["f_w"]), f_b=arr(weights["f_b"]))
    c = np.ascontiguousarray(cond, dtype=np.float32)
    n = np.ascontiguousarray(noise, dtype=np.float32)
    out = np.empty(shape.latent, np.float64)
    if lib(precision).orc_flow_step(C.byref(f), _ptr(c, C.c_float), _ptr(n, C.c_float),
                                    _ptr(out, C.c_double)):
        raise ValueError("orc_flow_step rejected its arguments")
    return out


def ring_attention(q, kr, vr, pr, window: int, pos: int, precision: str = "f32") -> np.ndarray:
    """q [H][d]; kr, vr [ring][H][d]; pr [ring] uint32 stamps -> out [H][d]."""
    q = _d(q)
    kr = _d(kr)
    vr = _d(vr)
    pr = np.ascontiguousarray(pr, dtype=np.uint32)
    H, d = q.shape
    ring = kr.shape[0]
    out = np.empty((H, d), np.float64)
    lib(precision).orc_ring_attention(_ptr(q, C.c_double), _ptr(kr, C.c_double),
                                      _ptr(vr, C.c_double), _ptr(pr, C.c_uint32), ring, window,
                                      pos, H, d, _ptr(out, C.c_double))
    return out


def set_threads(n: int) -> None:
    for p in ("f32", "f64"):
        lib(p).orc_set_threads(int(n))


# ---------------------------------------------------------------------------- the stack

class OracleModel:
    """The decode stack on the CPU, holding its own K/V state.

    ``syn`` is a :class:`tts_autoregressive_decode_gb300.workloads.Synthetic` (or anything
    with the same fields); the weight arrays are referenced, not copied.
    """

    def __init__(self, syn, precision: str = "f32", threads: Optional[int] = None):
        w = syn.workload
        self.w = w
        self.precision = precision
        self.L = lib(precision)
        if threads is not None:
            self.L.orc_set_threads(int(threads))
        cfg = OrcConfig(kind=ORC_TALKER if w.kind == "talker" else ORC_CODEC,
                        layers=w.layers, hidden=w.hidden, q_heads=w.q_heads,
                        kv_heads=w.kv_heads, head_dim=w.head_dim, inter=w.inter,
                        norm_eps=w.norm_eps, rope_theta=w.rope_theta,
                        weight_bf16=1 if w.weight_dtype == "bf16" else 0,
                        max_pos=syn.max_pos, ring=w.ring, window=w.window, streams=w.streams)
        self._keep: List[np.ndarray] = []
        arr = (OrcLayer * w.layers)()
        for i, d in enumerate(syn.layers):
            for name, a in d.items():
                a = np.ascontiguousarray(a)
                self._keep.append(a)
                setattr(arr[i], name, a.ctypes.data)
        fn = None
        if syn.final_norm is not None:
            fn_arr = np.ascontiguousarray(syn.final_norm, dtype=np.float32)
            self._keep.append(fn_arr)
            fn = _ptr(fn_arr, C.c_float)
        self._layers = arr
        self._cfg = cfg
        self.h = self.L.orc_create(C.byref(cfg), arr, fn)
        if not self.h:
            raise ValueError("oracle rejected the configuration")
        self.eos_bias = 0.0
        if getattr(syn, "head", None) is not None:
            hd = {k: np.ascontiguousarray(v, dtype=np.float32) for k, v in syn.head.items()}
            self._keep.extend(hd.values())
            if self.L.orc_set_head(self.h, _ptr(hd["norm_w"], C.c_float),
                                   _ptr(hd["norm_b"], C.c_float), _ptr(hd["eos_w"], C.c_float)):
                raise ValueError("oracle rejected the head")
            self.eos_bias = float(hd["eos_b"][0])
        for s, n in enumerate(syn.lengths):
            if n > 0:
                self.prefill_kv(s, syn.prefill_k[s], syn.prefill_v[s])

    def prefill_kv(self, stream: int, k: np.ndarray, v: np.ndarray) -> None:
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        rc = self.L.orc_prefill_kv(self.h, stream, _ptr(k, C.c_float), _ptr(v, C.c_float),
                                   k.shape[1])
        if rc != 0:
            raise ValueError(f"orc_prefill_kv failed ({rc})")

    def set_mrope(self, assign: Optional[Sequence[int]]) -> None:
        """Talker: the axis (0 t, 1 h, 2 w) of each of the head_dim/2 rope frequencies, or None
        for the 1-D rope."""
        a = None if assign is None else np.ascontiguousarray(assign, dtype=np.int32)
        if a is not None:
            if a.shape != (self.w.head_dim // 2,):
                raise ValueError("the axis map needs head_dim/2 entries")
            self._keep.append(a)
        if self.L.orc_set_mrope(self.h, _ptr(a, C.c_int) if a is not None else None):
            raise ValueError("oracle rejected the axis map")

    def step(self, x_in: np.ndarray, pos: Sequence[int], taps: bool = False, rope_pos=None):
        """One step; rope_pos [rows][3] (optional): the rows' t, h, w rotary positions."""
        x_in = np.ascontiguousarray(x_in, dtype=np.float32)
        rows = x_in.shape[0]
        p = np.ascontiguousarray(pos, dtype=np.int32)
        r3 = None if rope_pos is None else np.ascontiguousarray(rope_pos, dtype=np.int32)
        if r3 is not None and r3.shape != (rows, 3):
            raise ValueError("rope_pos must be [rows][3]")
        out = np.empty((rows, self.w.hidden), np.float64)
        t = np.empty((self.w.layers, rows, self.w.hidden), np.float64) if taps else None
        rc = self.L.orc_step_mrope(self.h, rows, _ptr(x_in, C.c_float), _ptr(p, C.c_int),
                                   _ptr(r3, C.c_int) if r3 is not None else None,
                                   _ptr(out, C.c_double), _ptr(t, C.c_double) if taps else None)
        if rc != 0:
            raise ValueError(f"orc_step failed ({rc})")
        return (out, t) if taps else out

    def prefill(self, stream: int, x_in: np.ndarray, rope_pos=None) -> np.ndarray:
        """Causal prefill of the rows of x_in [n][hidden] into `stream`: every position's
        final-norm hidden [n][hidden].  rope_pos [n][3] (optional): per-axis rotary positions."""
        x_in = np.ascontiguousarray(x_in, dtype=np.float32)
        n = x_in.shape[0]
        r3 = None if rope_pos is None else np.ascontiguousarray(rope_pos, dtype=np.int32)
        if r3 is not None and r3.shape != (n, 3):
            raise ValueError("rope_pos must be [n][3]")
        out = np.empty((n, self.w.hidden), np.float64)
        rc = self.L.orc_prefill_mrope(self.h, stream, n, _ptr(x_in, C.c_float),
                                      _ptr(r3, C.c_int) if r3 is not None else None,
                                      _ptr(out, C.c_double))
        if rc != 0:
            raise ValueError(f"orc_prefill failed ({rc})")
        return out

    def eos(self, stream: int) -> float:
        """The last step's EOS logit of `stream`, bias included (codec head only)."""
        return float(self.L.orc_eos(self.h, stream)) + self.eos_bias

    def length(self, stream: int) -> int:
        return int(self.L.orc_len(self.h, stream))

    def read_kv(self, layer: int, stream: int, pos: int):
        n = self.w.kv_heads * self.w.head_dim
        k = np.empty(n, np.float64)
        v = np.empty(n, np.float64)
        rc = self.L.orc_read_kv(self.h, layer, stream, pos, _ptr(k, C.c_double),
                                _ptr(v, C.c_double))
        if rc != 0:
            raise ValueError("orc_read_kv failed")
        return (k.reshape(self.w.kv_heads, self.w.head_dim),
                v.reshape(self.w.kv_heads, self.w.head_dim))

    def reset(self, stream: int) -> None:
        self.L.orc_reset(self.h, stream)

    def close(self) -> None:
        if getattr(self, "h", None):
            self.L.orc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
