"""Python face of the decode library: torch tensors in, C ABI calls out.

Only argument marshalling lives here.  Every step of the decode path runs in the CUDA kernels
of libttsdec.so; torch provides device memory and the current stream.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import _lib as L
from .workloads import Synthetic, Workload

_TALKER_MAP = {"wq": "q", "wk": "k", "wv": "v", "wo": "o", "wgate": "gate", "wup": "up",
               "wdown": "down", "in_norm": "in_norm", "q_norm": "q_norm", "k_norm": "k_norm",
               "post_norm": "post_norm"}
_CODEC_MAP = {n: n for n in ("in_proj", "out_proj", "lin1", "lin2", "ln1_w", "ln1_b", "ln2_w",
                             "ln2_b", "ls1", "ls2")}


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: torch.Tensor) -> int:
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _check_rope_pos(t: torch.Tensor, rows: int) -> None:
    if t.dtype != torch.int32 or tuple(t.shape) != (rows, 3):
        raise ValueError(f"rope_pos must be int32 [{rows}][3]")


def mrope_axes(head_dim: int, sections: Sequence[int], interleaved: bool = True) -> List[int]:
    """An axis map for Decoder.set_mrope from a (t, h, w) section split of the head_dim/2 rope
    frequencies: interleaved puts h on frequencies 1, 4, 7, ... and w on 2, 5, 8, ... (each up
    to its section) and t on the rest; contiguous gives t, then h, then w, in blocks."""
    half = head_dim // 2
    if len(sections) != 3 or sum(sections) != half or min(sections) < 0:
        raise ValueError("three non-negative sections summing to head_dim/2")
    if not interleaved:
        return [0] * sections[0] + [1] * sections[1] + [2] * sections[2]
    axes = [0] * half
    for axis in (1, 2):
        for i in range(axis, min(half, 3 * sections[axis]), 3):
            axes[i] = axis
    if [axes.count(a) for a in range(3)] != list(sections):
        raise ValueError("the h and w sections do not fit an interleaved layout")
    return axes


def to_device(a: np.ndarray, device) -> torch.Tensor:
    """numpy float32 / uint16 (bf16 bit patterns) array -> device tensor with the same bytes."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device)
    return torch.from_numpy(a.astype(np.float32, copy=False)).to(device)


def config_for(w: Workload, max_pos: int, flags: int = 0) -> L.DecConfig:
    return L.DecConfig(kind=L.DEC_QWEN3_TALKER if w.kind == "talker" else L.DEC_CODEC_WINDOWED,
                       layers=w.layers, hidden=w.hidden, q_heads=w.q_heads, kv_heads=w.kv_heads,
                       head_dim=w.head_dim, inter=w.inter, norm_eps=w.norm_eps,
                       rope_theta=w.rope_theta,
                       weight_dtype=L.DEC_BF16 if w.weight_dtype == "bf16" else L.DEC_F32,
                       max_pos=max_pos, ring=w.ring, window=w.window, max_streams=w.streams,
                       flags=flags)


class Decoder:
    """A decode context (dec_create .. dec_destroy) over device-resident weights."""

    def __init__(self, cfg: L.DecConfig, layers: List[Dict[str, torch.Tensor]],
                 final_norm: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None,
                 head: Optional[Dict[str, torch.Tensor]] = None, eos_b: float = 0.0):
        self.lib = L.load()
        self.cfg = cfg
        arr = (L.DecLayerWeights * cfg.layers)()
        for i, d in enumerate(layers):
            for name, t in d.items():
                setattr(arr[i], name, _ptr(t))
        w = L.DecWeights(layers=arr, final_norm=_ptr(final_norm) if final_norm is not None else None)
        if head is not None:  # codec: the FlowLM backbone's out_norm and EOS row
            w.final_norm = _ptr(head["norm_w"])
            w.final_norm_b = _ptr(head["norm_b"])
            w.eos_w = _ptr(head["eos_w"])
            w.eos_b = float(eos_b)
        h = C.c_void_p()
        st = self.lib.dec_create(C.byref(cfg), C.byref(w), _stream_handle(stream), C.byref(h))
        L.check(st, None)
        self.h = h
        self.hidden = cfg.hidden
        self.streams = cfg.max_streams

    # ---------------------------------------------------------------- construction helpers
    @classmethod
    def from_synthetic(cls, syn: Synthetic, device="cuda", flags: int = 0,
                       stream: Optional[torch.cuda.Stream] = None, prefill: bool = True):
        w = syn.workload
        cfg = config_for(w, syn.max_pos, flags)
        names = _TALKER_MAP if w.kind == "talker" else _CODEC_MAP
        layers = [{names[k]: to_device(v, device) for k, v in d.items()} for d in syn.layers]
        fn = to_device(syn.final_norm, device) if syn.final_norm is not None else None
        head = None
        if getattr(syn, "head", None) is not None:
            head = {k: to_device(syn.head[k], device) for k in ("norm_w", "norm_b", "eos_w")}
        eos_b = float(syn.head["eos_b"][0]) if head is not None else 0.0
        dec = cls(cfg, layers, fn, stream, head, eos_b)
        del layers, fn, head   # the context holds its own copy of the weights
        if prefill:
            for s, n in enumerate(syn.lengths):
                if n > 0:
                    dec.prefill_kv(s, to_device(syn.prefill_k[s], device),
                                   to_device(syn.prefill_v[s], device))
        return dec

    # ---------------------------------------------------------------- the ABI
    def set_stream(self, stream: Optional[torch.cuda.Stream]) -> None:
        L.check(self.lib.dec_set_stream(self.h, _stream_handle(stream)), self.h)

    def prefill_kv(self, stream: int, k: torch.Tensor, v: torch.Tensor) -> None:
        n = int(k.shape[1]) if k is not None else 0
        L.check(self.lib.dec_prefill_kv(self.h, stream, _ptr(k), _ptr(v), n), self.h)
        self.sync()  # keep the sources alive until the copy has run

    def prefill(self, stream: int, x: torch.Tensor, out: Optional[torch.Tensor] = None,
                rope_pos: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Append the n rows of x [n][hidden] (device f32) to `stream` at its next positions and
        return every position's final-norm hidden [n][hidden] (asynchronous).  rope_pos: the
        rows' t, h, w rotary positions, device int32 [n][3] (multimodal rope)."""
        n = int(x.shape[0])
        if out is None:
            out = torch.empty_like(x)
        if rope_pos is None:
            L.check(self.lib.dec_prefill(self.h, stream, n, _ptr(x), _ptr(out)), self.h)
        else:
            _check_rope_pos(rope_pos, n)
            L.check(self.lib.dec_prefill_mrope(self.h, stream, n, _ptr(x), _ptr(rope_pos),
                                               _ptr(out)), self.h)
        return out

    def set_mrope(self, axes: Optional[Sequence[int]]) -> None:
        """The axis (0 t, 1 h, 2 w) of each of the head_dim/2 rope frequencies (None: all t)."""
        if axes is None:
            L.check(self.lib.dec_set_mrope(self.h, None, 0), self.h)
            return
        a = (C.c_int32 * len(axes))(*[int(v) for v in axes])
        L.check(self.lib.dec_set_mrope(self.h, a, len(axes)), self.h)

    def read_eos(self, m: int) -> np.ndarray:
        """The EOS logits of the last step of streams 0..m-1 (bias included); blocking."""
        out = np.empty(m, np.float32)
        L.check(self.lib.dec_read_eos(self.h, m, out.ctypes.data), self.h)
        return out

    def prefill_rows(self) -> int:
        """Rows per prefill block (0: prefill not served)."""
        return int(self.lib.dec_prefill_block_rows(self.h))

    def step(self, x: torch.Tensor, pos: Sequence[int], out: Optional[torch.Tensor] = None,
             rope_pos: Optional[torch.Tensor] = None) -> torch.Tensor:
        """One step of streams 0..m-1 (asynchronous); rope_pos: the rows' t, h, w rotary
        positions, device int32 [m][3] (multimodal rope)."""
        m = int(x.shape[0])
        if out is None:
            out = torch.empty_like(x)
        p = (C.c_int32 * m)(*[int(v) for v in pos])
        if rope_pos is None:
            L.check(self.lib.dec_step(self.h, m, _ptr(x), p, _ptr(out)), self.h)
        else:
            _check_rope_pos(rope_pos, m)
            L.check(self.lib.dec_step_mrope(self.h, m, _ptr(x), p, _ptr(rope_pos), _ptr(out)),
                    self.h)
        return out

    def step_host(self, x: np.ndarray, pos: Sequence[int], out: Optional[np.ndarray] = None
                  ) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        m = x.shape[0]
        if out is None:
            out = np.empty_like(x)
        p = (C.c_int32 * m)(*[int(v) for v in pos])
        L.check(self.lib.dec_step_host(self.h, m, x.ctypes.data, p, out.ctypes.data), self.h)
        return out

    def step_host_ptr(self, m: int, x_ptr: int, pos_arr, out_ptr: int) -> None:
        """dec_step_host on raw host addresses (pinned buffers), pos as a ctypes int32 array."""
        L.check(self.lib.dec_step_host(self.h, m, x_ptr, pos_arr, out_ptr), self.h)

    def reset(self, stream: int) -> None:
        L.check(self.lib.dec_reset(self.h, stream), self.h)

    def sync(self) -> None:
        L.check(self.lib.dec_sync(self.h), self.h)

    def length(self, stream: int) -> int:
        return int(self.lib.dec_get_len(self.h, stream))

    def lengths(self, m: Optional[int] = None) -> List[int]:
        return [self.length(s) for s in range(m if m is not None else self.streams)]

    def read_kv(self, layer: int, stream: int, position: int):
        G, d = self.cfg.kv_heads, self.cfg.head_dim
        k = np.empty((G, d), np.float32)
        v = np.empty((G, d), np.float32)
        L.check(self.lib.dec_read_kv(self.h, layer, stream, position, k.ctypes.data,
                                     v.ctypes.data), self.h)
        return k, v

    def read_tap(self, layer: int, m: int) -> np.ndarray:
        out = np.empty((m, self.hidden), np.float32)
        L.check(self.lib.dec_read_tap(self.h, layer, m, out.ctypes.data), self.h)
        return out

    def kernels_per_step(self, m: int) -> int:
        return int(self.lib.dec_kernels_per_step(self.h, m))

    def inject_stall(self, phase: int, polls: int) -> None:
        """The next persistent-plan step waits in `phase` for activations no CTA writes, each
        wait bounded by `polls` loads (dec_inject_stall): a check of the bounded-wait path."""
        L.check(self.lib.dec_inject_stall(self.h, int(phase), int(polls)), self.h)

    def truncate(self, stream: int, new_len: int) -> None:
        L.check(self.lib.dec_truncate(self.h, stream, new_len), self.h)

    def launch_stage(self, layer: int, stage: int, m: int, chained: bool = False) -> None:
        L.check(self.lib.dec_launch_stage(self.h, layer, stage, m, 1 if chained else 0), self.h)

    def close(self) -> None:
        if getattr(self, "h", None):
            self.lib.dec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------ stateless kernel entries

def gemv(W: torch.Tensor, x: torch.Tensor, out: Optional[torch.Tensor] = None,
         bf16: Optional[bool] = None) -> torch.Tensor:
    """y[r] = W x[r] with W [N][K] float32 or int16 (bf16 bit patterns), x [m][K] float32."""
    lib = L.load()
    N, K = W.shape
    m = x.shape[0]
    if bf16 is None:
        bf16 = W.dtype in (torch.int16, torch.bfloat16)
    if out is None:
        out = torch.empty((m, N), dtype=torch.float32, device=x.device)
    L.check(lib.dec_gemv(L.DEC_BF16 if bf16 else L.DEC_F32, _ptr(W), N, K, _ptr(x), m, _ptr(out),
                         _stream_handle(None)))
    return out


def attention_workspace_bytes(m: int, H: int, G: int, d: int, capacity: int) -> int:
    return int(L.load().dec_attention_workspace_bytes(m, H, G, d, capacity))


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lens: torch.Tensor,
              out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None
              ) -> torch.Tensor:
    """q [m][H][d]; k, v [m][G][capacity][d]; lens int32 [m] on the device -> out [m][H][d]."""
    lib = L.load()
    m, H, d = q.shape
    _, G, cap, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    nbytes = attention_workspace_bytes(m, H, G, d, cap)
    if workspace is None:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    L.check(lib.dec_attention(m, H, G, d, cap, _ptr(q), _ptr(k), _ptr(v), _ptr(lens), _ptr(out),
                              _ptr(workspace), workspace.numel(), _stream_handle(None)))
    return out


# ----------------------------------------------------------------------------------------
class FlowHead:
    """The flow head (dec_flow_create .. dec_flow_destroy): one LSD step per call, conditioned
    on a device row (the backbone's hidden state, read in place)."""

    def __init__(self, shape, weights: Dict[str, np.ndarray], device="cuda",
                 stream: Optional[torch.cuda.Stream] = None):
        self.lib = L.load()
        self.shape = shape
        dev = {k: to_device(v, device) for k, v in weights.items() if k not in ("cond", "noise")}
        cfg = L.DecFlowConfig(dim=shape.dim, latent=shape.latent, cond=shape.cond,
                              blocks=shape.blocks, ln_eps=shape.ln_eps, lsd_steps=1)
        w = L.DecFlowWeights()
        for n in ("ip_w", "ip_b", "cond_w", "cond_b", "t_const", "fada_w", "fada_b", "f_w", "f_b"):
            setattr(w, n, _ptr(dev[n]))
        self._arrays = []
        for n in L.FLOW_BLOCK_FIELDS:
            arr = (C.c_void_p * max(1, shape.blocks))(*[_ptr(dev[f"{n}{i}"])
                                                        for i in range(shape.blocks)])
            self._arrays.append(arr)
            setattr(w, n, C.cast(arr, C.POINTER(C.c_void_p)))
        h = C.c_void_p()
        st = self.lib.dec_flow_create(C.byref(cfg), C.byref(w), _stream_handle(stream), C.byref(h))
        L.check_flow(st, None)
        self.h = h
        del dev   # the head holds its own copy of the weights

    def step(self, cond: torch.Tensor, noise: torch.Tensor,
             out: Optional[torch.Tensor] = None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(noise)
        L.check_flow(self.lib.dec_flow_step(self.h, _ptr(cond), _ptr(noise), _ptr(out)), self.h)
        return out

    def kernels_per_step(self) -> int:
        return int(self.lib.dec_flow_kernels_per_step(self.h))

    def close(self) -> None:
        if getattr(self, "h", None):
            self.lib.dec_flow_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
