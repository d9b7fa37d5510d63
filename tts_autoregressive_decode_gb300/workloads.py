"""Synthetic, seeded decode workloads: shapes, value distributions and draw order.

This module holds no arithmetic of the decode step.  It only states the workload shapes and
draws their inputs, so that the CUDA library and the CPU oracle consume the very same bytes.

Draw recipe (numpy PCG64; one child stream per category, spawned from the seed with
``np.random.SeedSequence(seed).spawn(4)`` so that one category never shifts another):

  child 0  stream lengths   -- only where lengths are random: integers in [lo, hi], inclusive
  child 1  weights          -- layer by layer, tensor by tensor in the order of
                               ``TALKER_TENSORS`` / ``CODEC_TENSORS`` (the codec's LayerScale
                               only where the workload has it), then the talker's final norm,
                               or the codec head where the workload has one: out_norm weight,
                               out_norm bias, EOS weights [hidden] (linear), EOS bias (scalar,
                               0.01 N(0, 1))
           linear weights   N(0, 1) float32 draws times 0.02 (in float32)
           norm weights     1 + 0.01 N(0, 1)
           LayerNorm biases 0.01 N(0, 1)
           LayerScale       0.01 + 0.001 N(0, 1)
           bf16 storage     round-to-nearest-even of the float32 draw (bit patterns, uint16)
  child 2  prefilled K/V    per stream: K then V, each [layers][n_pos][kv_heads][head_dim],
                            N(0, 1) float32, read as keys that already carry rope
  child 3  step inputs      talker/codec without feedback: [steps][streams][hidden] N(0, 1);
                            with feedback: x_0 [streams][hidden] then e [hidden], both N(0, 1),
                            and step s+1 takes hidden_s + e
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

TALKER_TENSORS = ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown",
                  "in_norm", "q_norm", "k_norm", "post_norm")
CODEC_TENSORS = ("in_proj", "out_proj", "lin1", "lin2",
                 "ln1_w", "ln1_b", "ln2_w", "ln2_b", "ls1", "ls2")


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "talker" or "codec"
    layers: int
    hidden: int
    q_heads: int
    kv_heads: int
    head_dim: int
    inter: int
    norm_eps: float
    rope_theta: float
    weight_dtype: str         # "f32" or "bf16"
    streams: int
    steps: int
    seed: int
    prefill: Tuple[int, ...] = ()          # per-stream prefill lengths (fixed)
    prefill_range: Optional[Tuple[int, int]] = None   # random per-stream lengths [lo, hi]
    feedback: bool = False    # step s+1 input = hidden_s + e
    ring: int = 0             # codec ring slots
    window: int = 0           # codec attention window
    max_pos: int = 0          # 0: derived (longest prefill + steps)
    layer_scale: bool = True  # codec: LayerScale on both residual branches
    head: bool = False        # codec: final LayerNorm and an EOS logit (the FlowLM backbone)
    description: str = ""

    @property
    def qw(self) -> int:
        return self.q_heads * self.head_dim

    @property
    def kvw(self) -> int:
        return self.kv_heads * self.head_dim

    def weight_shapes(self) -> Dict[str, Tuple[int, ...]]:
        h, I = self.hidden, self.inter
        if self.kind == "talker":
            return {"wq": (self.qw, h), "wk": (self.kvw, h), "wv": (self.kvw, h),
                    "wo": (h, self.qw), "wgate": (I, h), "wup": (I, h), "wdown": (h, I),
                    "in_norm": (h,), "q_norm": (self.head_dim,), "k_norm": (self.head_dim,),
                    "post_norm": (h,)}
        shapes = {"in_proj": (3 * h, h), "out_proj": (h, h), "lin1": (I, h), "lin2": (h, I),
                  "ln1_w": (h,), "ln1_b": (h,), "ln2_w": (h,), "ln2_b": (h,)}
        if self.layer_scale:
            shapes.update({"ls1": (h,), "ls2": (h,)})
        return shapes

    def matrix_bytes(self) -> int:
        es = 2 if self.weight_dtype == "bf16" else 4
        return self.layers * sum(int(np.prod(s)) * es for s in self.weight_shapes().values()
                                 if len(s) == 2)


def _seed_children(seed: int):
    return np.random.SeedSequence(seed).spawn(4)


def prefill_lengths(w: Workload) -> List[int]:
    if w.prefill_range is not None:
        lo, hi = w.prefill_range
        rng = np.random.Generator(np.random.PCG64(_seed_children(w.seed)[0]))
        return [int(v) for v in rng.integers(lo, hi, size=w.streams, endpoint=True)]
    if w.prefill:
        return list(w.prefill) + [w.prefill[-1]] * (w.streams - len(w.prefill))
    return [0] * w.streams


def max_pos(w: Workload) -> int:
    if w.max_pos:
        return w.max_pos
    return max(prefill_lengths(w)) + w.steps


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@dataclass
class Synthetic:
    workload: Workload
    layers: List[Dict[str, np.ndarray]]
    final_norm: Optional[np.ndarray]
    lengths: List[int]
    prefill_k: List[Optional[np.ndarray]]     # per stream [layers][n][G][d] float32
    prefill_v: List[Optional[np.ndarray]]
    inputs: Optional[np.ndarray]              # [steps][streams][hidden]
    x0: Optional[np.ndarray] = None           # feedback: [streams][hidden]
    e: Optional[np.ndarray] = None            # feedback: [hidden]
    max_pos: int = 0
    head: Optional[Dict[str, np.ndarray]] = None  # codec head: norm_w, norm_b, eos_w, eos_b


def _normal(rng, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def generate(w: Workload, steps: Optional[int] = None, with_inputs: bool = True) -> Synthetic:
    """Draw every array of workload ``w`` (see the module doc for the recipe)."""
    c = _seed_children(w.seed)
    lengths = prefill_lengths(w)
    rw = np.random.Generator(np.random.PCG64(c[1]))
    shapes = w.weight_shapes()
    order = TALKER_TENSORS if w.kind == "talker" else CODEC_TENSORS
    layers = []
    for _ in range(w.layers):
        d = {}
        for name in order:
            if name not in shapes:
                continue
            s = shapes[name]
            if len(s) == 2:
                a = _normal(rw, s) * np.float32(0.02)
                d[name] = f32_to_bf16_bits(a) if w.weight_dtype == "bf16" else a
            elif name.endswith("_b"):
                d[name] = _normal(rw, s) * np.float32(0.01)
            elif name.startswith("ls"):
                d[name] = np.float32(0.01) + _normal(rw, s) * np.float32(0.001)
            else:
                d[name] = np.float32(1.0) + _normal(rw, s) * np.float32(0.01)
        layers.append(d)
    final_norm = head = None
    if w.kind == "talker":
        final_norm = np.float32(1.0) + _normal(rw, (w.hidden,)) * np.float32(0.01)
    elif w.head:
        head = {"norm_w": np.float32(1.0) + _normal(rw, (w.hidden,)) * np.float32(0.01),
                "norm_b": _normal(rw, (w.hidden,)) * np.float32(0.01),
                "eos_w": _normal(rw, (w.hidden,)) * np.float32(0.02),
                "eos_b": _normal(rw, (1,)) * np.float32(0.01)}

    rk = np.random.Generator(np.random.PCG64(c[2]))
    pk, pv = [], []
    for n in lengths:
        if n > 0:
            pk.append(_normal(rk, (w.layers, n, w.kv_heads, w.head_dim)))
            pv.append(_normal(rk, (w.layers, n, w.kv_heads, w.head_dim)))
        else:
            pk.append(None)
            pv.append(None)

    nsteps = w.steps if steps is None else steps
    ri = np.random.Generator(np.random.PCG64(c[3]))
    inputs = x0 = e = None
    if with_inputs:
        if w.feedback:
            x0 = _normal(ri, (w.streams, w.hidden))
            e = _normal(ri, (w.hidden,))
        else:
            inputs = _normal(ri, (nsteps, w.streams, w.hidden))
    return Synthetic(w, layers, final_norm, lengths, pk, pv, inputs, x0, e, max_pos(w), head)


# ----------------------------------------------------------------------------------------
# the workloads
# ----------------------------------------------------------------------------------------

TALKER_H256_L1 = Workload(
    name="talker_h256_l1_f32", kind="talker", layers=1, hidden=256, q_heads=4, kv_heads=2,
    head_dim=64, inter=768, norm_eps=1e-6, rope_theta=1e6, weight_dtype="f32", streams=1,
    steps=1, seed=0, prefill=(32,),
    description="1 layer f32, h256, 4/2 heads, d64, SwiGLU 768; 32 prefilled positions; "
                "one step at pos 32")

TALKER_H1024_L4 = Workload(
    name="talker_h1024_l4_f32_feedback", kind="talker", layers=4, hidden=1024, q_heads=16,
    kv_heads=8, head_dim=128, inter=3072, norm_eps=1e-6, rope_theta=1e6, weight_dtype="f32",
    streams=1, steps=64, seed=1, prefill=(256,), feedback=True,
    description="4 layers f32, h1024, 16/8 heads, d128, SwiGLU 3072; 256 prefilled positions; "
                "64 steps, output hidden + fixed N(0,1) embedding fed back")

TALKER_H2048_L28 = Workload(
    name="talker_h2048_l28_bf16", kind="talker", layers=28, hidden=2048, q_heads=16,
    kv_heads=8, head_dim=128, inter=6144, norm_eps=1e-6, rope_theta=1e6, weight_dtype="bf16",
    streams=1, steps=128, seed=2, prefill=(2048,),
    description="28 layers, bf16-stored weights widened to f32, h2048, 16/8 heads, d128, "
                "SwiGLU 6144; f32 KV prefilled with 2048 positions; 128 steps")

CODEC_D512_L8 = Workload(
    name="codec_d512_l8_ring250", kind="codec", layers=8, hidden=512, q_heads=8, kv_heads=8,
    head_dim=64, inter=2048, norm_eps=1e-5, rope_theta=1e4, weight_dtype="f32", streams=1,
    steps=600, seed=3, ring=250, window=250,
    description="8-layer windowed codec transformer f32, d512, 8 heads MHA d64, LayerNorm, "
                "GELU(erf) MLP 2048, LayerScale, 250-slot KV ring + position ring; "
                "600 steps from an empty ring (two wraps)")

TALKER_H2048_L28_M8 = Workload(
    name="talker_h2048_l28_bf16_m8", kind="talker", layers=28, hidden=2048, q_heads=16,
    kv_heads=8, head_dim=128, inter=6144, norm_eps=1e-6, rope_theta=1e6, weight_dtype="bf16",
    streams=8, steps=64, seed=4, prefill_range=(512, 4096),
    description="batched decode of 8 streams sharing one read of each weight; 28-layer "
                "bf16 talker; per-stream f32 KV prefilled to lengths U[512, 4096]; 64 steps")

# The FlowLM backbone shape (Pocket TTS on wgpu, PocketBackboneGpu): the codec-style stack
# without LayerScale and with an unbounded window (window = ring = the utterance's positions),
# then the final LayerNorm and the EOS logit.  The FFN width is not on the pages: 4 x d_model.
FLOWLM_D1024_L6 = Workload(
    name="flowlm_d1024_l6", kind="codec", layers=6, hidden=1024, q_heads=16, kv_heads=16,
    head_dim=64, inter=4096, norm_eps=1e-5, rope_theta=1e4, weight_dtype="f32", streams=1,
    steps=64, seed=5, prefill=(256,), ring=320, window=320, max_pos=320, layer_scale=False,
    head=True,
    description="FlowLM backbone: 6 layers f32, d1024, 16 heads MHA d64, LayerNorm, GELU(erf) "
                "MLP 4096, no LayerScale, unbounded window (ring = window = 320 positions), "
                "final LayerNorm + EOS logit; 256 prefilled positions (a voice), 64 steps")

WORKLOADS: Dict[str, Workload] = {w.name: w for w in (
    TALKER_H256_L1, TALKER_H1024_L4, TALKER_H2048_L28, CODEC_D512_L8, TALKER_H2048_L28_M8,
    FLOWLM_D1024_L6)}

# Small shapes for element-by-element parity: several tiles and a ragged tail everywhere
# (hidden and inter not multiples of the 256-element warp step, prefills not multiples of
# the 64-key attention chunk, a GQA group of 3, streams of different lengths).
SMALL_TALKER_F32 = Workload(
    name="small_talker_f32", kind="talker", layers=2, hidden=392, q_heads=6, kv_heads=2,
    head_dim=64, inter=1000, norm_eps=1e-6, rope_theta=1e6, weight_dtype="f32", streams=3,
    steps=5, seed=11, prefill=(70, 129, 1))
SMALL_TALKER_BF16 = dataclasses.replace(
    SMALL_TALKER_F32, name="small_talker_bf16", weight_dtype="bf16", seed=12,
    head_dim=128, q_heads=4, kv_heads=2, prefill=(0, 191, 64))
SMALL_CODEC = Workload(
    name="small_codec", kind="codec", layers=2, hidden=256, q_heads=4, kv_heads=4,
    head_dim=64, inter=520, norm_eps=1e-5, rope_theta=1e4, weight_dtype="f32", streams=2,
    steps=45, seed=13, ring=20, window=17, prefill=(0, 9), max_pos=64)

SMALL_FLOWLM = dataclasses.replace(
    SMALL_CODEC, name="small_flowlm", seed=14, ring=40, window=40, max_pos=40, prefill=(7, 0),
    steps=30, layer_scale=False, head=True)

# ----------------------------------------------------------------------------------------
# the flow head (Pocket TTS on wgpu, PocketFlowGpu: SimpleMLPAdaLN, one LSD step)
# ----------------------------------------------------------------------------------------
@dataclass(frozen=True)
class FlowShape:
    name: str
    dim: int          # the head's width
    latent: int       # latent (noise) width
    cond: int         # conditioning width: the backbone's d_model
    blocks: int
    seed: int
    ln_eps: float = 1e-6


# Widths the pages do not give; the conditioning is the FlowLM backbone's d_model (1024).
FLOW_D512 = FlowShape(name="flow_d512_l32_b3", dim=512, latent=32, cond=1024, blocks=3, seed=6)
SMALL_FLOW = FlowShape(name="small_flow", dim=136, latent=24, cond=256, blocks=2, seed=15)


def generate_flow(f: FlowShape, calls: int = 4) -> Dict[str, np.ndarray]:
    """Weights of the flow head, then `calls` conditioning rows and noise rows.

    Draw order (PCG64 from the seed): input_proj W [dim][latent], b [dim]; cond W [dim][cond],
    b [dim]; the time constant [dim]; per block: adaLN W [3 dim][dim], b [3 dim], in_ln w, b
    [dim], m0 W [dim][dim], b [dim], m2 W [dim][dim], b [dim]; final adaLN W [2 dim][dim],
    b [2 dim]; final W [latent][dim], b [latent]; then the inputs: cond [calls][cond] and noise
    [calls][latent], N(0, 1).  Linear weights N(0, 1) x 0.02, biases and the time constant
    N(0, 1) x 0.1, LayerNorm weights 1 + 0.01 N, biases 0.01 N.
    """
    r = np.random.Generator(np.random.PCG64(f.seed))
    lin = lambda n, k: _normal(r, (n, k)) * np.float32(0.02)
    vec = lambda n, s: _normal(r, (n,)) * np.float32(s)
    d = {"ip_w": lin(f.dim, f.latent), "ip_b": vec(f.dim, 0.1),
         "cond_w": lin(f.dim, f.cond), "cond_b": vec(f.dim, 0.1), "t_const": vec(f.dim, 0.1)}
    for i in range(f.blocks):
        d[f"ada_w{i}"] = lin(3 * f.dim, f.dim)
        d[f"ada_b{i}"] = vec(3 * f.dim, 0.1)
        d[f"ln_w{i}"] = np.float32(1.0) + vec(f.dim, 0.01)
        d[f"ln_b{i}"] = vec(f.dim, 0.01)
        d[f"m0_w{i}"] = lin(f.dim, f.dim)
        d[f"m0_b{i}"] = vec(f.dim, 0.1)
        d[f"m2_w{i}"] = lin(f.dim, f.dim)
        d[f"m2_b{i}"] = vec(f.dim, 0.1)
    d["fada_w"] = lin(2 * f.dim, f.dim)
    d["fada_b"] = vec(2 * f.dim, 0.1)
    d["f_w"] = lin(f.latent, f.dim)
    d["f_b"] = vec(f.latent, 0.1)
    d["cond"] = _normal(r, (calls, f.cond))
    d["noise"] = _normal(r, (calls, f.latent))
    return d


SMALL: Dict[str, Workload] = {w.name: w for w in (SMALL_TALKER_F32, SMALL_TALKER_BF16,
                                                  SMALL_CODEC, SMALL_FLOWLM)}
