"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks a primitive (or the assembled stack) against a closed form, an invariant,
a special case that reduces to a library routine (numpy matmul, scipy softmax / normal CDF /
logistic), brute force on tiny inputs, or a value the pages print.  They are chosen so that a
plausible slip -- a dropped term, a flipped sign, a wrong index, a transposed operand, eps in
the wrong place -- fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special as sps

import oracle
from tts_autoregressive_decode_gb300 import workloads as W

U32 = 2.0 ** -24  # unit roundoff of f32


def _rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------------ bf16 widening

def test_bf16_widening_matches_format_facts(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "bf16_bit_patterns.json")))
    for c in g["cases"]:
        got = oracle.bf16_to_f32(int(c["bits"], 16))
        want = float(c["value"])
        assert (got == want) and (math.copysign(1, got) == math.copysign(1, want)), c


# ------------------------------------------------------------------------ GEMV

@pytest.mark.parametrize("prec", ["f32", "f64"])
@pytest.mark.parametrize("N,K", [(1, 1), (3, 7), (17, 64), (40, 333)])
def test_matvec_within_f32_bound_of_numpy(prec, N, K):
    r = _rng(N * 1000 + K)
    Wt = r.standard_normal((N, K)).astype(np.float32)
    x = r.standard_normal(K).astype(np.float32).astype(np.float64)
    y = oracle.matvec(Wt, x, prec)
    ref = Wt.astype(np.float64) @ x                    # library matmul in f64
    bound = (2 * K * U32 if prec == "f32" else 1e-12) * (np.abs(Wt) @ np.abs(x)) + 1e-30
    assert np.all(np.abs(y - ref) <= bound)


def test_matvec_permutation_is_exact_and_not_transposed():
    # y[n] = sum_k W[n,k] x[k]: with W the permutation matrix of p, y[n] = x[p[n]].
    # A transposed operand would give the inverse permutation instead.
    K = 9
    p = np.array([3, 0, 7, 1, 8, 2, 6, 4, 5])
    Wt = np.zeros((K, K), np.float32)
    Wt[np.arange(K), p] = 1.0
    assert not np.array_equal(p[p], np.arange(K))     # not an involution
    x = _rng(1).standard_normal(K).astype(np.float32)
    y = oracle.matvec(Wt, x)
    assert np.array_equal(y, x[p].astype(np.float64))


def test_matvec_bf16_uses_exact_widening():
    r = _rng(2)
    Wf = (r.standard_normal((5, 24)) * 0.02).astype(np.float32)
    bits = W.f32_to_bf16_bits(Wf)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    x = r.standard_normal(24).astype(np.float32)
    # the bf16 path must equal the f32 path run on the widened values, bit for bit
    assert np.array_equal(oracle.matvec(bits, x), oracle.matvec(widened, x))
    # and bf16 rounding is to nearest: within half a bf16 ulp of the f32 draw
    assert np.all(np.abs(widened - Wf) <= np.abs(Wf) * 2.0 ** -8)


# ------------------------------------------------------------------------ RMSNorm / LayerNorm

def test_rms_norm_closed_form_eps_inside_the_root():
    # x = (3, 4): mean(x^2) = 12.5; with eps = 12.5 the root is exactly 5
    y = oracle.rms_norm([3.0, 4.0], np.ones(2, np.float32), 12.5, "f64")
    assert np.allclose(y, [0.6, 0.8], atol=1e-15)
    y = oracle.rms_norm([3.0, 4.0], np.array([2.0, -1.0], np.float32), 12.5, "f64")
    assert np.allclose(y, [1.2, -0.8], atol=1e-15)


@pytest.mark.parametrize("n", [1, 64, 2048])
def test_rms_norm_unit_rms_and_scale_invariance(n):
    r = _rng(n)
    x = r.standard_normal(n) * 3.0
    w = np.ones(n, np.float32)
    y = oracle.rms_norm(x, w, 0.0, "f64")
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-12
    y2 = oracle.rms_norm(x * 7.5, w, 0.0, "f64")
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-14)
    ww = (1 + 0.01 * r.standard_normal(n)).astype(np.float32)
    y3 = oracle.rms_norm(x, ww, 0.0, "f64")
    assert np.allclose(y3 / ww, y, rtol=1e-12)


def test_layer_norm_closed_form_and_moments():
    x = np.array([1.0, 2.0, 3.0, 4.0])          # mean 2.5, biased var 1.25
    y = oracle.layer_norm(x, np.ones(4, np.float32), np.zeros(4, np.float32), 3.75, "f64")
    assert np.allclose(y, (x - 2.5) / math.sqrt(5.0), atol=1e-15)
    y = oracle.layer_norm(x, np.full(4, 2, np.float32), np.ones(4, np.float32), 3.75, "f64")
    assert np.allclose(y, 2 * (x - 2.5) / math.sqrt(5.0) + 1, atol=1e-14)
    r = _rng(5)
    z = r.standard_normal(512) * 4 + 3
    y = oracle.layer_norm(z, np.ones(512, np.float32), np.zeros(512, np.float32), 0.0, "f64")
    assert abs(y.mean()) < 1e-12 and abs(y.var() - 1.0) < 1e-12


# ------------------------------------------------------------------------ RoPE

def test_rope_pos0_is_identity():
    r = _rng(3)
    for d, theta in ((64, 1e6), (128, 1e6), (64, 1e4)):
        c, s = oracle.rope_table(d, theta, 0)
        assert np.all(c == 1.0) and np.all(s == 0.0)
        x = r.standard_normal(d).astype(np.float32)
        assert np.array_equal(oracle.rope_rotate_half(x, c, s), x.astype(np.float64))
        assert np.array_equal(oracle.rope_interleaved(x, c, s), x.astype(np.float64))


def test_rope_d2_is_rotation_by_pos():
    # d = 2 has the single frequency theta^0 = 1: the pair turns by `pos` radians,
    # counter-clockwise, (1, 0) -> (cos p, sin p) (ROPE_SRC: out = x c + rot s, rot0 = -x1)
    for pos in (1, 5, 33, 1000):
        c, s = oracle.rope_table(2, 1e6, pos, "f64")
        assert c[0] == math.cos(pos) and s[0] == math.sin(pos)
        y = oracle.rope_rotate_half([1.0, 0.0], c, s, "f64")
        assert np.allclose(y, [math.cos(pos), math.sin(pos)], atol=1e-15)
        y = oracle.rope_interleaved([0.0, 1.0], c, s, "f64")
        assert np.allclose(y, [-math.sin(pos), math.cos(pos)], atol=1e-15)


def test_rope_table_frequency_ladder():
    # theta^(-2i/d) at i = d/4 is theta^(-1/2): 1e-3 for theta = 1e6, 1e-2 for 1e4
    for d, theta, f in ((128, 1e6, 1e-3), (64, 1e6, 1e-3), (64, 1e4, 1e-2)):
        for pos in (7, 2048, 4159):
            c, s = oracle.rope_table(d, theta, pos, "f64")
            assert abs(c[d // 4] - math.cos(pos * f)) < 1e-13
            assert abs(s[d // 4] - math.sin(pos * f)) < 1e-13
    # the f32 table is the f64 table rounded once to f32
    c64, s64 = oracle.rope_table(128, 1e6, 2049, "f64")
    c32, s32 = oracle.rope_table(128, 1e6, 2049, "f32")
    assert np.array_equal(c32, c64.astype(np.float32).astype(np.float64))
    assert np.array_equal(s32, s64.astype(np.float32).astype(np.float64))


def test_rope_preserves_pair_norms_and_is_relative():
    r = _rng(4)
    d = 128
    q = r.standard_normal(d)
    k = r.standard_normal(d)
    for fn in (oracle.rope_rotate_half, oracle.rope_interleaved):
        def rot(x, p):
            c, s = oracle.rope_table(d, 1e6, p, "f64")
            return fn(x, c, s, "f64")
        y = rot(q, 77)
        assert abs(np.linalg.norm(y) - np.linalg.norm(q)) < 1e-12
        # RoPE(q, m) . RoPE(k, n) depends on m - n only
        a = rot(q, 100) @ rot(k, 90)
        b = rot(q, 1010) @ rot(k, 1000)
        c0 = rot(q, 10) @ rot(k, 0)
        assert abs(a - b) < 1e-9 and abs(a - c0) < 1e-9
        assert abs(a - rot(q, 11) @ rot(k, 0)) > 1e-6


def test_rope_interleaved_is_rotate_half_on_deinterleaved_lanes():
    # pairs (2j, 2j+1) of the codec rope are pairs (j, j + d/2) of rotate_half
    r = _rng(6)
    d = 64
    x = r.standard_normal(d)
    c, s = oracle.rope_table(d, 1e4, 123, "f64")
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
    y_int = oracle.rope_interleaved(x, c, s, "f64")
    y_rh = oracle.rope_rotate_half(x[perm], c, s, "f64")
    back = np.empty(d)
    back[perm] = y_rh
    assert np.allclose(y_int, back, atol=1e-15)


def test_mrope_uniform_positions_equal_1d_rope():
    d = 128
    half = d // 2
    assigns = [
        [0] * 16 + [1] * 24 + [2] * 24,               # contiguous sections
        [i % 3 for i in range(half)],                  # interleaved round robin
        [(i * 7) % 3 for i in range(half)],
    ]
    for pos in (0, 1, 513, 4095):
        c1, s1 = oracle.rope_table(d, 1e6, pos)
        for a in assigns:
            c3, s3 = oracle.mrope_table(d, 1e6, [pos, pos, pos], a)
            assert np.array_equal(c1, c3) and np.array_equal(s1, s3)
        c3, s3 = oracle.mrope_table(d, 1e6, [pos, pos + 1, pos + 2], assigns[1])
        assert not np.array_equal(c1, c3)


# ------------------------------------------------------------------------ activations

def test_silu_and_gelu_against_library_routines():
    for v in (-6.0, -2.0, -1.0, -0.5, 0.0, 0.3, 1.0, 2.0, 5.0):
        assert abs(oracle.silu(v, "f64") - v * sps.expit(v)) < 1e-15 * max(1, abs(v))
        assert abs(oracle.gelu(v, "f64") - v * sps.ndtr(v)) < 1e-15 * max(1, abs(v))
        assert abs(oracle.silu(v) - v * sps.expit(v)) < 4 * U32 * max(1, abs(v))
        assert abs(oracle.gelu(v) - v * sps.ndtr(v)) < 4 * U32 * max(1, abs(v))
    assert oracle.silu(0.0) == 0.0 and oracle.gelu(0.0) == 0.0
    for v in (0.25, 1.5, 3.0):     # odd parts: f(x) - f(-x) = x for both
        assert abs(oracle.silu(v, "f64") - oracle.silu(-v, "f64") - v) < 1e-15
        assert abs(oracle.gelu(v, "f64") - oracle.gelu(-v, "f64") - v) < 1e-15


def test_gelu_uses_the_pages_constant(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "page_constants.json")))
    k = g["gelu_inv_sqrt2"]["value"]
    assert abs(k - math.sqrt(0.5)) <= 2.3e-16
    v = 0.8
    assert abs(oracle.gelu(v, "f64") - 0.5 * v * (1 + math.erf(v * k))) < 1e-16


# ------------------------------------------------------------------------ attention

def test_attention_single_key_returns_its_value():
    r = _rng(7)
    H, G, d = 4, 2, 64
    q = r.standard_normal((H, d))
    k = r.standard_normal((1, G, d))
    v = r.standard_normal((1, G, d))
    out = oracle.gqa_attention(q, k, v, "f64")
    out32 = oracle.gqa_attention(q, k, v, "f32")
    assert np.array_equal(out32, out.astype(np.float32).astype(np.float64))
    for h in range(H):
        assert np.array_equal(out[h], v[0, h // (H // G)])


def test_attention_kv_head_mapping_is_consecutive_grouping():
    # q heads 0..2 read kv head 0, heads 3..5 read kv head 1 (kvh = head / group)
    H, G, d = 6, 2, 8
    q = np.zeros((H, d))
    k = np.zeros((1, G, d))
    v = np.stack([np.full(d, 10.0), np.full(d, -20.0)])[None]
    out = oracle.gqa_attention(q, k, v, "f64")
    assert np.all(out[:3] == 10.0) and np.all(out[3:] == -20.0)


def test_attention_probabilities_match_scipy_softmax():
    # with one-hot value rows the output is the probability vector itself
    r = _rng(8)
    for H, G, d, L in ((2, 1, 64, 5), (4, 2, 64, 33), (16, 8, 128, 64)):
        q = r.standard_normal((H, d)) * 2
        k = r.standard_normal((L, G, d))
        v = np.zeros((L, G, d))
        for j in range(L):
            v[j, :, j] = 1.0
        out = oracle.gqa_attention(q, k, v, "f64")
        for h in range(H):
            kv = h // (H // G)
            p = sps.softmax(q[h] @ k[:, kv, :].T / math.sqrt(d))
            assert np.allclose(out[h, :L], p, rtol=1e-12, atol=1e-15)
        out32 = oracle.gqa_attention(q, k, v, "f32")
        assert np.allclose(out32, out, atol=64 * U32 * max(1.0, float(np.abs(q).max()) ** 2))


def test_attention_equal_keys_average_values():
    r = _rng(9)
    L, d = 10, 64
    q = r.standard_normal((2, d))
    k = np.repeat(r.standard_normal((1, 1, d)), L, axis=0)
    v = r.standard_normal((L, 1, d))
    out = oracle.gqa_attention(q, k, v, "f64")
    assert np.allclose(out[0], v[:, 0].mean(axis=0), atol=1e-14)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    r = _rng(10)
    H, G, d, L = 6, 2, 64, 21
    q = r.standard_normal((H, d))
    k = r.standard_normal((L, G, d))
    v = r.standard_normal((L, G, d))
    out = oracle.gqa_attention(q, k, v)
    kd = np.repeat(k, H // G, axis=1)
    vd = np.repeat(v, H // G, axis=1)
    assert np.array_equal(out, oracle.gqa_attention(q, kd, vd))


def _ring_brute(q, kr, vr, pr, window, pos, prec="f32"):
    # legal keys gathered in ascending slot order, then plain MHA attention over them
    legal = [j for j in range(len(pr))
             if pr[j] != oracle.INVALID_POS and pr[j] <= pos and pos - pr[j] < window]
    H, d = q.shape
    return oracle.gqa_attention(q, kr[legal], vr[legal], prec) if legal else np.zeros((H, d))


def test_ring_attention_masks_by_stamp_and_window(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "page_constants.json")))
    assert g["invalid_pos"]["value"] == oracle.INVALID_POS
    r = _rng(11)
    ring, H, d = 12, 2, 64
    for trial in range(20):
        pos = int(r.integers(0, 40))
        pr = r.integers(0, 45, size=ring).astype(np.uint32)
        pr[r.random(ring) < 0.3] = oracle.INVALID_POS
        pr[int(r.integers(0, ring))] = pos           # the key just pushed is always legal
        window = int(r.integers(1, ring + 1))
        q = r.standard_normal((H, d))
        kr = r.standard_normal((ring, H, d))
        vr = r.standard_normal((ring, H, d))
        # the codec page divides the value sum by the denominator at the end, the talker
        # page divides each weight first: equal in exact arithmetic, not in f32 rounding
        out = oracle.ring_attention(q, kr, vr, pr, window, pos, "f64")
        assert np.allclose(out, _ring_brute(q, kr, vr, pr, window, pos, "f64"),
                           rtol=0, atol=1e-13), trial
        out = oracle.ring_attention(q, kr, vr, pr, window, pos)
        assert np.allclose(out, _ring_brute(q, kr, vr, pr, window, pos),
                           rtol=0, atol=2e-6), trial


def test_ring_attention_empty_ring_first_step_returns_value():
    r = _rng(12)
    ring, H, d = 250, 8, 64
    pr = np.full(ring, oracle.INVALID_POS, np.uint32)
    pr[0] = 0
    q = r.standard_normal((H, d)).astype(np.float32)
    kr = r.standard_normal((ring, H, d)).astype(np.float32)
    vr = r.standard_normal((ring, H, d)).astype(np.float32)
    out = oracle.ring_attention(q, kr, vr, pr, 250, 0)
    assert np.array_equal(out, vr[0].astype(np.float64))


def test_unbounded_window_is_plain_causal_attention():
    """window = ring >= every position (the FlowLM backbone): nothing is masked but the empty
    slots, so ring attention equals plain attention over the filled history."""
    r = _rng(13)
    ring, H, d, L = 40, 4, 64, 29
    pr = np.full(ring, oracle.INVALID_POS, np.uint32)
    pr[:L] = np.arange(L)
    q = r.standard_normal((H, d)).astype(np.float32)
    kr = r.standard_normal((ring, H, d)).astype(np.float32)
    vr = r.standard_normal((ring, H, d)).astype(np.float32)
    got = oracle.ring_attention(q, kr, vr, pr, ring, L - 1, "f64")
    want = oracle.gqa_attention(q, kr[:L], vr[:L], "f64")
    assert np.max(np.abs(got - want)) < 1e-12


# ------------------------------------------------------------------------ the stack

def _f32(a):
    return np.asarray(a, dtype=np.float32)


def _talker_by_primitives(syn, x_in, pos, kv):
    """Compose one talker step from individually pinned oracle primitives in the order of
    the talker's step plan.  kv[l] = (K list, V list) of earlier positions (mutated)."""
    w = syn.workload
    d, H, G = w.head_dim, w.q_heads, w.kv_heads
    x = _f32(x_in)
    for l, L in enumerate(syn.layers):
        n = _f32(oracle.rms_norm(x, L["in_norm"], w.norm_eps))
        q = _f32(oracle.matvec(L["wq"], n)).reshape(H, d)
        k = _f32(oracle.matvec(L["wk"], n)).reshape(G, d)
        v = _f32(oracle.matvec(L["wv"], n)).reshape(G, d)
        q = np.stack([_f32(oracle.rms_norm(q[i], L["q_norm"], w.norm_eps)) for i in range(H)])
        k = np.stack([_f32(oracle.rms_norm(k[i], L["k_norm"], w.norm_eps)) for i in range(G)])
        c, s = oracle.rope_table(d, w.rope_theta, pos)
        q = np.stack([_f32(oracle.rope_rotate_half(q[i], c, s)) for i in range(H)])
        k = np.stack([_f32(oracle.rope_rotate_half(k[i], c, s)) for i in range(G)])
        kv[l][0].append(k)
        kv[l][1].append(v)
        att = _f32(oracle.gqa_attention(q, np.stack(kv[l][0]), np.stack(kv[l][1])))
        x = x + _f32(oracle.matvec(L["wo"], att.reshape(-1)))
        n = _f32(oracle.rms_norm(x, L["post_norm"], w.norm_eps))
        gt = _f32(oracle.matvec(L["wgate"], n))
        up = _f32(oracle.matvec(L["wup"], n))
        a = _f32([oracle.silu(float(t)) for t in gt]) * up
        x = x + _f32(oracle.matvec(L["wdown"], a))
    return _f32(oracle.rms_norm(x, syn.final_norm, w.norm_eps))


def test_prefill_is_causal_steps_of_pinned_primitives():
    """A prefill block of n rows: row r is the page-order step at position len + r, attending to
    every earlier key including the block's own earlier rows (causal within the block)."""
    w = W.TALKER_H256_L1
    syn = W.generate(w)
    syn.max_pos = 40
    m = oracle.OracleModel(syn)
    x = np.random.default_rng(5).standard_normal((4, w.hidden)).astype(np.float32)
    got = m.prefill(0, x)
    kv = [([syn.prefill_k[0][l, p] for p in range(32)], [syn.prefill_v[0][l, p] for p in range(32)])
          for l in range(w.layers)]
    for r in range(4):
        want = _talker_by_primitives(syn, x[r], 32 + r, kv)
        assert np.array_equal(got[r], want.astype(np.float64)), r
    assert m.length(0) == 36
    with pytest.raises(ValueError):  # 36 + 5 > max_pos
        m.prefill(0, np.zeros((5, w.hidden), np.float32))


def test_flowlm_head_is_layer_norm_then_eos_of_pinned_primitives():
    """The FlowLM backbone's head: the step output is out_norm(x) of the last layer's residual
    stream (the last tap) and the EOS logit is eos_w . out plus its bias."""
    w = W.SMALL_FLOWLM
    syn = W.generate(w)
    m = oracle.OracleModel(syn)
    hd = syn.head
    for t in range(3):
        pos = [m.length(s) for s in range(w.streams)]
        out, taps = m.step(syn.inputs[t], pos, taps=True)
        for s in range(w.streams):
            want = _f32(oracle.layer_norm(_f32(taps[-1][s]), hd["norm_w"], hd["norm_b"], w.norm_eps))
            assert np.array_equal(out[s], want.astype(np.float64))
            e = np.float32(0)
            for i in range(w.hidden):  # ascending, in f32
                e = np.float32(e + np.float32(hd["eos_w"][i]) * np.float32(want[i]))
            assert m.eos(s) == float(e) + float(hd["eos_b"][0])


def test_missing_layer_scale_is_a_scale_of_one():
    """A codec layer without LayerScale (FlowLM) equals one with LayerScale vectors of ones."""
    import dataclasses
    syn = W.generate(W.SMALL_FLOWLM)
    ones = dataclasses.replace(syn, layers=[dict(d, ls1=np.ones(W.SMALL_FLOWLM.hidden, np.float32),
                                                 ls2=np.ones(W.SMALL_FLOWLM.hidden, np.float32))
                                            for d in syn.layers])
    a, b = oracle.OracleModel(syn), oracle.OracleModel(ones)
    for t in range(3):
        pos = [a.length(s) for s in range(W.SMALL_FLOWLM.streams)]
        assert np.array_equal(a.step(syn.inputs[t], pos), b.step(syn.inputs[t], pos))


def test_matvec_bias_starts_the_accumulator_at_the_bias():
    """MV_BIAS (Pocket TTS on wgpu, the flow head): acc = b[n], then acc += w[n,k] x[k] in
    ascending k, each step rounded to float32; act = 1 passes the sum through SiLU."""
    r = _rng(31)
    N, K = 7, 23
    W = r.standard_normal((N, K)).astype(np.float32)
    b = (100.0 * r.standard_normal(N)).astype(np.float32)   # large: the order shows in the bits
    x = r.standard_normal(K).astype(np.float32)
    want = np.empty(N, np.float32)
    for n in range(N):
        acc = np.float32(b[n])
        for k in range(K):
            acc = np.float32(acc + np.float32(W[n, k] * x[k]))
        want[n] = acc
    got = oracle.matvec_bias(W, x, b)
    assert np.array_equal(got, want.astype(np.float64))
    # the bias-last order rounds differently on at least one row of this case
    last = (_f32(oracle.matvec(W, x)) + b).astype(np.float64)
    assert not np.array_equal(got, last)
    s = oracle.matvec_bias(W, x, b, act=1)
    assert np.array_equal(s, np.array([oracle.silu(float(v)) for v in want], np.float64))


def _flow_by_primitives(f, d, cond, noise):
    """The flow head's LSD step composed from individually pinned oracle primitives, one
    float32 rounding per operation, in the order of the page's dispatch plan."""
    f32 = np.float32
    sil = lambda v: _f32([oracle.silu(float(t)) for t in v])
    mvb = lambda w, x, b, act=0: _f32(oracle.matvec_bias(w, x, b, act))
    x = mvb(d["ip_w"], noise, d["ip_b"])
    y = sil(d["t_const"] + mvb(d["cond_w"], cond, d["cond_b"]))
    D = f.dim
    for i in range(f.blocks):
        m = mvb(d[f"ada_w{i}"], y, d[f"ada_b{i}"])
        u = _f32(oracle.layer_norm(x, d[f"ln_w{i}"], d[f"ln_b{i}"], f.ln_eps))
        u = u * (f32(1) + m[D:2 * D]) + m[:D]
        h = mvb(d[f"m0_w{i}"], u, d[f"m0_b{i}"], 1)
        x = x + m[2 * D:] * mvb(d[f"m2_w{i}"], h, d[f"m2_b{i}"])
    m = mvb(d["fada_w"], y, d["fada_b"])
    u = _f32(oracle.layer_norm(x, np.ones(D, np.float32), np.zeros(D, np.float32), f.ln_eps))
    u = u * (f32(1) + m[D:]) + m[:D]
    return noise + mvb(d["f_w"], u, d["f_b"]) * f32(1)


def test_flow_head_adaln_wiring_closed_form():
    """The page fixes the fused adaLN projection as [shift | scale | gate], modulate as
    x (1 + scale) + shift, the gate on the third chunk multiplying the block's MLP branch, and a
    final [shift | scale] over a LayerNorm WITHOUT affine weights (Pocket TTS on wgpu,
    PocketFlowGpu::new, MODULATE, GATED_ADD).  With zero projection matrices every chunk is its
    bias, with identity MLP matrices the branch is silu(modulate(LN(x0))), and with a selection
    matrix as the final linear the output is closed-form in float64: no value below comes from
    the oracle.  Shift, scale and gate are distinct, so any swap or dropped term moves it."""
    D, Lt, C_ = 12, 5, 9
    r = _rng(41)
    x0 = r.standard_normal(D).astype(np.float32)
    shift = (0.3 * r.standard_normal(D)).astype(np.float32)
    scale = (0.5 + 0.3 * r.standard_normal(D)).astype(np.float32)
    gate = (-0.7 + 0.2 * r.standard_normal(D)).astype(np.float32)
    fshift = (0.2 * r.standard_normal(D)).astype(np.float32)
    fscale = (-0.4 + 0.2 * r.standard_normal(D)).astype(np.float32)
    lnw = (1.0 + 0.3 * r.standard_normal(D)).astype(np.float32)
    lnb = (0.2 * r.standard_normal(D)).astype(np.float32)
    sel = np.zeros((Lt, D), np.float32)
    sel[np.arange(Lt), 2 * np.arange(Lt)] = 1.0            # out j reads feature 2 j
    z = lambda *s: np.zeros(s, np.float32)
    d = {"ip_w": z(D, Lt), "ip_b": x0, "cond_w": z(D, C_), "cond_b": z(D),
         "t_const": r.standard_normal(D).astype(np.float32),
         "ada_w0": z(3 * D, D), "ada_b0": np.concatenate([shift, scale, gate]),
         "ln_w0": lnw, "ln_b0": lnb,
         "m0_w0": np.eye(D, dtype=np.float32), "m0_b0": z(D),
         "m2_w0": np.eye(D, dtype=np.float32), "m2_b0": z(D),
         "fada_w": z(2 * D, D), "fada_b": np.concatenate([fshift, fscale]),
         "f_w": sel, "f_b": z(Lt)}
    import dataclasses
    f = dataclasses.replace(W.SMALL_FLOW, dim=D, latent=Lt, cond=C_, blocks=1)
    noise = r.standard_normal(Lt).astype(np.float32)
    cond = r.standard_normal(C_).astype(np.float32)
    got = oracle.flow_step(f, d, cond, noise)

    e = np.float64
    eps = f.ln_eps

    def ln(v):
        v = v.astype(e)
        mu = v.mean()
        return (v - mu) / np.sqrt(((v - mu) ** 2).mean() + eps)

    silu = lambda v: v / (1.0 + np.exp(-v))
    u = ln(x0) * lnw.astype(e) + lnb.astype(e)                  # affine block LayerNorm
    u = u * (1.0 + scale.astype(e)) + shift.astype(e)            # modulate
    x1 = x0.astype(e) + gate.astype(e) * silu(u)                 # identity m0 (SiLU), m2, gate
    v = ln(x1) * (1.0 + fscale.astype(e)) + fshift.astype(e)     # final: no affine weights
    want = noise.astype(e) + v[2 * np.arange(Lt)]
    assert np.max(np.abs(got - want)) <= 2e-6 * (1.0 + np.max(np.abs(want)))


def test_flow_head_is_the_page_order_of_pinned_primitives():
    f = W.SMALL_FLOW
    d = W.generate_flow(f)
    for c in range(2):
        got = oracle.flow_step(f, d, d["cond"][c], d["noise"][c])
        want = _flow_by_primitives(f, d, d["cond"][c], d["noise"][c])
        assert np.array_equal(got, want.astype(np.float64)), c


def test_flow_head_with_zero_gates_skips_its_blocks():
    """adaLN-Zero: with every gate zero the blocks leave x as input_proj made it, so the step
    equals the head with no blocks."""
    import dataclasses
    f = W.SMALL_FLOW
    d = W.generate_flow(f)
    for i in range(f.blocks):
        d[f"ada_w{i}"][2 * f.dim:] = 0
        d[f"ada_b{i}"][2 * f.dim:] = 0
    none = dataclasses.replace(f, blocks=0)
    a = oracle.flow_step(f, d, d["cond"][0], d["noise"][0])
    b = oracle.flow_step(none, d, d["cond"][0], d["noise"][0])
    assert np.array_equal(a, b)
    # and with a zero final linear the step returns the noise plus the final bias
    d["f_w"][:] = 0
    out = oracle.flow_step(f, d, d["cond"][0], d["noise"][0])
    assert np.array_equal(out, (d["noise"][0] + d["f_b"]).astype(np.float64))


def test_talker_step_is_the_page_order_of_pinned_primitives():
    w = W.TALKER_H256_L1
    syn = W.generate(w)
    m = oracle.OracleModel(syn)
    kv = [([syn.prefill_k[0][l, p] for p in range(32)], [syn.prefill_v[0][l, p] for p in range(32)])
          for l in range(w.layers)]
    want = _talker_by_primitives(syn, syn.inputs[0, 0], 32, kv)
    got = m.step(syn.inputs[0], [32])
    assert np.array_equal(got[0], want.astype(np.float64))
    # the appended K row is the normed, roped key
    k, v = m.read_kv(0, 0, 32)
    assert np.array_equal(k, kv[0][0][32].astype(np.float64))


def _codec_by_primitives(syn, x_in, pos, hist):
    """One codec step from pinned primitives, keeping an explicit position -> (k, v)
    history instead of a ring; attention runs over the last `window` positions."""
    w = syn.workload
    D, H, d = w.hidden, w.q_heads, w.head_dim
    x = _f32(x_in)
    for l, L in enumerate(syn.layers):
        hb = _f32(oracle.layer_norm(x, L["ln1_w"], L["ln1_b"], w.norm_eps))
        qkv = _f32(oracle.matvec(L["in_proj"], hb))
        q, k, v = qkv[:D].reshape(H, d), qkv[D:2 * D].reshape(H, d), qkv[2 * D:].reshape(H, d)
        c, s = oracle.rope_table(d, w.rope_theta, pos)
        q = np.stack([_f32(oracle.rope_interleaved(q[i], c, s)) for i in range(H)])
        k = np.stack([_f32(oracle.rope_interleaved(k[i], c, s)) for i in range(H)])
        hist[l][pos] = (k, v)
        keys = [p for p in sorted(hist[l]) if p <= pos and pos - p < w.window]
        # ring slot order = ascending (p mod ring); attention is order-independent up to
        # rounding, so compare this part with a tolerance
        keys.sort(key=lambda p: p % w.ring)
        att = _f32(oracle.gqa_attention(q, np.stack([hist[l][p][0] for p in keys]),
                                        np.stack([hist[l][p][1] for p in keys])))
        o = _f32(oracle.matvec(L["out_proj"], att.reshape(-1)))
        x = x + _f32(L["ls1"]) * o
        hb = _f32(oracle.layer_norm(x, L["ln2_w"], L["ln2_b"], w.norm_eps))
        f = _f32([oracle.gelu(float(t)) for t in oracle.matvec(L["lin1"], hb)])
        x = x + _f32(L["ls2"]) * _f32(oracle.matvec(L["lin2"], f))
    return x


def test_codec_steps_match_history_model_across_ring_wraps():
    w = W.SMALL_CODEC                       # ring 20, window 17, 45 steps: two wraps
    syn = W.generate(w)
    m = oracle.OracleModel(syn)
    hist = [[{}, {}] for _ in range(w.layers)]
    for s in range(w.streams):
        for l in range(w.layers):
            for p in range(syn.lengths[s]):
                hist[l][s][p] = (syn.prefill_k[s][l, p], syn.prefill_v[s][l, p])
    for t in range(w.steps):
        pos = [m.length(s) for s in range(w.streams)]
        got = m.step(syn.inputs[t], pos)
        for s in range(w.streams):
            want = _codec_by_primitives(syn, syn.inputs[t, s], pos[s],
                                        [hist[l][s] for l in range(w.layers)])
            assert np.allclose(got[s], want, rtol=0, atol=2e-6), (t, s)


def test_stack_with_zero_matrices_passes_the_residual_through():
    for base in (W.SMALL_TALKER_F32, W.SMALL_CODEC):
        syn = W.generate(base)
        for L in syn.layers:
            for name, a in L.items():
                if a.ndim == 2:
                    L[name] = np.zeros_like(a)
        m = oracle.OracleModel(syn)
        x = syn.inputs[0]
        out = m.step(x, [m.length(s) for s in range(base.streams)])
        for s in range(base.streams):
            if base.kind == "talker":
                want = oracle.rms_norm(x[s], syn.final_norm, base.norm_eps)
            else:
                want = x[s].astype(np.float64)
            assert np.array_equal(out[s], want)


def test_streams_are_independent_and_thread_count_is_irrelevant():
    w = W.SMALL_TALKER_BF16
    syn = W.generate(w)
    both = oracle.OracleModel(syn, threads=4)
    outs = [both.step(syn.inputs[t], [both.length(s) for s in range(w.streams)])
            for t in range(3)]
    for s in range(w.streams):
        alone = oracle.OracleModel(syn, threads=1)
        for t in range(3):
            x = np.zeros((w.streams, w.hidden), np.float32)
            x[: s + 1] = syn.inputs[t, : s + 1]
            got = alone.step(x[: s + 1], [alone.length(i) for i in range(s + 1)])
            assert np.array_equal(got[s], outs[t][s])
    oracle.set_threads(1)


def test_f32_oracle_tracks_f64_shadow():
    syn = W.generate(W.SMALL_TALKER_F32)
    a = oracle.OracleModel(syn, "f32")
    b = oracle.OracleModel(syn, "f64")
    for t in range(3):
        pos = [a.length(s) for s in range(syn.workload.streams)]
        ya, yb = a.step(syn.inputs[t], pos), b.step(syn.inputs[t], pos)
        assert np.max(np.abs(ya - yb)) < 2e-5


def test_step_rejects_wrong_position_and_capacity():
    syn = W.generate(W.TALKER_H256_L1)
    m = oracle.OracleModel(syn)
    with pytest.raises(ValueError):
        m.step(syn.inputs[0], [31])
    m.step(syn.inputs[0], [32])
    with pytest.raises(ValueError):          # max_pos = 33 positions
        m.step(syn.inputs[0], [33])
