"""Pins of the oracle's multimodal rope for the talker (Qwen3-TTS talker on wgpu, module notes:
the talker uses interleaved MRoPE, and with equal positions on its three axes it is the 1-D rope
with theta 1e6).

The pages give no section split, so the axis of each rope frequency is an input (an axis map).
The pins below hold for any map:
- equal positions on all axes give exactly the 1-D step (the pages' identity);
- a cached key differs from the 1-D key only by a rotation of each frequency pair through the
  angle its axis's offset gives (composition of plane rotations);
- attention scores depend only on per-axis position differences, so shifting every rotary
  position of a sequence by a constant per-axis offset leaves the outputs unchanged;
- bad maps and out-of-range positions are rejected without changing the state.
"""
import numpy as np
import pytest

import oracle
from tts_autoregressive_decode_gb300 import workloads as W


def interleaved_map(half, sections):
    """Round-robin t, h, w over the frequencies, h and w each limited to its section (the
    interleaved layout), every other frequency on t."""
    a = np.zeros(half, np.int32)
    for axis in (1, 2):
        for i in range(axis, min(half, 3 * sections[axis]), 3):
            a[i] = axis
    return a


def contiguous_map(half, sections):
    return np.repeat(np.arange(3, dtype=np.int32), sections)[:half]


def test_map_helpers_have_their_sections():
    a = interleaved_map(64, (24, 20, 20))
    assert [int((a == k).sum()) for k in range(3)] == [24, 20, 20]
    assert list(a[:6]) == [0, 1, 2, 0, 1, 2] and list(a[60:]) == [0, 0, 0, 0]
    b = contiguous_map(64, (16, 24, 24))
    assert list(b[15:17]) == [0, 1] and list(b[39:41]) == [1, 2]


@pytest.mark.parametrize("name", ["small_talker_f32", "small_talker_bf16"])
def test_uniform_positions_reduce_to_the_1d_step(name):
    w = W.SMALL[name]
    syn = W.generate(w)
    syn.max_pos = max(syn.max_pos, max(syn.lengths) + 8)
    a, b = oracle.OracleModel(syn), oracle.OracleModel(syn)
    half = w.head_dim // 2
    a.set_mrope(interleaved_map(half, (half - 2 * (half // 3), half // 3, half // 3)))
    for t in range(3):
        pos = [a.length(s) for s in range(w.streams)]
        r3 = np.repeat(np.array(pos, np.int32)[:, None], 3, axis=1)
        assert np.array_equal(a.step(syn.inputs[t], pos, rope_pos=r3), b.step(syn.inputs[t], pos))
    x = np.random.default_rng(1).standard_normal((3, w.hidden)).astype(np.float32)
    n0 = a.length(1)
    r3 = np.repeat(np.arange(n0, n0 + 3, dtype=np.int32)[:, None], 3, axis=1)
    assert np.array_equal(a.prefill(1, x, rope_pos=r3), b.prefill(1, x))


def test_cached_keys_turn_by_their_axis_offset():
    w = W.TALKER_H256_L1
    syn = W.generate(w, steps=1)
    syn.max_pos = max(syn.lengths) + 64
    d, half = w.head_dim, w.head_dim // 2
    amap = interleaved_map(half, (half - 2 * (half // 3), half // 3, half // 3))
    u = oracle.OracleModel(syn, precision="f64")
    m = oracle.OracleModel(syn, precision="f64")
    m.set_mrope(amap)
    p = u.length(0)
    r3 = np.array([[p + 3, p + 17, p + 40]], np.int32)
    x = syn.inputs[0][:1]
    u.step(x, [p])
    m.step(x, [p], rope_pos=r3)
    ku, vu = u.read_kv(0, 0, p)
    km, vm = m.read_kv(0, 0, p)
    assert np.array_equal(vu, vm)  # values carry no rope
    i = np.arange(half)
    phi = (r3[0][amap] - p) * w.rope_theta ** (-2.0 * i / d)
    c, s = np.cos(phi), np.sin(phi)
    want = np.concatenate([ku[:, :half] * c - ku[:, half:] * s, ku[:, half:] * c + ku[:, :half] * s],
                          axis=1)
    assert np.max(np.abs(km - want)) <= 1e-12 * np.max(np.abs(ku))
    # a map that swaps two axes turns the keys differently
    m2 = oracle.OracleModel(syn, precision="f64")
    m2.set_mrope(np.where(amap == 1, 2, np.where(amap == 2, 1, 0)).astype(np.int32))
    m2.step(x, [p], rope_pos=r3)
    assert np.max(np.abs(m2.read_kv(0, 0, p)[0] - km)) > 1e-3 * np.max(np.abs(ku))


def test_outputs_depend_only_on_per_axis_position_differences():
    w = W.SMALL_TALKER_F32
    syn = W.generate(w)
    syn.max_pos = max(syn.max_pos, 64)
    half = w.head_dim // 2
    amap = interleaved_map(half, (half - 2 * (half // 3), half // 3, half // 3))
    a = oracle.OracleModel(syn, precision="f64")
    b = oracle.OracleModel(syn, precision="f64")
    for o in (a, b):
        o.set_mrope(amap)
        o.reset(0)
    rng = np.random.default_rng(3)
    shift = np.array([7, 3, 12], np.int32)
    ya, yb = [], []
    for t in range(6):
        r3 = np.array([[t, (2 * t) % 5, 3 + (t > 2)]], np.int32)
        x = rng.standard_normal((1, w.hidden)).astype(np.float32)
        ya.append(a.step(x, [t], rope_pos=r3))
        yb.append(b.step(x, [t], rope_pos=r3 + shift))
    ya, yb = np.concatenate(ya), np.concatenate(yb)
    assert np.max(np.abs(ya - yb)) <= 1e-9 * np.max(np.abs(ya))
    # the same sequence without the rotary offsets is a different sequence
    c = oracle.OracleModel(syn, precision="f64")
    c.reset(0)
    rng = np.random.default_rng(3)
    yc = np.concatenate([c.step(rng.standard_normal((1, w.hidden)).astype(np.float32), [t])
                         for t in range(6)])
    assert np.max(np.abs(ya - yc)) > 1e-6 * np.max(np.abs(ya))


def test_bad_maps_and_positions_are_rejected():
    w = W.SMALL_TALKER_F32
    syn = W.generate(w)
    m = oracle.OracleModel(syn)
    half = w.head_dim // 2
    bad = np.zeros(half, np.int32)
    bad[5] = 3
    with pytest.raises(ValueError):
        m.set_mrope(bad)
    with pytest.raises(ValueError):
        m.set_mrope(np.zeros(half + 1, np.int32))
    m.set_mrope(np.zeros(half, np.int32))
    p = m.length(0)
    for r3 in ([[p, p, syn.max_pos]], [[p, -1, p]]):
        with pytest.raises(ValueError):
            m.step(syn.inputs[0][:1], [p], rope_pos=np.array(r3, np.int32))
        with pytest.raises(ValueError):
            m.prefill(0, syn.inputs[0][:1], rope_pos=np.array(r3, np.int32))
    assert m.length(0) == p
    codec = oracle.OracleModel(W.generate(W.SMALL_CODEC))
    with pytest.raises(ValueError):
        codec.set_mrope(np.zeros(W.SMALL_CODEC.head_dim // 2, np.int32))
    m.set_mrope(None)
    assert np.array_equal(m.step(syn.inputs[0], [m.length(s) for s in range(w.streams)]),
                          oracle.OracleModel(syn).step(syn.inputs[0], list(syn.lengths)))
