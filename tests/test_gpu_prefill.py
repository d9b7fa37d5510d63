"""Batched causal prefill (dec_prefill) on the GPU against the CPU oracle's prefill (row r = the
step at position len + r), and against the same rows fed one step at a time on the GPU (chunk
invariance within the step tolerance).  Blocks of up to 8 rows; ragged tails; a stream other than
0; steps after the prefill continue from the appended cache."""
import os

import numpy as np
import pytest

import oracle
from tts_autoregressive_decode_gb300 import workloads as W

from _parity import Stats, check_rows  # noqa: E402

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tts_autoregressive_decode_gb300 import decoder, native_build
    native_build.build()
    oracle.set_threads(os.cpu_count() or 1)
    return decoder


def _rows(seed, n, h):
    return np.random.default_rng(seed).standard_normal((n, h)).astype(np.float32)


@pytest.mark.parametrize("name,n", [("small_talker_f32", 13), ("small_talker_bf16", 8),
                                    ("small_talker_bf16", 1), ("small_talker_f32", 3)])
def test_prefill_matches_oracle_then_steps_continue(D, name, n):
    w = W.SMALL[name]
    syn = W.generate(w)
    syn.max_pos = max(syn.max_pos, max(syn.lengths) + n + 4)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn)
    bf16 = w.weight_dtype == "bf16"
    st = Stats()
    s = 1                                     # not stream 0: the block's cache is its own
    x = _rows(7, n, w.hidden)
    base = dec.length(s)
    got = dec.prefill(s, torch.from_numpy(x).cuda()).cpu().numpy()
    want = orc.prefill(s, x)
    check_rows(got, want, bf16, st, f"{name} prefill n={n}")
    assert dec.length(s) == orc.length(s) == base + n
    # the appended rows are the step's keys: the next steps agree on every stream
    for t in range(2):
        pos = dec.lengths()
        assert pos == [orc.length(i) for i in range(w.streams)]
        xs = _rows(100 + t, w.streams, w.hidden)
        g = dec.step(torch.from_numpy(xs).cuda(), pos).cpu().numpy()
        check_rows(g, orc.step(xs, pos), bf16, st, f"{name} step {t} after prefill")
    dec.sync()
    print(f"{name} n={n}: {st.line()}")


def test_prefill_equals_single_steps_within_tolerance(D):
    """Chunk invariance: one 11-row prefill vs 11 one-row steps of the same stream."""
    w = W.SMALL_TALKER_BF16
    syn = W.generate(w)
    syn.max_pos = max(syn.max_pos, max(syn.lengths) + 16)
    a = D.Decoder.from_synthetic(syn)
    b = D.Decoder.from_synthetic(syn)
    x = _rows(3, 11, w.hidden)
    ya = a.prefill(0, torch.from_numpy(x).cuda()).cpu().numpy()
    yb = []
    for r in range(11):
        xb = torch.from_numpy(x[r: r + 1].copy()).cuda()
        yb.append(b.step(xb, b.lengths(1)).cpu().numpy()[0])
    yb = np.stack(yb)
    check_rows(ya, yb.astype(np.float64), True, None, "prefill vs steps")
    for l in range(w.layers):
        for p in (a.length(0) - 11, a.length(0) - 1):
            ka, va = a.read_kv(l, 0, p)
            kb, vb = b.read_kv(l, 0, p)
            assert np.max(np.abs(ka - kb)) <= 1e-4 * max(1.0, float(np.max(np.abs(kb))))
            assert np.max(np.abs(va - vb)) <= 1e-4 * max(1.0, float(np.max(np.abs(vb))))


def test_prefill_28_layer_bf16_at_2048(D):
    """The 28-layer bf16 talker: a 20-row block (8 + 8 + 4) after the 2048-position prefill."""
    w = W.TALKER_H2048_L28
    syn = W.generate(w, steps=2)
    syn.max_pos = 2048 + 24
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn)
    st = Stats()
    x = _rows(11, 20, w.hidden)
    got = dec.prefill(0, torch.from_numpy(x).cuda()).cpu().numpy()
    check_rows(got, orc.prefill(0, x), True, st, "28-layer prefill")
    print(f"28-layer prefill: {st.line()}")


def test_prefill_errors_leave_state_unchanged(D):
    syn = W.generate(W.SMALL_CODEC)
    dec = D.Decoder.from_synthetic(syn)
    x = torch.zeros((2, syn.workload.hidden), device="cuda")
    with pytest.raises(D.L.DecError) as e:
        dec.prefill(0, x)
    assert e.value.status == D.L.DEC_E_UNSUPPORTED
    syn = W.generate(W.SMALL_TALKER_F32)
    dec = D.Decoder.from_synthetic(syn)
    x = torch.zeros((syn.max_pos + 1, syn.workload.hidden), device="cuda")
    before = dec.lengths()
    with pytest.raises(D.L.DecError) as e:
        dec.prefill(0, x)
    assert e.value.status == D.L.DEC_E_CAPACITY
    with pytest.raises(D.L.DecError) as e:
        dec.prefill(syn.workload.streams, x[:1])
    assert e.value.status == D.L.DEC_E_ARG
    assert dec.lengths() == before
    dec.sync()
