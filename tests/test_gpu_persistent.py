"""The persistent step kernel (DEC_FLAG_PERSISTENT: one cooperative launch per step of m <= 2
rows) against the default multi-kernel plan and against the CPU oracle.

Both plans split every GEMV, attention chunk and merge the same way inside a CTA, so their
outputs must agree bit for bit; the oracle comparison uses the same bounds as the other step
tests.  Steps of different widths are interleaved on one decoder, so the two plans also hand
the cache and the lengths to each other."""
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


def _widths(S, n):
    """Step widths 1, 2, ..., S, 1, 2, ... (each step covers streams 0..m-1)."""
    return [1 + t % S for t in range(n)]


@pytest.mark.parametrize("name", ["small_talker_f32", "small_talker_bf16", "small_codec",
                                  "small_flowlm"])
def test_persistent_equals_multikernel_bitwise(D, name):
    w = W.SMALL[name]
    syn = W.generate(w)
    a = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT)
    b = D.Decoder.from_synthetic(syn)
    for m in (1, 2):
        assert a.kernels_per_step(m) == 1, m
        assert b.kernels_per_step(m) == 6 * w.layers + 1, m
    for t, m in enumerate(_widths(w.streams, w.steps)):
        x = torch.from_numpy(syn.inputs[t][:m].copy()).cuda()
        pos = a.lengths(m)
        assert pos == b.lengths(m)
        ya, yb = a.step(x, pos), b.step(x, pos)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), (name, t, m, float((ya - yb).abs().max()))
    a.sync()
    b.sync()
    # the caches the two plans leave behind are identical as well
    for s in range(w.streams):
        n = a.lengths(w.streams)[s]
        if n:
            ka, va = a.read_kv(w.layers - 1, s, n - 1)
            kb, vb = b.read_kv(w.layers - 1, s, n - 1)
            assert np.array_equal(ka, kb) and np.array_equal(va, vb)


@pytest.mark.parametrize("persistent", [False, True])
@pytest.mark.parametrize("name", ["small_talker_f32", "small_talker_bf16", "small_codec"])
def test_interleaved_widths_match_oracle(D, name, persistent):
    """Steps of 1, 2, 3 streams in turn vs the oracle (with the persistent flag: persistent,
    persistent, multi-kernel)."""
    w = W.SMALL[name]
    syn = W.generate(w)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT if persistent else 0)
    bf16 = w.weight_dtype == "bf16"
    st = Stats()
    for t, m in enumerate(_widths(w.streams, w.steps)):
        pos = dec.lengths(m)
        assert pos == [orc.length(s) for s in range(m)]
        x = np.ascontiguousarray(syn.inputs[t][:m])
        got = dec.step(torch.from_numpy(x).cuda(), pos).cpu().numpy()
        want = orc.step(x, pos)
        check_rows(got, want, bf16, st, f"{name} step {t} m {m}")
    dec.sync()
    print(f"{name}: {st.line()}")


@pytest.mark.parametrize("name", ["talker_h256_l1_f32", "talker_h1024_l4_f32_feedback",
                                  "talker_h2048_l28_bf16", "codec_d512_l8_ring250"])
def test_full_workloads_bitwise_first_steps(D, name):
    w = W.WORKLOADS[name]
    n = min(w.steps, 6)
    syn = W.generate(w, steps=n)
    a = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT)
    b = D.Decoder.from_synthetic(syn)
    assert a.kernels_per_step(w.streams) == 1
    x = torch.from_numpy(syn.x0.copy()).cuda() if w.feedback else None
    e = torch.from_numpy(syn.e).cuda() if w.feedback else None
    for t in range(n):
        if not w.feedback:
            x = torch.from_numpy(syn.inputs[t]).cuda()
        pos = a.lengths(w.streams)
        ya, yb = a.step(x, pos), b.step(x, pos)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), (name, t, float((ya - yb).abs().max()))
        if w.feedback:
            x = ya + e  # the next input is the output plus the fixed offset
    a.sync()
    b.sync()
