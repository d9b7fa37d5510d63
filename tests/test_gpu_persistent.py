"""The persistent streamed step (DEC_FLAG_PERSISTENT: one cooperative launch per step of m <= 2
rows) against the CPU oracle and against the chain of kernels, and its bounded waits.

The streamed kernel splits the GEMV rows, the attention keys and the merge differently from the
kernel chain, so the two plans agree within floating-point rounding, not bit for bit: both are
held to the oracle with the bounds of the other step tests.  Steps of different widths are
interleaved on one decoder, so the two plans also hand the cache and the lengths to each other."""
import os
import time

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
def test_interleaved_widths_match_oracle(D, name):
    """Steps of 1, 2, 3 streams in turn (persistent, persistent, kernel chain) vs the oracle,
    with the last step's cache rows and (FlowLM head) EOS logits checked as well."""
    w = W.SMALL[name]
    syn = W.generate(w)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT)
    for m in range(1, w.streams + 1):
        assert dec.kernels_per_step(m) == (1 if m <= 2 else 6 * w.layers + 1), m
    bf16 = w.weight_dtype == "bf16"
    st = Stats()
    for t, m in enumerate(_widths(w.streams, w.steps)):
        pos = dec.lengths(m)
        assert pos == [orc.length(s) for s in range(m)]
        x = np.ascontiguousarray(syn.inputs[t][:m])
        got = dec.step(torch.from_numpy(x).cuda(), pos).cpu().numpy()
        want = orc.step(x, pos)
        check_rows(got, want, bf16, st, f"{name} step {t} m {m}")
        if w.head:
            ge = dec.read_eos(m)
            for s in range(m):
                assert abs(float(ge[s]) - orc.eos(s)) <= 5e-4, (t, s)
        for s in range(m):  # the row the step appended (codec: its ring slot)
            k, v = dec.read_kv(w.layers - 1, s, pos[s])
            ko, vo = orc.read_kv(w.layers - 1, s, pos[s])
            assert np.max(np.abs(k.reshape(-1) - ko.reshape(-1))) <= 1e-3, (t, s)
            assert np.max(np.abs(v.reshape(-1) - vo.reshape(-1))) <= 1e-3, (t, s)
    dec.sync()
    print(f"{name}: {st.line()}")


@pytest.mark.parametrize("name", ["talker_h256_l1_f32", "talker_h1024_l4_f32_feedback",
                                  "talker_h2048_l28_bf16", "codec_d512_l8_ring250"])
def test_full_workloads_first_steps_match_oracle_and_chain(D, name):
    """The four one-stream workloads, first steps, persistent plan vs the oracle; the kernel
    chain on the same inputs agrees with it within the same bound."""
    w = W.WORKLOADS[name]
    n = min(w.steps, 6)
    syn = W.generate(w, steps=n)
    orc = oracle.OracleModel(syn)
    a = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT)
    b = D.Decoder.from_synthetic(syn)
    assert a.kernels_per_step(w.streams) == 1
    bf16 = w.weight_dtype == "bf16"
    sa, sb = Stats(), Stats()
    x = syn.x0.copy() if w.feedback else None
    for t in range(n):
        if not w.feedback:
            x = syn.inputs[t]
        pos = a.lengths(w.streams)
        xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        ya = a.step(xt, pos).cpu().numpy()
        yb = b.step(xt, pos).cpu().numpy()
        want = orc.step(x, pos)
        check_rows(ya, want, bf16, sa, f"{name} step {t} persistent")
        check_rows(yb, want, bf16, sb, f"{name} step {t} chain")
        if w.feedback:  # both sides feed the oracle's own output back
            x = (want.astype(np.float32) + syn.e).astype(np.float32)
    a.sync()
    b.sync()
    print(f"{name}: persistent {sa.line()} | chain {sb.line()}")


@pytest.mark.parametrize("phase_of", ["attention", "o-proj", "gate/up", "down", "next qkv",
                                      "output"])
def test_a_wait_that_runs_out_is_reported_and_the_context_recovers(D, phase_of):
    """A bounded wait made to run out (its consumers wait for a tag that no CTA writes): the
    kernel returns within the bound instead of hanging, dec_sync reports DEC_E_DEVICE_CHECK
    (wait limit), and after a rewind the next steps match the oracle again."""
    w = W.SMALL_TALKER_BF16
    syn = W.generate(w)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT)
    L = w.layers
    phase = {"attention": 1, "o-proj": 2, "gate/up": 3, "down": 4, "next qkv": 5,
             "output": 5 * L}[phase_of]
    bf16 = w.weight_dtype == "bf16"
    m = 2
    # one good step first, so that the failing one is not the plan's first launch
    pos = dec.lengths(m)
    x0 = np.ascontiguousarray(syn.inputs[0][:m])
    check_rows(dec.step(torch.from_numpy(x0).cuda(), pos).cpu().numpy(), orc.step(x0, pos), bf16)
    dec.sync()
    # the stalled step
    pos = dec.lengths(m)
    x1 = torch.from_numpy(np.ascontiguousarray(syn.inputs[1][:m])).cuda()
    dec.inject_stall(phase, polls=2000)
    t0 = time.perf_counter()
    dec.step(x1, pos)
    with pytest.raises(D.L.DecError) as e:
        dec.sync()
    waited = time.perf_counter() - t0
    assert e.value.status == D.L.DEC_E_DEVICE_CHECK and "wait-limit" in str(e.value)
    assert waited < 10.0, waited
    dec.sync()  # the check word was cleared
    # rewind the two streams and take the step again, then one more
    for s in range(m):
        dec.truncate(s, pos[s])
    for t in (1, 2):
        p = dec.lengths(m)
        assert p == [orc.length(s) for s in range(m)]
        x = np.ascontiguousarray(syn.inputs[t][:m])
        check_rows(dec.step(torch.from_numpy(x).cuda(), p).cpu().numpy(), orc.step(x, p), bf16,
                   None, f"after recovery, step {t}")
    dec.sync()


def test_stall_of_a_phase_without_waits_runs_normally(D):
    """Layer 0's q/k/v reads the step input, which it never waits for: a stall there changes
    nothing, and with a poll bound that the step's ordinary waits stay within, the step is
    correct."""
    w = W.SMALL_TALKER_F32
    syn = W.generate(w)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT)
    pos = dec.lengths(1)
    x = np.ascontiguousarray(syn.inputs[0][:1])
    dec.inject_stall(0, polls=200000)
    got = dec.step(torch.from_numpy(x).cuda(), pos).cpu().numpy()
    dec.sync()
    check_rows(got, orc.step(x, pos), False)
