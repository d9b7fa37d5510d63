"""Whole decode steps on the GPU (C ABI, CUDA-graph replay, the launch configuration the
benchmark times) against the CPU oracle on the same seeded inputs, step by step."""
import os

import numpy as np
import pytest

import oracle
from tts_autoregressive_decode_gb300 import workloads as W

from _parity import Stats, check_rows, cosine  # noqa: E402

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


def run_parity(D, w, steps=None, flags=0, taps=False, report=None, eos=False):
    """Run `steps` steps on both sides (each side feeds back its own output when the workload
    says so) and check every row of every step.  Returns the stats."""
    syn = W.generate(w, steps=steps)
    nsteps = w.steps if steps is None else steps
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn, flags=flags | (D.L.DEC_FLAG_TAPS if taps else 0))
    m = w.streams
    bf16 = w.weight_dtype == "bf16"
    st, st_delta = Stats(), Stats()
    x_gpu = x_orc = None
    if w.feedback:
        x_gpu = syn.x0.copy()
        x_orc = syn.x0.copy()
    xbuf = torch.empty((m, w.hidden), dtype=torch.float32, device="cuda")
    out = torch.empty_like(xbuf)
    for t in range(nsteps):
        pos = dec.lengths(m)
        assert pos == [orc.length(s) for s in range(m)]
        xg = x_gpu if w.feedback else syn.inputs[t]
        xo = x_orc if w.feedback else syn.inputs[t]
        xbuf.copy_(torch.from_numpy(np.ascontiguousarray(xg)))
        dec.step(xbuf, pos, out)
        if taps:
            want, want_taps = orc.step(xo, pos, taps=True)
        else:
            want = orc.step(xo, pos)
        got = out.cpu().numpy()
        check_rows(got, want, bf16, st, f"{w.name} step {t}")
        if w.kind == "codec" and not w.head:
            # the codec output is input + O(0.01) LayerScale terms: check the change as well
            check_rows(got - xg, want - xo.astype(np.float64), bf16, st_delta,
                       f"{w.name} step {t} delta")
        if eos:  # the FlowLM head's EOS logits, bias included
            ge = dec.read_eos(m)
            for s in range(m):
                assert abs(float(ge[s]) - orc.eos(s)) <= 5e-4, (t, s, float(ge[s]), orc.eos(s))
        if taps:
            for l in range(w.layers):
                check_rows(dec.read_tap(l, m), want_taps[l], bf16, None, f"{w.name} step {t} tap {l}")
        if w.feedback:
            x_gpu = (got + syn.e).astype(np.float32)
            x_orc = (want.astype(np.float32) + syn.e).astype(np.float32)
    dec.sync()
    if report is not None:
        report.append(f"{w.name}: {st.line()}" + (f" | delta {st_delta.line()}" if w.kind == "codec" else ""))
    return st, dec, orc, syn


@pytest.mark.parametrize("name", list(W.SMALL))
def test_small_workloads_every_step(D, name):
    rep = []
    run_parity(D, W.SMALL[name], taps=True, report=rep)
    print(rep[-1])


def test_talker_h256_l1(D):
    rep = []
    run_parity(D, W.TALKER_H256_L1, report=rep)
    print(rep[-1])


def test_talker_h1024_l4_feedback_64_steps(D):
    rep = []
    run_parity(D, W.TALKER_H1024_L4, report=rep)
    print(rep[-1])


def test_codec_d512_l8_600_steps_two_ring_wraps(D):
    rep = []
    st, dec, orc, syn = run_parity(D, W.CODEC_D512_L8, report=rep)
    print(rep[-1])
    # the ring holds the last 250 positions: position 599 sits in slot 599 % 250
    k, v = dec.read_kv(7, 0, 599)
    ko, vo = orc.read_kv(7, 0, 599)
    assert np.max(np.abs(k.reshape(-1) - ko.reshape(-1))) < 1e-3


def test_flowlm_d1024_l6_64_steps_with_eos(D):
    rep = []
    run_parity(D, W.FLOWLM_D1024_L6, report=rep, eos=True)
    print(rep[-1])


def test_small_flowlm_eos_every_step(D):
    rep = []
    run_parity(D, W.SMALL_FLOWLM, report=rep, eos=True)
    print(rep[-1])


def test_talker_h2048_l28_bf16_128_steps(D):
    rep = []
    run_parity(D, W.TALKER_H2048_L28, report=rep)
    print(rep[-1])


@pytest.mark.slow
def test_talker_h2048_l28_bf16_m8_every_step(D):
    # 8 streams, lengths U[512, 4096]: every row of all 64 steps against the oracle
    rep = []
    run_parity(D, W.TALKER_H2048_L28_M8, report=rep)
    print(rep[-1])


def test_talker_h2048_l28_bf16_m8_last_steps(D):
    # The same 8-stream stack brought to the last positions of its 64 steps directly: each
    # stream is prefilled to its length + 61, then steps 61..63 run on both sides.  The longest
    # stream passes 4096 positions here, and every stream crosses its own chunk boundaries.
    import dataclasses
    w = W.TALKER_H2048_L28_M8
    late = dataclasses.replace(w, name=w.name + "_last3", prefill_range=None,
                               prefill=tuple(n + 61 for n in W.prefill_lengths(w)), steps=3)
    assert W.max_pos(late) == W.max_pos(w) and max(late.prefill) + 2 >= 4096
    rep = []
    run_parity(D, late, report=rep)
    print(rep[-1])


def test_graph_replay_equals_direct_launches_bitwise(D):
    w = W.SMALL_TALKER_BF16
    syn = W.generate(w)
    a = D.Decoder.from_synthetic(syn)
    b = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_NO_GRAPH)
    c = D.Decoder.from_synthetic(syn)
    for t in range(w.steps):
        x = torch.from_numpy(syn.inputs[t]).cuda()
        pos = a.lengths()
        ya, yb, yc = a.step(x, pos), b.step(x, pos), c.step(x, pos)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb) and torch.equal(ya, yc), t


@pytest.mark.parametrize("name", ["small_talker_bf16", "small_codec"])
def test_one_graph_serves_changing_buffers_bitwise(D, name):
    """Inputs and outputs in a different buffer at every step (rotating pools of 3 and 2):
    the replayed graph with its pointers rewritten equals direct launches bit for bit, and
    every output lands in the buffer given for its step."""
    w = W.SMALL[name]
    syn = W.generate(w)
    a = D.Decoder.from_synthetic(syn)
    b = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_NO_GRAPH)
    m = w.streams
    xs = [torch.empty((m, w.hidden), device="cuda") for _ in range(3)]
    outs = [torch.full((m, w.hidden), float("nan"), device="cuda") for _ in range(2)]
    for t in range(w.steps):
        x = xs[t % 3]
        x.copy_(torch.from_numpy(syn.inputs[t]))
        o = outs[t % 2]
        o.fill_(float("nan"))
        pos = a.lengths()
        ya = a.step(x, pos, o)
        yb = b.step(x.clone(), pos)
        torch.cuda.synchronize()
        assert ya.data_ptr() == o.data_ptr()
        assert torch.equal(o, yb), (name, t)
    a.sync()
    b.sync()


@pytest.mark.parametrize("name", ["small_talker_f32", "small_talker_bf16"])
def test_attention_grid_choice_leaves_results_unchanged(D, name):
    """A small cache capacity gives the paired attention grid (two chunks per CTA, one wave);
    a capacity of thousands of positions gives one chunk per CTA.  Every chunk is computed the
    same way, so the two contexts agree bit for bit on the same steps."""
    w = W.SMALL[name]
    syn = W.generate(w)
    big = W.generate(w)
    big.max_pos = 64 * 2 * 160  # ceil(chunks / 2) * kv heads * streams > any SM count
    a = D.Decoder.from_synthetic(syn)
    b = D.Decoder.from_synthetic(big)
    for t in range(w.steps):
        x = torch.from_numpy(syn.inputs[t]).cuda()
        pos = a.lengths()
        ya, yb = a.step(x, pos), b.step(x, pos)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), (name, t)
    a.sync()
    b.sync()


def test_kv_append_matches_oracle(D):
    w = W.SMALL_TALKER_F32
    syn = W.generate(w, steps=2)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn)
    for t in range(2):
        pos = dec.lengths()
        dec.step(torch.from_numpy(syn.inputs[t]).cuda(), pos)
        orc.step(syn.inputs[t], pos)
        for s in range(w.streams):
            for l in range(w.layers):
                k, v = dec.read_kv(l, s, pos[s])
                ko, vo = orc.read_kv(l, s, pos[s])
                assert np.max(np.abs(k - ko)) < 1e-4 and np.max(np.abs(v - vo)) < 1e-4
                # a prefilled row is untouched
                if syn.lengths[s] > 0:
                    k0, _ = dec.read_kv(l, s, 0)
                    assert np.array_equal(k0, syn.prefill_k[s][l, 0])


def test_step_host_equals_step(D):
    w = W.SMALL_CODEC
    syn = W.generate(w, steps=4)
    a = D.Decoder.from_synthetic(syn)
    b = D.Decoder.from_synthetic(syn)
    for t in range(4):
        pos = a.lengths()
        ya = a.step(torch.from_numpy(syn.inputs[t]).cuda(), pos)
        yb = b.step_host(syn.inputs[t], pos)
        torch.cuda.synchronize()
        assert np.array_equal(ya.cpu().numpy(), yb)


def test_reset_and_prefill_restart_a_stream(D):
    w = W.SMALL_CODEC
    syn = W.generate(w, steps=6)
    dec = D.Decoder.from_synthetic(syn)
    x = torch.from_numpy(syn.inputs[0]).cuda()
    first = dec.step(x, dec.lengths()).clone()
    for t in range(1, 6):
        dec.step(torch.from_numpy(syn.inputs[t]).cuda(), dec.lengths())
    # restart both streams exactly as they were created
    dec.reset(0)
    dec.prefill_kv(1, D.to_device(syn.prefill_k[1], "cuda"), D.to_device(syn.prefill_v[1], "cuda"))
    assert dec.lengths() == [0, syn.lengths[1]]
    again = dec.step(x, dec.lengths())
    torch.cuda.synchronize()
    assert torch.equal(first, again)


def test_host_errors_leave_state_unchanged(D):
    w = W.TALKER_H256_L1
    syn = W.generate(w)
    dec = D.Decoder.from_synthetic(syn)
    x = torch.from_numpy(syn.inputs[0]).cuda()
    with pytest.raises(D.L.DecError) as e:
        dec.step(x, [31])
    assert e.value.status == D.L.DEC_E_POS
    assert dec.lengths() == [32]
    with pytest.raises(D.L.DecError) as e:
        dec.step(torch.empty((2, w.hidden), device="cuda"), [32, 0])
    assert e.value.status == D.L.DEC_E_ARG
    dec.step(x, [32])
    with pytest.raises(D.L.DecError) as e:   # max_pos = 33
        dec.step(x, [33])
    assert e.value.status == D.L.DEC_E_CAPACITY
    with pytest.raises(D.L.DecError) as e:
        dec.prefill_kv(0, torch.zeros((1, 40, 2, 64), device="cuda"),
                       torch.zeros((1, 40, 2, 64), device="cuda"))
    assert e.value.status == D.L.DEC_E_CAPACITY
    with pytest.raises(D.L.DecError) as e:
        dec.step(x, [33], out=x)               # output overlapping the input
    assert e.value.status in (D.L.DEC_E_ARG, D.L.DEC_E_CAPACITY)
    dec.sync()                                  # no device check fired


def test_runs_are_deterministic(D):
    w = W.SMALL_TALKER_F32
    outs = []
    for _ in range(2):
        syn = W.generate(w)
        dec = D.Decoder.from_synthetic(syn)
        ys = [dec.step(torch.from_numpy(syn.inputs[t]).cuda(), dec.lengths()).cpu()
              for t in range(w.steps)]
        outs.append(torch.stack(ys))
    assert torch.equal(outs[0], outs[1])
