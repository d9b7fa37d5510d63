"""Multimodal rope of the talker (dec_set_mrope, dec_step_mrope, dec_prefill_mrope) on the GPU
against the CPU oracle with the same axis map and rotary positions.

Rows carry distinct t, h, w rotary positions (seeded, anywhere in 0..max_pos-1, unrelated to
the cache row); equal positions must give the 1-D step bit for bit; prefill blocks with ragged
tails; the persistent flag (steps with positions run the multi-kernel plan); the 28-layer bf16
talker at position 2048; a position outside the table is reported by the device check."""
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


def _axes(D, w):
    half = w.head_dim // 2
    return D.mrope_axes(w.head_dim, (half - 2 * (half // 3), half // 3, half // 3))


def _rope_pos(rng, rows, max_pos):
    return rng.integers(0, max_pos, size=(rows, 3)).astype(np.int32)


@pytest.mark.parametrize("name", ["small_talker_f32", "small_talker_bf16"])
def test_distinct_axis_positions_match_oracle(D, name):
    w = W.SMALL[name]
    syn = W.generate(w)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn)
    axes = _axes(D, w)
    orc.set_mrope(axes)
    dec.set_mrope(axes)
    bf16 = w.weight_dtype == "bf16"
    st = Stats()
    rng = np.random.default_rng(11)
    rp = torch.empty((w.streams, 3), dtype=torch.int32, device="cuda")  # one buffer, rewritten
    for t in range(w.steps):
        m = 1 + t % w.streams
        pos = dec.lengths(m)
        r3 = _rope_pos(rng, m, syn.max_pos)
        rp[:m].copy_(torch.from_numpy(r3))
        x = np.ascontiguousarray(syn.inputs[t][:m])
        got = dec.step(torch.from_numpy(x).cuda(), pos, rope_pos=rp[:m]).cpu().numpy()
        check_rows(got, orc.step(x, pos, rope_pos=r3), bf16, st, f"{name} step {t} m {m}")
    dec.sync()
    print(f"{name} mrope: {st.line()}")


def test_uniform_axis_positions_equal_the_1d_step_bitwise(D):
    w = W.SMALL_TALKER_BF16
    syn = W.generate(w)
    a = D.Decoder.from_synthetic(syn)
    b = D.Decoder.from_synthetic(syn)
    a.set_mrope(_axes(D, w))
    for t in range(w.steps):
        pos = a.lengths(w.streams)
        r3 = torch.tensor([[p, p, p] for p in pos], dtype=torch.int32, device="cuda")
        x = torch.from_numpy(syn.inputs[t]).cuda()
        ya = a.step(x, pos, rope_pos=r3)
        yb = b.step(x, pos)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), t
    a.sync()


@pytest.mark.parametrize("name,n", [("small_talker_f32", 13), ("small_talker_bf16", 8),
                                    ("small_talker_bf16", 3)])
def test_prefill_with_axis_positions_matches_oracle(D, name, n):
    w = W.SMALL[name]
    syn = W.generate(w)
    syn.max_pos = max(syn.max_pos, max(syn.lengths) + n + 4)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn)
    axes = _axes(D, w)
    orc.set_mrope(axes)
    dec.set_mrope(axes)
    bf16 = w.weight_dtype == "bf16"
    st = Stats()
    rng = np.random.default_rng(5 + n)
    x = rng.standard_normal((n, w.hidden)).astype(np.float32)
    r3 = _rope_pos(rng, n, syn.max_pos)
    got = dec.prefill(1, torch.from_numpy(x).cuda(),
                      rope_pos=torch.from_numpy(r3).cuda()).cpu().numpy()
    check_rows(got, orc.prefill(1, x, rope_pos=r3), bf16, st, f"{name} prefill n={n}")
    # the next steps (1-D rope again) read the appended keys
    for t in range(2):
        pos = dec.lengths(w.streams)
        xs = rng.standard_normal((w.streams, w.hidden)).astype(np.float32)
        g = dec.step(torch.from_numpy(xs).cuda(), pos).cpu().numpy()
        check_rows(g, orc.step(xs, pos), bf16, st, f"{name} step {t} after prefill")
    dec.sync()
    print(f"{name} mrope prefill n={n}: {st.line()}")


def test_persistent_flag_steps_with_positions_run_the_kernel_chain(D):
    w = W.SMALL_TALKER_BF16
    syn = W.generate(w)
    syn.max_pos = max(syn.max_pos, max(syn.lengths) + 10)
    a = D.Decoder.from_synthetic(syn, flags=D.L.DEC_FLAG_PERSISTENT)
    b = D.Decoder.from_synthetic(syn)
    axes = _axes(D, w)
    a.set_mrope(axes)
    b.set_mrope(axes)
    rng = np.random.default_rng(2)
    for t in range(8):
        m = 1 + t % 2
        pos = a.lengths(m)
        x = torch.from_numpy(np.ascontiguousarray(syn.inputs[t % w.steps][:m])).cuda()
        if t % 3 == 2:  # a plain step in between: the persistent plan, equal within rounding
            ya, yb = a.step(x, pos), b.step(x, pos)
            torch.cuda.synchronize()
            bound = 2e-3 * float(yb.abs().max())
            assert float((ya - yb).abs().max()) <= bound, t
        else:  # steps with positions take the kernel chain in both contexts: the same bits
            # until a plain step has appended cache rows that agree only within rounding
            r3 = torch.from_numpy(_rope_pos(rng, m, syn.max_pos)).cuda()
            ya, yb = a.step(x, pos, rope_pos=r3), b.step(x, pos, rope_pos=r3)
            torch.cuda.synchronize()
            if t < 2:
                assert torch.equal(ya, yb), t
            else:
                assert float((ya - yb).abs().max()) <= 2e-3 * float(yb.abs().max()), t
    a.sync()


def test_talker_h2048_l28_bf16_with_axis_positions(D):
    """The 28-layer bf16 talker after its 2048-position prefill: steps whose t axis follows the
    cache position and whose h / w axes hold other positions."""
    w = W.TALKER_H2048_L28
    syn = W.generate(w, steps=3)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn)
    axes = D.mrope_axes(w.head_dim, (24, 20, 20))
    orc.set_mrope(axes)
    dec.set_mrope(axes)
    st = Stats()
    for t in range(3):
        pos = dec.lengths(w.streams)
        r3 = np.array([[p, 17 + 5 * t, 2040 - t] for p in pos], np.int32)
        got = dec.step(torch.from_numpy(syn.inputs[t]).cuda(), pos,
                       rope_pos=torch.from_numpy(r3).cuda()).cpu().numpy()
        check_rows(got, orc.step(syn.inputs[t], pos, rope_pos=r3), True, st, f"28-layer step {t}")
    dec.sync()
    print(f"28-layer mrope: {st.line()}")


def test_errors_and_out_of_table_positions(D):
    w = W.SMALL_TALKER_F32
    syn = W.generate(w)
    dec = D.Decoder.from_synthetic(syn)
    half = w.head_dim // 2
    with pytest.raises(D.L.DecError) as e:
        dec.set_mrope([0] * (half + 1))
    assert e.value.status == D.L.DEC_E_ARG
    with pytest.raises(D.L.DecError) as e:
        dec.set_mrope([3] + [0] * (half - 1))
    assert e.value.status == D.L.DEC_E_ARG
    codec = D.Decoder.from_synthetic(W.generate(W.SMALL_CODEC))
    with pytest.raises(D.L.DecError) as e:
        codec.set_mrope([0] * (W.SMALL_CODEC.head_dim // 2))
    assert e.value.status == D.L.DEC_E_UNSUPPORTED
    x = torch.from_numpy(syn.inputs[0][:1]).cuda()
    with pytest.raises(ValueError):
        dec.step(x, dec.lengths(1), rope_pos=torch.zeros((1, 3), dtype=torch.int64, device="cuda"))
    # a position past the rope table: the row's attention is skipped and the check fires
    dec.set_mrope(_axes(D, w))
    p = dec.lengths(1)
    bad = torch.tensor([[p[0], syn.max_pos, 0]], dtype=torch.int32, device="cuda")
    dec.step(x, p, rope_pos=bad)
    with pytest.raises(D.L.DecError) as e:
        dec.sync()
    assert e.value.status == D.L.DEC_E_DEVICE_CHECK
    dec.sync()  # the check word was cleared: the context stays usable
