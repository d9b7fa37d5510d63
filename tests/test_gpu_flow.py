"""The flow head (dec_flow_*) on the GPU against the CPU oracle's flow_step, for a small ragged
shape and the full one, and conditioned in place on a FlowLM backbone step's hidden state."""
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


@pytest.mark.parametrize("shape", [W.SMALL_FLOW, W.FLOW_D512], ids=lambda f: f.name)
def test_flow_head_matches_oracle(D, shape):
    d = W.generate_flow(shape, calls=4)
    head = D.FlowHead(shape, d)
    assert head.kernels_per_step() == 3 + 2 * shape.blocks + 1
    st = Stats()
    cond = torch.from_numpy(d["cond"]).cuda()
    noise = torch.from_numpy(d["noise"]).cuda()
    for c in range(4):
        got = head.step(cond[c], noise[c]).cpu().numpy()
        want = oracle.flow_step(shape, d, d["cond"][c], d["noise"][c])
        check_rows(got, want, False, st, f"{shape.name} call {c}")
    # a second pass over the same buffers replays the captured graph
    got = head.step(cond[0], noise[0]).cpu().numpy()
    check_rows(got, oracle.flow_step(shape, d, d["cond"][0], d["noise"][0]), False, st, "replay")
    print(f"{shape.name}: {st.line()}")


def test_flow_head_reads_the_backbone_hidden_in_place(D):
    """One generation frame: a FlowLM-shaped backbone step, then the flow head conditioned on
    the step's output buffer (no copy), against the oracle doing the same."""
    w = W.SMALL_FLOWLM
    syn = W.generate(w)
    shape = W.FlowShape(name="small_flow_on_backbone", dim=136, latent=24, cond=w.hidden,
                        blocks=2, seed=16)
    d = W.generate_flow(shape, calls=3)
    orc = oracle.OracleModel(syn)
    dec = D.Decoder.from_synthetic(syn)
    head = D.FlowHead(shape, d)
    hidden = torch.empty((w.streams, w.hidden), device="cuda")
    noise = torch.from_numpy(d["noise"]).cuda()
    st = Stats()
    for t in range(3):
        pos = dec.lengths()
        dec.step(torch.from_numpy(syn.inputs[t]).cuda(), pos, hidden)
        latent = head.step(hidden[0], noise[t]).cpu().numpy()   # row 0 of the step's output
        h_orc = orc.step(syn.inputs[t], pos)
        want = oracle.flow_step(shape, d, h_orc[0].astype(np.float32), d["noise"][t])
        check_rows(latent, want, False, st, f"frame {t}")
    dec.sync()
    print(f"backbone + flow head: {st.line()}")
