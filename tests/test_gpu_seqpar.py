"""Sequence-parallel TTT-Linear (affine maps of segments, scan, segment outputs)
against the fp64 oracle through the C ABI: several segments per chain, a ragged last
segment, per-token eta, per-batch initial weights, both masks, every supported head
dimension, and the long-context workload on every chain."""
import pytest
import torch

from test_sequence_layers_gb300 import abi
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _run(inp, per_batch_w0=False):
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    W0 = inp.params["W0"]
    if per_batch_w0:
        W0 = W0.expand(inp.B, *W0.shape).contiguous()
    eta = inp.eta.to(dev) if inp.eta is not None else None
    z, W = abi.ttt_linear_fwd_seqpar(q, k, v, W0.to(dev), inp.b, inp.causal, eta=eta,
                                     eta_scalar=inp.eta_scalar)
    abi.ttt_sync_status()
    return z.double().cpu().numpy(), W.double().cpu().numpy()


def _check(inp, chains=None, per_batch_w0=False):
    ws = abi.ttt_linear_seqpar_workspace(inp.B, inp.H, inp.T, inp.d, inp.b, inp.causal)
    assert ws > 0, "the case is meant to split"
    zg, Wg = _run(inp, per_batch_w0)
    zr, Wr = G.oracle_linear(inp, chains)
    if chains is not None:
        zg, Wg = G.pick(zg, chains), G.pick(Wg, chains)
    ez, eW = G.rel_err(zg, zr), G.rel_err(Wg, Wr)
    assert ez <= G.TOL_BF16 and eW <= G.TOL_BF16, (ez, eW)
    return ez, eW


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("T", [1000, 2000, 2048])
def test_segments_match_oracle(d, T):
    inp = G.synth.make("linear", B=1, H=2, T=T, d=d, b=16, causal=True, eta="sigmoid", seed=500 + d + T)
    _check(inp)


def test_more_than_two_segments_use_maps_and_scan():
    """Two chains over 4096 tokens split into more than two segments: the workspace
    holds affine maps (segments 1 .. P-2) besides the start weights, so the map role
    and the scan run; the result still matches the oracle."""
    d = 64
    ws = abi.ttt_linear_seqpar_workspace(1, 2, 4096, d, 16)
    start_weights_of_two = 2 * 1 * d * d * 4
    assert ws > start_weights_of_two, ws
    inp = G.synth.make("linear", B=1, H=2, T=4096, d=d, b=16, causal=True, eta="sigmoid", seed=560)
    _check(inp)


@pytest.mark.parametrize("causal", [True, False])
def test_segments_noncausal_and_per_batch_w0(causal):
    inp = G.synth.make("linear", B=2, H=3, T=1500, d=64, b=16, causal=causal, eta=1.0, seed=600 + causal)
    _check(inp, per_batch_w0=True)


@pytest.mark.parametrize("d,T,H", [(64, 1000, 2), (32, 2048, 2), (16, 1500, 3), (64, 4096, 2)])
def test_delta_rule_segments_match_oracle(d, T, H):
    """b = 1 (the delta rule, 16-token chunks with a forward substitution) cut into
    segments: the chunks are affine in the weights, so the state chain, the maps and the
    scan apply unchanged; two or more segments, ragged lengths, per-token eta."""
    inp = G.synth.make("linear", B=1, H=H, T=T, d=d, b=1, causal=True, eta="sigmoid", seed=650 + d + T)
    _check(inp)


def test_workload_125m_delta_rule_split_every_chain():
    """linear_125m_b1 (B1 H12 T2048 d64, b = 1) through the split, every chain."""
    inp = G.synth.workload("linear_125m_b1")
    ez, eW = _check(inp)
    print(f"linear_125m_b1 (split) rel err z {ez:.3e} W {eW:.3e}")


def test_split_equals_unsplit_up_to_rounding():
    """The split and the one-unit-per-chain path evaluate the same rule: outputs and
    final weights agree far inside the bf16 tolerance."""
    inp = G.synth.make("linear", B=1, H=4, T=1800, d=64, b=16, causal=True, eta="sigmoid", seed=610)
    zs, Ws = _run(inp)
    zp, Wp = G.gpu_linear(inp)
    assert G.rel_err(zs, zp) <= 1e-2 and G.rel_err(Ws, Wp) <= 1e-2


def test_workspace_too_small_is_rejected():
    inp = G.synth.make("linear", B=1, H=2, T=1024, d=64, b=16, causal=True, seed=620)
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    W0 = inp.params["W0"].to(dev)
    need = abi.ttt_linear_seqpar_workspace(1, 2, 1024, 64, 16)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(abi.TTTError) as e:
        abi.ttt_linear_fwd_seqpar(q, k, v, W0, 16, workspace=small)
    assert e.value.code == -1
    # W_out may not alias shared initial weights (they are read while it is written)
    Wpb = W0.expand(1, *W0.shape).contiguous()
    with pytest.raises(abi.TTTError):
        abi.ttt_linear_fwd_seqpar(q, k, v, Wpb, 16, W_out=Wpb)


def test_unsplit_problem_runs_the_plain_path():
    """Enough chains to fill the GPU: no workspace, same results as ttt_linear_fwd."""
    inp = G.synth.make("linear", B=16, H=12, T=128, d=64, b=16, causal=True, seed=630)
    assert abi.ttt_linear_seqpar_workspace(16, 12, 128, 64, 16) == 0
    zs, Ws = _run(inp)
    zp, Wp = G.gpu_linear(inp)
    assert (zs == zp).all() and (Ws == Wp).all()


def test_workload_long_context_gated_split_full():
    """B2 H32 T32768, per-token eta = sigmoid(g), on the split path: every chain over
    the whole sequence."""
    inp = G.synth.workload("linear_long_gated")
    ez, eW = _check(inp)
    print(f"linear_long_gated (split) rel err z {ez:.3e} W {eW:.3e}")


def test_dot_loss_runs_unsplit():
    """The negative dot-product loss has no serial chain to split: no workspace,
    and the entry point gives ttt_linear_fwd's results."""
    inp = G.synth.make("linear", B=1, H=2, T=1024, d=64, b=16, causal=True, seed=640)
    assert abi.ttt_linear_seqpar_workspace(1, 2, 1024, 64, 16, loss="dot") == 0
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    W0 = inp.params["W0"].to(dev)
    zs, Ws = abi.ttt_linear_fwd_seqpar(q, k, v, W0, 16, loss="dot")
    zp, Wp = abi.ttt_linear_fwd(q, k, v, W0, 16, loss="dot")
    abi.ttt_sync_status()
    assert torch.equal(zs, zp) and torch.equal(Ws, Wp)
