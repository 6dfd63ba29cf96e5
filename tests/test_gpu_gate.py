"""The input-dependent inner learning rate on the GPU against the fp64 oracle,
element by element, through the C ABI; then the rate it writes driving TTT-Linear
against the oracle's layer fed with the oracle's own rate."""
import numpy as np
import pytest
import torch

import oracle
from test_sequence_layers_gb300 import abi, synth
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

# fp32 accumulation of exact bf16 products and an fp32 sigmoid: a few fp32 ulps of
# the rate
TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _gpu(x, theta, eta_base):
    eta = abi.ttt_eta_gate(x.cuda(), theta.cuda(), eta_base)
    abi.ttt_sync_status()
    return eta.double().cpu().numpy()


@pytest.mark.parametrize("B,T,H,dm", [(1, 1, 1, 8), (2, 75, 5, 64), (3, 130, 16, 200), (2, 33, 17, 24),
                                      (1, 200, 64, 72), (2, 64, 32, 2048), (1, 257, 33, 136)])
def test_gate_matches_oracle(B, T, H, dm):
    x, theta = synth.gate_inputs(B, T, H, dm, seed=B * 1000 + T + H + dm)
    for eta_base in (1.0, 0.1):
        got = _gpu(x, theta, eta_base)
        ref = oracle.eta_gate(x, theta, eta_base)
        assert got.shape == ref.shape
        err = np.abs(got - ref).max() / eta_base
        assert err <= TOL, err


def test_gate_zero_vectors_give_half_the_base_rate():
    x, _ = synth.gate_inputs(2, 70, 3, 64, seed=5)
    got = _gpu(x, torch.zeros(3, 64, dtype=torch.bfloat16), 0.1)
    assert np.all(got == np.float32(0.05))


def test_gate_empty_and_in_place_output():
    x, theta = synth.gate_inputs(2, 0, 4, 64, seed=1)
    assert abi.ttt_eta_gate(x.cuda(), theta.cuda()).shape == (2, 4, 0)
    x, theta = synth.gate_inputs(2, 40, 4, 64, seed=2)
    out = torch.full((2, 4, 40), -1.0, device="cuda")
    r = abi.ttt_eta_gate(x.cuda(), theta.cuda(), 1.0, eta=out)
    abi.ttt_sync_status()
    assert r.data_ptr() == out.data_ptr()
    np.testing.assert_allclose(out.double().cpu().numpy(), oracle.eta_gate(x, theta, 1.0), atol=TOL)


def test_gate_full_size_every_token():
    """The gated long workload's width (32 heads x 64 = 2048) over 2 x 32768 tokens,
    in the launch the benchmark times; every token against the oracle."""
    B, T, H, dm = 2, 32768, 32, 2048
    x, theta = synth.gate_inputs(B, T, H, dm, seed=77)
    got = _gpu(x, theta, 1.0)
    ref = oracle.eta_gate(x, theta, 1.0)
    err = np.abs(got - ref).max()
    print(f"eta_gate full size max abs err {err:.3e}")
    assert err <= TOL


@pytest.mark.parametrize("causal", [True, False])
def test_gate_feeds_ttt_linear(causal):
    """x -> eta (this kernel) -> TTT-Linear, against the oracle layer fed with the
    oracle's rate."""
    B, H, T, d, dm = 2, 4, 80, 64, 256
    inp = synth.make("linear", B=B, H=H, T=T, d=d, b=16, causal=causal, eta=1.0, seed=31)
    x, theta = synth.gate_inputs(B, T, H, dm, seed=32)
    eta = abi.ttt_eta_gate(x.cuda(), theta.cuda(), 1.0)
    z, W = abi.ttt_linear_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.params["W0"].cuda(), 16, causal,
                              eta=eta)
    abi.ttt_sync_status()
    zr, Wr = oracle.linear(inp.q, inp.k, inp.v, inp.params["W0"], 16, causal,
                           eta=oracle.eta_gate(x, theta, 1.0))
    assert G.rel_err(z.double().cpu().numpy(), zr) <= G.TOL_BF16
    assert G.rel_err(W.double().cpu().numpy(), Wr) <= G.TOL_BF16
