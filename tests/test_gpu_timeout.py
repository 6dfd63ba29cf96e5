"""The timeout path of the bounded on-chip waits, made to happen on the host's
request and without a GPU fault: ttt_debug_wait_limit makes the first consumer wait
of the b = 16 and full-batch TTT-Linear kernels, and of the full-batch TTT-MLP
kernel's elementwise warps, wait on a barrier that nothing arrives at, for a
millisecond.  The kernel must record the timeout, unwind (drain its
copies, free its tensor memory) and leave the context usable: ttt_sync_status reports
TTT_ERR_TIMEOUT, clears it, and the next normal call matches the oracle."""
import pytest
import torch

from test_sequence_layers_gb300 import abi
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000  # one millisecond


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _run(inp):
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    eta = inp.eta.to(dev) if inp.eta is not None else None
    return abi.ttt_linear_fwd(q, k, v, inp.params["W0"].to(dev), inp.b, inp.causal, eta=eta,
                              eta_scalar=inp.eta_scalar)


@pytest.mark.parametrize("kind", ["b16_causal", "b16_noncausal", "full_batch"])
def test_wait_timeout_is_reported_and_the_context_stays_usable(kind):
    if kind == "full_batch":
        inp = G.synth.make("linear", B=3, H=2, T=196, d=64, b=196, causal=False, eta="sigmoid", seed=1700)
    else:
        inp = G.synth.make("linear", B=2, H=3, T=600, d=64, b=16, causal=kind == "b16_causal",
                           eta="sigmoid", seed=1701)
    abi.ttt_sync_status()  # nothing pending before the test
    abi.ttt_debug_wait_limit(LIMIT_NS)
    try:
        _run(inp)
        with pytest.raises(abi.TTTError) as e:
            abi.ttt_sync_status()
        assert e.value.code == -5 and "timed out" in str(e.value)
    finally:
        abi.ttt_debug_wait_limit(0)
    abi.ttt_sync_status()  # the status word was cleared by the report
    z, W = _run(inp)
    abi.ttt_sync_status()
    zr, Wr = G.oracle_linear(inp)
    ez = G.rel_err(z.double().cpu().numpy(), zr)
    eW = G.rel_err(W.double().cpu().numpy(), Wr)
    assert ez <= G.TOL_BF16 and eW <= G.TOL_BF16, (ez, eW)


@pytest.mark.parametrize("ln", [False, True])
def test_mlp_full_batch_wait_timeout_unwinds(ln):
    """The full-batch tensor-memory MLP kernel: its elementwise warps give up first, stop
    arriving on barriers and raise the CTA's abort flag; the issuing thread leaves its
    loop at its next wait, drains the copies and products in flight, and the tensor
    memory is released.  Several chains per CTA, so the unwinding crosses chain
    boundaries; the next normal call matches the oracle."""
    import numpy as np
    import oracle
    B, H, T = 41, 8, 150
    inp = G.synth.make("mlp", B=B, H=H, T=T, d=64, m=256, b=T, causal=False, eta=0.1, seed=1710)
    dev = torch.device("cuda")
    P = [inp.params[n] for n in ("W1", "c1", "W2", "c2")]
    kw = {}
    if ln:
        g = torch.Generator().manual_seed(1711)
        kw = dict(ln_gamma=1.0 + 0.1 * torch.randn((H, 64), generator=g), ln_beta=0.1 * torch.randn((H, 64), generator=g))

    def run():
        return abi.ttt_mlp_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), *(x.to(dev) for x in P), T, False,
                               eta_scalar=inp.eta_scalar, **{k: v.to(dev) for k, v in kw.items()})
    abi.ttt_sync_status()
    abi.ttt_debug_wait_limit(LIMIT_NS)
    try:
        run()
        with pytest.raises(abi.TTTError) as e:
            abi.ttt_sync_status()
        assert e.value.code == -5 and "timed out" in str(e.value)
    finally:
        abi.ttt_debug_wait_limit(0)
    abi.ttt_sync_status()
    z, outs = run()
    abi.ttt_sync_status()
    zr, *Wr = oracle.mlp(inp.q, inp.k, inp.v, *P, T, False, eta_scalar=inp.eta_scalar, **kw)
    errs = [G.rel_err(z.double().cpu().numpy(), zr)] + [G.rel_err(o.double().cpu().numpy(), r) for o, r in zip(outs, Wr)]
    assert np.isfinite(zr).all() and max(errs) <= G.TOL_BF16, errs
