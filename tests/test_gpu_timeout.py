"""The timeout path of the bounded on-chip waits, made to happen on the host's
request and without a GPU fault: ttt_debug_wait_limit makes the first consumer wait
of the b = 16 and full-batch TTT-Linear kernels wait on a barrier that nothing
arrives at, for a millisecond.  The kernel must record the timeout, unwind (drain its
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
