"""ttt_linear_fwd_seqpar_noalloc: the sequence-parallel TTT-Linear forward for callers
that cannot allocate device memory while they run (the scratch is a fixed array
inside the library), checked through the C ABI against the workspace entry point
ttt_linear_fwd_seqpar on two calls in a row, against the fp64 oracle, and for the
error it returns when a split needs more than the fixed scratch.

Kept in a file of its own that collects last: the fixed array is shared by every
call in the process, so this also runs after all other GPU tests have used the
library."""
import pytest
import torch

from test_sequence_layers_gb300 import abi
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _dev(inp):
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    eta = inp.eta.to(dev) if inp.eta is not None else None
    return q, k, v, eta, inp.params["W0"].to(dev)


def _noalloc(inp):
    """One no-allocation call: outputs are preallocated here, before the call."""
    q, k, v, eta, W0 = _dev(inp)
    z = torch.empty_like(q)
    W = torch.empty((inp.B, inp.H, inp.d, inp.d), device=q.device)
    n0 = abi.ttt_launch_count()
    abi.ttt_linear_fwd_seqpar_noalloc(q, k, v, W0, z, W, inp.b, inp.causal, eta=eta,
                                      eta_scalar=inp.eta_scalar)
    abi.ttt_sync_status()
    return z, W, abi.ttt_launch_count() - n0


def _with_workspace(inp):
    q, k, v, eta, W0 = _dev(inp)
    z, W = abi.ttt_linear_fwd_seqpar(q, k, v, W0, inp.b, inp.causal, eta=eta,
                                     eta_scalar=inp.eta_scalar)
    abi.ttt_sync_status()
    return z, W


def _rel(a, b):
    return G.rel_err(a.double().cpu().numpy(), b.double().cpu().numpy())


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    first = G.synth.make("linear", B=1, H=4, T=2048, d=64, b=16, causal=True, eta="sigmoid", seed=700)
    second = G.synth.make("linear", B=2, H=3, T=1500, d=32, b=16, causal=True, eta=1.0, seed=701)
    for inp in (first, second):
        z, W, launches = _noalloc(inp)
        assert launches >= 2, "the problem was meant to run split"
        zr, Wr = _with_workspace(inp)
        assert _rel(z, zr) <= G.TOL_BF16 and _rel(W, Wr) <= G.TOL_BF16, (_rel(z, zr), _rel(W, Wr))
        zo, Wo = G.oracle_linear(inp)
        assert G.rel_err(z.double().cpu().numpy(), zo) <= G.TOL_BF16
        assert G.rel_err(W.double().cpu().numpy(), Wo) <= G.TOL_BF16
    # the array keeps the last call's contents; a repeat of the first problem is
    # unaffected by them
    z1, W1, _ = _noalloc(first)
    z2, W2, _ = _noalloc(first)
    assert torch.equal(z1, z2) and torch.equal(W1, W2)


def test_split_beyond_the_fixed_scratch_is_rejected():
    """16 chains of d = 64 over 4096 tokens split eight ways: maps and start weights
    take more than 4 MiB, so the call returns TTT_ERR_SCRATCH and queues nothing.
    The planner gives each chain at most (SMs / chains) segments, so eight segments
    (about 4.75 MiB of scratch) need at least 128 SMs; on a smaller GPU the split is
    coarser and fits, which says nothing about this entry point."""
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    if nsm < 128:
        pytest.skip(f"{nsm} SMs: the planner splits 16 chains fewer than eight ways")
    inp = G.synth.make("linear", B=1, H=16, T=4096, d=64, b=16, causal=True, seed=702)
    q, k, v, eta, W0 = _dev(inp)
    z = torch.empty_like(q)
    W = torch.empty((1, 16, 64, 64), device=q.device)
    n0 = abi.ttt_launch_count()
    with pytest.raises(abi.TTTError) as e:
        abi.ttt_linear_fwd_seqpar_noalloc(q, k, v, W0, z, W, 16)
    assert e.value.code == -6 and "scratch" in str(e.value)
    assert abi.ttt_launch_count() == n0
