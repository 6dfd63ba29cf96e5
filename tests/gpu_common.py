"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and
the fp64 oracle on the same seeded inputs, and compare with the relative metric
max|delta| / max|reference|."""
import numpy as np
import torch

import oracle
from test_sequence_layers_gb300 import abi, build, synth

# tolerances of the accuracy classes (relative to the reference's largest entry)
TOL_F32 = 1e-4    # fp32 operands
TOL_BF16 = 2e-2   # bf16 operands, fp32 accumulation and state


def ensure_built():
    build.build()
    abi.lib()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    assert np.isfinite(got).all(), "non-finite output"
    scale = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (scale if scale > 0 else 1.0))


def tol_for(inp):
    return TOL_F32 if inp.q.dtype == torch.float32 else TOL_BF16


def gpu_linear(inp, per_batch_w0=False, causal=None):
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    W0 = inp.params["W0"]
    if per_batch_w0:
        W0 = W0.expand(inp.B, *W0.shape).contiguous()
    eta = inp.eta.to(dev) if inp.eta is not None else None
    z, W = abi.ttt_linear_fwd(q, k, v, W0.to(dev), inp.b, inp.causal if causal is None else causal,
                              eta=eta, eta_scalar=inp.eta_scalar)
    abi.ttt_sync_status()
    return z.double().cpu().numpy(), W.double().cpu().numpy()


def _select(x, chains, H):
    """[B,H,...] -> [1, n, ...] for the listed flat (b*H + h) chains."""
    idx = torch.tensor(chains)
    flat = x.reshape(-1, *x.shape[2:])
    return flat[idx].unsqueeze(0)


def oracle_linear(inp, chains=None, causal=None):
    """Oracle outputs for all chains, or for the listed flat chain indices
    (shapes [1, n, ...])."""
    causal = inp.causal if causal is None else causal
    W0 = inp.params["W0"]
    if chains is None:
        return oracle.linear(inp.q, inp.k, inp.v, W0, inp.b, causal, eta=inp.eta,
                             eta_scalar=inp.eta_scalar)
    q, k, v = (_select(x, chains, inp.H) for x in (inp.q, inp.k, inp.v))
    eta = _select(inp.eta, chains, inp.H) if inp.eta is not None else None
    W0s = torch.stack([W0[c % inp.H] for c in chains]).unsqueeze(0)
    return oracle.linear(q, k, v, W0s, inp.b, causal, eta=eta, eta_scalar=inp.eta_scalar)


def gpu_mlp(inp, causal=None):
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    P = [inp.params[n].to(dev) for n in ("W1", "c1", "W2", "c2")]
    eta = inp.eta.to(dev) if inp.eta is not None else None
    z, outs = abi.ttt_mlp_fwd(q, k, v, *P, inp.b, inp.causal if causal is None else causal,
                              eta=eta, eta_scalar=inp.eta_scalar)
    abi.ttt_sync_status()
    return z.double().cpu().numpy(), [o.double().cpu().numpy() for o in outs]


def oracle_mlp(inp, chains=None, causal=None):
    causal = inp.causal if causal is None else causal
    P = [inp.params[n] for n in ("W1", "c1", "W2", "c2")]
    if chains is None:
        z, *W = oracle.mlp(inp.q, inp.k, inp.v, *P, inp.b, causal, eta=inp.eta,
                           eta_scalar=inp.eta_scalar)
        return z, W
    q, k, v = (_select(x, chains, inp.H) for x in (inp.q, inp.k, inp.v))
    eta = _select(inp.eta, chains, inp.H) if inp.eta is not None else None
    Ps = [torch.stack([p[c % inp.H] for c in chains]).unsqueeze(0) for p in P]
    z, *W = oracle.mlp(q, k, v, *Ps, inp.b, causal, eta=eta, eta_scalar=inp.eta_scalar)
    return z, W


def pick(flat_arr, chains):
    """Rows of a [B,H,...] numpy array for flat chain indices, as [1, n, ...]."""
    f = flat_arr.reshape(-1, *flat_arr.shape[2:])
    return f[np.array(chains)][None]


synth = synth
