"""Depthwise 3x3 convolution inner model (full-batch inner GD over the token grid)
on the GPU against the fp64 oracle, through the C ABI: several grids (square,
ragged, one row), head dimensions, both losses, one and several epochs, per-token
eta, per-batch taps, fp32 I/O, and the vision workload on every chain."""
import numpy as np
import pytest
import torch

import oracle
from test_sequence_layers_gb300 import abi
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _check(inp, hh, ww, loss="mse", epochs=1, per_batch=False, chains=None):
    dev = torch.device("cuda")
    W0 = inp.params["W0"]
    if per_batch:
        W0 = W0.expand(inp.B, *W0.shape).contiguous()
    eta = inp.eta.to(dev) if inp.eta is not None else None
    z, W = abi.ttt_dwconv_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), W0.to(dev), hh, ww, eta=eta,
                              eta_scalar=inp.eta_scalar, loss=loss, epochs=epochs)
    abi.ttt_sync_status()
    zg, Wg = z.double().cpu().numpy(), W.double().cpu().numpy()
    if chains is None:
        zr, Wr = oracle.dwconv(inp.q, inp.k, inp.v, W0, hh, ww, eta=inp.eta, eta_scalar=inp.eta_scalar,
                               loss=loss, epochs=epochs)
    else:
        sel = lambda x: x.reshape(-1, *x.shape[2:])[chains].unsqueeze(0)
        W0s = torch.stack([W0[c % inp.H] for c in chains]).unsqueeze(0)
        zr, Wr = oracle.dwconv(sel(inp.q), sel(inp.k), sel(inp.v), W0s, hh, ww,
                               eta=sel(inp.eta) if inp.eta is not None else None,
                               eta_scalar=inp.eta_scalar, loss=loss, epochs=epochs)
        zg, Wg = G.pick(zg, chains), G.pick(Wg, chains)
    tol = G.tol_for(inp)
    ez, eW = G.rel_err(zg, zr), G.rel_err(Wg, Wr)
    assert ez <= tol and eW <= tol, (ez, eW, tol)
    return ez, eW


@pytest.mark.parametrize("hh,ww", [(14, 14), (7, 9), (1, 30), (3, 3)])
@pytest.mark.parametrize("loss", ["mse", "dot"])
def test_grids_and_losses(hh, ww, loss):
    inp = G.synth.make("dwconv", B=2, H=3, T=hh * ww, d=64, b=hh * ww, causal=False, eta="sigmoid",
                       seed=1000 + hh * ww)
    _check(inp, hh, ww, loss=loss)


@pytest.mark.parametrize("d", [8, 16, 128])
@pytest.mark.parametrize("epochs", [1, 3])
def test_head_dims_and_epochs(d, epochs):
    inp = G.synth.make("dwconv", B=2, H=2, T=80, d=d, b=80, causal=False, eta=0.5, seed=1100 + d)
    _check(inp, 8, 10, epochs=epochs, per_batch=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_wide_head_row_copies(dtype):
    """d = 512, past the 256-element box of a tensor map: one bulk copy per grid row
    with the border zeroed in shared memory, a single buffer, runtime strides."""
    inp = G.synth.make("dwconv", B=1, H=3, T=12, d=512, b=12, causal=False, dtype=dtype, eta="sigmoid",
                       seed=1400)
    _check(inp, 3, 4, loss="mse", epochs=2)


def test_largest_grid_on_chip():
    """22 x 22 tokens at d = 64 in bf16: the largest square grid one CTA holds (the
    padded K and Q grids, V and the partial sums); 23 x 23 is rejected."""
    inp = G.synth.make("dwconv", B=1, H=2, T=484, d=64, b=484, causal=False, eta="sigmoid", seed=1150)
    _check(inp, 22, 22, loss="mse")
    big = G.synth.make("dwconv", B=1, H=1, T=529, d=64, b=529, causal=False, seed=1151)
    dev = torch.device("cuda")
    with pytest.raises(abi.TTTError) as e:
        abi.ttt_dwconv_fwd(big.q.to(dev), big.k.to(dev), big.v.to(dev), big.params["W0"].to(dev), 23, 23)
    assert e.value.code == -2


def test_fp32_io():
    inp = G.synth.make("dwconv", B=1, H=2, T=42, d=32, b=42, causal=False, dtype=torch.float32,
                       eta="sigmoid", seed=1200)
    _check(inp, 6, 7, loss="mse", epochs=2)


def test_empty_grid():
    inp = G.synth.make("dwconv", B=1, H=2, T=0, d=16, b=1, causal=False, seed=1300)
    dev = torch.device("cuda")
    z, W = abi.ttt_dwconv_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.params["W0"].to(dev), 0, 5)
    abi.ttt_sync_status()
    assert z.numel() == 0
    assert torch.equal(W.cpu(), inp.params["W0"].expand(1, 2, 9, 16))


def test_workload_vision_dwconv_full():
    """B256 H6, 14 x 14 grid, d = 64, dot loss, eta = 1 (the ViT3 block's inner
    training): every chain against the oracle."""
    inp = G.synth.workload("vision_dwconv")
    o = inp.options
    ez, eW = _check(inp, o["height"], o["width"], loss=o["loss"])
    print(f"vision_dwconv rel err z {ez:.3e} W {eW:.3e}")
