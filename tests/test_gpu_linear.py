"""TTT-Linear on the GPU against the fp64 oracle (element by element), through the
C ABI.  Small cases span several tiles and ragged tails; the full-size workloads
run in the launch configuration the benchmark times and are compared on every
(batch, head) chain over its whole sequence."""
import numpy as np
import pytest
import torch

from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _check(inp, chains=None, per_batch_w0=False, tol=None):
    tol = tol or G.tol_for(inp)
    zg, Wg = G.gpu_linear(inp, per_batch_w0=per_batch_w0)
    zr, Wr = G.oracle_linear(inp, chains)
    if chains is not None:
        zg, Wg = G.pick(zg, chains), G.pick(Wg, chains)
    ez, eW = G.rel_err(zg, zr), G.rel_err(Wg, Wr)
    assert ez <= tol and eW <= tol, (ez, eW, tol)
    return ez, eW


def test_tiny_fp32_workload():
    """B1 H2 T64 d16 b16 causal fp32, eta 0.5 (fp32 path, 1e-4)."""
    _check(G.synth.workload("linear_tiny_f32"), tol=G.TOL_F32)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("b,causal", [(16, True), (1, True), (5, True), (40, True),
                                      (16, False), (7, False), (40, False)])
def test_bf16_small(d, b, causal):
    inp = G.synth.make("linear", B=2, H=3, T=75, d=d, b=b, causal=causal, eta=1.0, seed=d + b)
    _check(inp)


@pytest.mark.parametrize("d", [16, 64])
@pytest.mark.parametrize("b,causal", [(16, True), (3, True), (24, False)])
def test_fp32_small(d, b, causal):
    inp = G.synth.make("linear", B=2, H=2, T=50, d=d, b=b, causal=causal, dtype=torch.float32,
                       eta="sigmoid", seed=100 + d + b)
    _check(inp)


@pytest.mark.parametrize("T", [0, 1, 15, 16, 17, 33])
def test_short_and_empty_sequences(T):
    inp = G.synth.make("linear", B=1, H=2, T=T, d=64, b=16, causal=True, seed=7 + T)
    _check(inp)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("T", [16, 48, 64, 128, 130, 191, 250, 320])
def test_b16_d64_block_boundaries(T, causal):
    """b = 16, d = 64 (tokens arrive in 64-token blocks; the last mini-batch of a block
    releases it and loads the next block's first fragments, skipping only the wait past
    the end): one mini-batch, a block without its last mini-batch, whole last blocks,
    partial last blocks and a partial last mini-batch, per-token eta."""
    inp = G.synth.make("linear", B=2, H=2, T=T, d=64, b=16, causal=causal, eta="sigmoid", seed=200 + T)
    _check(inp)


@pytest.mark.parametrize("B,H", [(1, 1), (1, 3), (3, 3)])
def test_b16_d64_odd_chain_counts(B, H):
    """b = 16, d = 64 with one, three and nine (batch, head) chains, one CTA each."""
    inp = G.synth.make("linear", B=B, H=H, T=200, d=64, b=16, causal=True, seed=300 + 3 * B + H)
    _check(inp)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("T", [0, 1, 15, 17, 63, 64, 65, 129])
def test_b1_delta_rule_lengths(d, T):
    """b = 1 (the delta rule: d <= 64 in 16-token chunks with a forward substitution,
    d = 128 on the column-parallel kernel): lengths around 16-token chunks and 64-token
    blocks, per-token eta, per-batch W0, both masks (a one-token mini-batch reads its
    own write either way)."""
    for causal in (True, False):
        inp = G.synth.make("linear", B=3, H=1, T=T, d=d, b=1, causal=causal, eta="sigmoid", seed=900 + d + T)
        _check(inp, per_batch_w0=True)


def test_per_token_eta_and_per_batch_w0():
    inp = G.synth.make("linear", B=3, H=2, T=130, d=64, b=16, causal=True, eta="sigmoid", seed=11)
    _check(inp, per_batch_w0=True)


def test_full_batch_noncausal_single_block():
    """b = T: one full-batch GD step, every query reads the updated weights."""
    inp = G.synth.make("linear", B=4, H=2, T=196, d=64, b=196, causal=False, seed=12)
    _check(inp)


def test_full_batch_weights_not_16_byte_aligned():
    """Initial and final weights that are only 4-byte aligned (views at an odd float
    offset), which the boundary accepts: the full-batch kernel reads and writes them
    as single floats."""
    inp = G.synth.make("linear", B=2, H=2, T=196, d=64, b=196, causal=False, eta="sigmoid", seed=450)
    dev = torch.device("cuda")
    from test_sequence_layers_gb300 import abi
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    W0 = inp.params["W0"]
    buf = torch.zeros(W0.numel() + 1, device=dev)
    buf[1:] = W0.reshape(-1).to(dev)
    W0u = buf[1:].view(W0.shape)
    obuf = torch.zeros(2 * 2 * 64 * 64 + 1, device=dev)
    Wout = obuf[1:].view(2, 2, 64, 64)
    z, W = abi.ttt_linear_fwd(q, k, v, W0u, inp.b, False, eta=inp.eta.to(dev), W_out=Wout)
    abi.ttt_sync_status()
    zr, Wr = G.oracle_linear(inp)
    ez, eW = G.rel_err(z.double().cpu(), zr), G.rel_err(Wout.double().cpu(), Wr)
    assert ez <= G.TOL_BF16 and eW <= G.TOL_BF16, (ez, eW)


@pytest.mark.parametrize("T", [1, 17, 48, 64, 80, 100, 196, 240, 256, 300])
def test_full_batch_lengths(T):
    """b >= T, non-causal (one inner GD step over the whole sequence, every query
    reads the updated weights): short, ragged, box-aligned and longest on-chip
    lengths, one beyond them, per-token eta, per-batch W0."""
    inp = G.synth.make("linear", B=2, H=2, T=T, d=64, b=T + 5, causal=False, eta="sigmoid", seed=400 + T)
    _check(inp, per_batch_w0=True)


@pytest.mark.parametrize("split", [64, 128, 48, 80])
def test_split_run_continues_sequence(split):
    """W_final passed back as W0 continues the sequence (chunked prefill).  The b = 16
    kernel advances the state once per mini-batch and forms each 16-token chunk's
    outputs from that chunk's start weights, so a split at any mini-batch boundary
    (64-token block boundaries or not) regroups nothing: z and the final weights are
    bit-identical to one run."""
    inp = G.synth.make("linear", B=2, H=2, T=160, d=64, b=16, causal=True, seed=13)
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    W0 = inp.params["W0"].to(dev)
    from test_sequence_layers_gb300 import abi
    z, W = abi.ttt_linear_fwd(q, k, v, W0, 16)
    z1, W1 = abi.ttt_linear_fwd(q[:, :, :split].contiguous(), k[:, :, :split].contiguous(),
                                v[:, :, :split].contiguous(), W0, 16)
    # continue in place: the final-weight buffer is the initial-weight input
    z2, W2 = abi.ttt_linear_fwd(q[:, :, split:].contiguous(), k[:, :, split:].contiguous(),
                                v[:, :, split:].contiguous(), W1, 16, W_out=W1)
    abi.ttt_sync_status()
    assert torch.equal(W2, W)
    assert torch.equal(torch.cat([z1, z2], 2), z)


def test_deterministic():
    inp = G.synth.make("linear", B=2, H=4, T=300, d=64, b=16, causal=True, seed=14)
    a = G.gpu_linear(inp)
    b = G.gpu_linear(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------ full workloads


def test_workload_125m_layer_full():
    """B8 H12 T2048 d64 b16 causal bf16, eta 1: every chain against the oracle."""
    inp = G.synth.workload("linear_125m")
    ez, eW = _check(inp)
    print(f"linear_125m rel err z {ez:.3e} W {eW:.3e}")


def test_workload_125m_delta_rule_b1():
    """The b = 1 check of the 125M-layer shape (delta rule), B1 H12 T2048."""
    inp = G.synth.workload("linear_125m_b1")
    ez, eW = _check(inp)
    print(f"linear_125m_b1 rel err z {ez:.3e} W {eW:.3e}")


def test_workload_long_context_gated_full():
    """B2 H32 T32768 with per-token eta = sigmoid(g): every chain, full length."""
    inp = G.synth.workload("linear_long_gated")
    ez, eW = _check(inp)
    print(f"linear_long_gated rel err z {ez:.3e} W {eW:.3e}")


def test_workload_vision_full_batch_full():
    """B256 N196 H6, b = N, non-causal: every chain."""
    inp = G.synth.workload("vision_linear")
    ez, eW = _check(inp)
    print(f"vision_linear rel err z {ez:.3e} W {eW:.3e}")


# ------------------------------------------- dot-product loss and inner epochs


def _check_variant(inp, loss="mse", epochs=1, tol=None):
    """GPU vs oracle with the given inner loss and number of inner epochs."""
    tol = tol or G.tol_for(inp)
    dev = torch.device("cuda")
    from test_sequence_layers_gb300 import abi
    import oracle
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    eta = inp.eta.to(dev) if inp.eta is not None else None
    z, W = abi.ttt_linear_fwd(q, k, v, inp.params["W0"].to(dev), inp.b, inp.causal, eta=eta,
                              eta_scalar=inp.eta_scalar, loss=loss, epochs=epochs)
    abi.ttt_sync_status()
    zr, Wr = oracle.linear(inp.q, inp.k, inp.v, inp.params["W0"], inp.b, inp.causal, eta=inp.eta,
                           eta_scalar=inp.eta_scalar, loss=loss, epochs=epochs)
    ez, eW = G.rel_err(z.double().cpu(), zr), G.rel_err(W.double().cpu(), Wr)
    assert ez <= tol and eW <= tol, (ez, eW, tol)


@pytest.mark.parametrize("d,b,causal", [(16, 16, True), (64, 16, True), (64, 16, False), (32, 5, True),
                                        (128, 16, True), (64, 1, True), (16, 1, False), (128, 1, True),
                                        (64, 196, False)])
def test_dot_loss_bf16(d, b, causal):
    """Negative dot-product loss (the ViT3 block's inner loss): residual -V; every
    bf16 kernel (b = 16, general, full batch)."""
    T = 196 if b == 196 else 150
    inp = G.synth.make("linear", B=2, H=2, T=T, d=d, b=b, causal=causal, eta="sigmoid", seed=800 + d + b)
    _check_variant(inp, loss="dot")


@pytest.mark.parametrize("b,causal", [(3, True), (50, False)])
def test_dot_loss_fp32(b, causal):
    inp = G.synth.make("linear", B=2, H=2, T=50, d=16, b=b, causal=causal, dtype=torch.float32,
                       eta="sigmoid", seed=810 + b)
    _check_variant(inp, loss="dot", tol=G.TOL_F32)


@pytest.mark.parametrize("loss", ["mse", "dot"])
@pytest.mark.parametrize("epochs,T", [(2, 196), (3, 100), (2, 17)])
def test_full_batch_epochs_bf16(loss, epochs, T):
    """Several inner epochs of full-batch GD (ViT3 article, observation 2): b >= T,
    non-causal, every query reads the last weights."""
    inp = G.synth.make("linear", B=2, H=3, T=T, d=64, b=T, causal=False, eta="sigmoid", seed=820 + T + epochs)
    _check_variant(inp, loss=loss, epochs=epochs)


def test_full_batch_epochs_fp32():
    inp = G.synth.make("linear", B=1, H=2, T=40, d=16, b=40, causal=False, dtype=torch.float32,
                       eta=0.5, seed=830)
    _check_variant(inp, epochs=3, tol=G.TOL_F32)


def test_epochs_outside_the_full_batch_kernel_are_unsupported():
    inp = G.synth.make("linear", B=1, H=1, T=64, d=32, b=64, causal=False, seed=840)
    dev = torch.device("cuda")
    from test_sequence_layers_gb300 import abi
    with pytest.raises(abi.TTTError) as e:
        abi.ttt_linear_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.params["W0"].to(dev), 64,
                           causal=False, epochs=2)
    assert e.value.code == -2


# ------------------------------------------------- inner layer norm + residual


def _check_ln(inp, tol=None, per_batch_w0=False, chains=None):
    """GPU vs oracle for f(x; W) = x + LN(x W) (scale / shift from the inputs)."""
    import oracle
    from test_sequence_layers_gb300 import abi
    tol = tol or G.tol_for(inp)
    dev = torch.device("cuda")
    W0 = inp.params["W0"]
    if per_batch_w0:
        W0 = W0.expand(inp.B, *W0.shape).contiguous()
    gam, bet = inp.params["ln_gamma"], inp.params["ln_beta"]
    eta = inp.eta.to(dev) if inp.eta is not None else None
    z, W = abi.ttt_linear_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), W0.to(dev), inp.b, inp.causal,
                              eta=eta, eta_scalar=inp.eta_scalar, ln_gamma=gam.to(dev), ln_beta=bet.to(dev))
    abi.ttt_sync_status()
    zg, Wg = z.double().cpu().numpy(), W.double().cpu().numpy()
    if chains is None:
        zr, Wr = oracle.linear(inp.q, inp.k, inp.v, W0, inp.b, inp.causal, eta=inp.eta,
                               eta_scalar=inp.eta_scalar, ln_gamma=gam, ln_beta=bet)
    else:
        sel = lambda x: x.reshape(-1, *x.shape[2:])[chains].unsqueeze(0)
        W0s = torch.stack([W0[c % inp.H] for c in chains]).unsqueeze(0)
        gs = torch.stack([gam[c % inp.H] for c in chains])
        bs = torch.stack([bet[c % inp.H] for c in chains])
        zr, Wr = oracle.linear(sel(inp.q), sel(inp.k), sel(inp.v), W0s, inp.b, inp.causal,
                               eta=sel(inp.eta) if inp.eta is not None else None,
                               eta_scalar=inp.eta_scalar, ln_gamma=gs, ln_beta=bs)
        zg, Wg = G.pick(zg, chains), G.pick(Wg, chains)
    ez, eW = G.rel_err(zg, zr), G.rel_err(Wg, Wr)
    assert ez <= tol and eW <= tol, (ez, eW, tol)
    return ez, eW


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("T", [150, 64, 13])
def test_inner_norm_bf16(d, causal, T):
    """x + LN(x W) (the walkthrough's TTT-Linear) on the b = 16 kernel: several
    blocks, a partial last block and a partial last mini-batch, per-token eta."""
    inp = G.synth.make("linear", B=2, H=3, T=T, d=d, b=16, causal=causal, eta="sigmoid",
                       seed=1400 + d + T, ln=True)
    _check_ln(inp, per_batch_w0=(T == 64))


@pytest.mark.parametrize("b,causal", [(16, True), (3, True), (20, False)])
def test_inner_norm_fp32(b, causal):
    inp = G.synth.make("linear", B=2, H=2, T=40, d=16, b=b, causal=causal, dtype=torch.float32,
                       eta=0.5, seed=1500 + b, ln=True)
    _check_ln(inp, tol=G.TOL_F32)


def test_inner_norm_other_mini_batches_unsupported_in_bf16():
    from test_sequence_layers_gb300 import abi
    inp = G.synth.make("linear", B=1, H=1, T=40, d=64, b=5, causal=True, seed=1600, ln=True)
    dev = torch.device("cuda")
    with pytest.raises(abi.TTTError) as e:
        abi.ttt_linear_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.params["W0"].to(dev), 5,
                           ln_gamma=inp.params["ln_gamma"].to(dev), ln_beta=inp.params["ln_beta"].to(dev))
    assert e.value.code == -2


def test_workload_125m_inner_norm_full():
    """B8 H12 T2048 d64 b16 causal with the inner norm: every chain."""
    inp = G.synth.workload("linear_125m_ln")
    ez, eW = _check_ln(inp)
    print(f"linear_125m_ln rel err z {ez:.3e} W {eW:.3e}")
