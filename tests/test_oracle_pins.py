"""Pins of the fp64 oracle against what the pages and the mathematics fix.

No GPU.  Every test compares the oracle with a route that shares none of its code:
the delta rule as the pages print it, brute-force linear attention, Theorem 1,
autograd on the layer's definition, central finite differences, and the matrix
("dual") form of a mini-batch step.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import _defs

rng = np.random.default_rng(1234)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _qkv(B, H, T, d, unit=True, seed=0):
    r = np.random.default_rng(seed)
    q, k, v = (r.standard_normal((B, H, T, d)) for _ in range(3))
    if unit:
        q, k = _unit(q), _unit(k)
    return q, k, v


def _mlp_params(H, d, m, seed=0, scale=0.3, bias=True):
    r = np.random.default_rng(seed)
    W1 = r.standard_normal((H, d, m)) * scale
    W2 = r.standard_normal((H, m, d)) * scale
    c1 = r.standard_normal((H, m)) * (0.1 if bias else 0.0)
    c2 = r.standard_normal((H, d)) * (0.1 if bias else 0.0)
    return W1, c1, W2, c2


# --------------------------------------------------------------- TTT-Linear


def test_b1_is_delta_rule_column_convention():
    """b = 1 must equal the delta rule W_t = W_{t-1} + eta (v_t - W_{t-1} k_t) k_t^T
    ("Fast weights 与 TTT layers", section 1, column convention f(k;W) = W k).
    The oracle's row convention is its transpose: W_row = W_col^T."""
    B, H, T, d = 1, 2, 23, 5
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.1, 1.2, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.3
    z, Wf = oracle.linear(q, k, v, W0, b=1, causal=True, eta=eta)
    for h in range(H):
        Wc = W0[h].T.copy()
        for t in range(T):
            kt, vt = k[0, h, t][:, None], v[0, h, t][:, None]
            Wc = Wc + eta[0, h, t] * (vt - Wc @ kt) @ kt.T
            np.testing.assert_allclose(z[0, h, t], (Wc @ q[0, h, t][:, None])[:, 0], atol=1e-12)
        np.testing.assert_allclose(Wf[0, h], Wc.T, atol=1e-12)


def test_b1_unit_key_unit_rate_writes_exactly():
    """With a unit-norm key and eta = 1, one delta-rule write makes f(k_t;W_t) = v_t
    exactly (the repeated-write remark of "Fast weights 与 TTT layers", section 1).
    Query = key reads that back."""
    B, H, T, d = 2, 1, 17, 6
    _, k, v = _qkv(B, H, T, d)
    z, _ = oracle.linear(k, k, v, rng.standard_normal((H, d, d)), b=1, causal=True,
                         eta_scalar=1.0)
    np.testing.assert_allclose(z, v, atol=1e-12)


@pytest.mark.parametrize("b,causal", [(1, True), (4, True), (7, True), (4, False), (7, False)])
def test_dot_loss_is_linear_attention(b, causal):
    """Negative dot-product loss: grad = -k^T v does not depend on W, so with W0 = 0
    z_t = eta * sum_{s visible to t} (q_t . k_s) v_s, the linear-attention recurrence
    S_t = S_{t-1} + k_t v_t^T read by q_t ("TTT：Test-Time Training", sections
    线性注意力 and 如何理解).  Causal: s <= t; non-causal: s up to t's block end."""
    B, H, T, d = 1, 2, 19, 4
    q, k, v = _qkv(B, H, T, d, unit=False)
    eta = 0.7
    z, Wf = oracle.linear(q, k, v, np.zeros((H, d, d)), b=b, causal=causal,
                          eta_scalar=eta, loss="dot")
    for h in range(H):
        for t in range(T):
            last = t if causal else min((t // b + 1) * b, T) - 1
            ref = sum(eta * (q[0, h, t] @ k[0, h, s]) * v[0, h, s] for s in range(last + 1))
            np.testing.assert_allclose(z[0, h, t], ref, atol=1e-11)
        S = sum(np.outer(k[0, h, s], v[0, h, s]) for s in range(T))
        np.testing.assert_allclose(Wf[0, h], eta * S, atol=1e-11)


def test_theorem1_batch_gd_zero_init_is_linear_attention():
    """Theorem 1 (walkthrough section 2.1.1): linear inner model, batch GD (b = T),
    W0 = 0 and the MSE loss give causal linear attention: every gradient is taken
    at W0 = 0 where the residual is -v_s, so z_t = eta sum_{s<=t} (q_t . k_s) v_s."""
    B, H, T, d = 2, 1, 21, 5
    q, k, v = _qkv(B, H, T, d)
    eta = 0.9
    z, _ = oracle.linear(q, k, v, np.zeros((H, d, d)), b=T, causal=True, eta_scalar=eta)
    for bi in range(B):
        A = np.tril(q[bi, 0] @ k[bi, 0].T)
        np.testing.assert_allclose(z[bi, 0], eta * A @ v[bi, 0], atol=1e-12)


def test_full_batch_is_one_gd_step_linear():
    """b = T, non-causal: W1 = W0 - grad(sum_s eta_s l_s)(W0), every query reads W1
    (ViT3 article, observation 2; spec definition).  Gradient by autograd."""
    B, H, T, d = 1, 2, 13, 6
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.2, 1.0, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.2
    z, Wf = oracle.linear(q, k, v, W0, b=T, causal=False, eta=eta)
    for h in range(H):
        W = torch.tensor(W0[h], requires_grad=True)
        K, V = torch.tensor(k[0, h]), torch.tensor(v[0, h])
        L = (torch.tensor(eta[0, h])[:, None] * 0.5 * (K @ W - V) ** 2).sum()
        (g,) = torch.autograd.grad(L, W)
        W1 = (W - g).detach().numpy()
        np.testing.assert_allclose(Wf[0, h], W1, atol=1e-12)
        np.testing.assert_allclose(z[0, h], q[0, h] @ W1, atol=1e-12)


@pytest.mark.parametrize("epochs", [2, 3])
def test_full_batch_epochs_are_repeated_gd_steps(epochs):
    """b = T, non-causal, several inner epochs (ViT3 article, observation 2: an epoch
    of full-batch inner training is one update over all N tokens): W_{e+1} =
    W_e - grad(sum_s eta_s l_s)(W_e) by autograd, every query reads the last W."""
    B, H, T, d = 1, 2, 13, 6
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.2, 1.0, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.2
    z, Wf = oracle.linear(q, k, v, W0, b=T, causal=False, eta=eta, epochs=epochs)
    for h in range(H):
        W = torch.tensor(W0[h])
        K, V = torch.tensor(k[0, h]), torch.tensor(v[0, h])
        for _ in range(epochs):
            Wg = W.clone().requires_grad_(True)
            L = (torch.tensor(eta[0, h])[:, None] * 0.5 * (K @ Wg - V) ** 2).sum()
            (g,) = torch.autograd.grad(L, Wg)
            W = (Wg - g).detach()
        np.testing.assert_allclose(Wf[0, h], W.numpy(), atol=1e-12)
        np.testing.assert_allclose(z[0, h], q[0, h] @ W.numpy(), atol=1e-12)


def test_full_batch_epochs_dot_loss_closed_form():
    """Dot loss: the gradient -K^T V does not depend on W, so E epochs move W by
    E * eta * K^T V exactly."""
    B, H, T, d = 2, 1, 9, 5
    q, k, v = _qkv(B, H, T, d, unit=False)
    W0 = rng.standard_normal((H, d, d))
    z, Wf = oracle.linear(q, k, v, W0, b=T, causal=False, eta_scalar=0.3, loss="dot", epochs=3)
    for bi in range(B):
        W = W0[0] + 3 * 0.3 * k[bi, 0].T @ v[bi, 0]
        np.testing.assert_allclose(Wf[bi, 0], W, atol=1e-12)
        np.testing.assert_allclose(z[bi, 0], q[bi, 0] @ W, atol=1e-12)


def test_epochs_need_one_noncausal_block():
    q, k, v = _qkv(1, 1, 8, 4)
    W0 = np.zeros((1, 4, 4))
    with pytest.raises(ValueError):
        oracle.linear(q, k, v, W0, b=8, causal=True, epochs=2)
    with pytest.raises(ValueError):
        oracle.linear(q, k, v, W0, b=4, causal=False, epochs=2)


@pytest.mark.parametrize("T,b,causal", [(11, 1, True), (11, 3, True), (11, 4, False),
                                        (12, 4, True), (10, 10, True), (9, 20, False)])
def test_linear_matches_definition_autograd(T, b, causal):
    """Every mini-batch size, ragged tails included: the oracle equals the layer's
    definition evaluated with autograd gradients."""
    B, H, d = 1, 1, 4
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.1, 1.0, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.3
    z, Wf = oracle.linear(q, k, v, W0, b=b, causal=causal, eta=eta)
    t = lambda a: torch.tensor(a)
    zr, (Wr,) = _defs.definition_autograd(_defs.f_linear, [t(W0[0])], t(q[0, 0]), t(k[0, 0]),
                                          t(v[0, 0]), t(eta[0, 0]), b, causal)
    np.testing.assert_allclose(z[0, 0], zr.numpy(), atol=1e-12)
    np.testing.assert_allclose(Wf[0, 0], Wr.numpy(), atol=1e-12)


@pytest.mark.parametrize("b,causal", [(1, True), (16, True), (5, True), (16, False), (64, False)])
def test_linear_dual_form_equals_primal(b, causal):
    """The matrix form of a mini-batch (dual form, walkthrough section 1.2.2: a
    lower-triangular mask of zeros instead of explicit per-token gradients) gives
    the same outputs as the token loop.  This pins the algebra the kernels use."""
    B, H, T, d = 2, 3, 70, 16
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.1, 1.0, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.05
    z, Wf = oracle.linear(q, k, v, W0, b=b, causal=causal, eta=eta)
    for bi in range(B):
        for h in range(H):
            zr, Wr = _defs.dual_linear(q[bi, h], k[bi, h], v[bi, h], W0[h], eta[bi, h], b, causal)
            np.testing.assert_allclose(z[bi, h], zr, atol=1e-11)
            np.testing.assert_allclose(Wf[bi, h], Wr, atol=1e-11)


def test_linear_eta_zero_is_identity():
    B, H, T, d = 1, 2, 9, 4
    q, k, v = _qkv(B, H, T, d)
    W0 = rng.standard_normal((H, d, d))
    z, Wf = oracle.linear(q, k, v, W0, b=3, eta_scalar=0.0)
    np.testing.assert_allclose(Wf[0], W0, atol=0)
    np.testing.assert_allclose(z[0], np.einsum("htd,hde->hte", q[0], W0), atol=1e-13)


def test_linear_column_separable():
    """Column j of W, E and Z only involves column j of W0 and V (plus the shared
    Q, K, eta), so running on a column slice gives that slice of the full run."""
    B, H, T, d = 1, 1, 30, 8
    q, k, v = _qkv(B, H, T, d)
    W0 = rng.standard_normal((H, d, d)) * 0.1
    z, Wf = oracle.linear(q, k, v, W0, b=4)
    cols = [1, 5, 6]
    # pad the sliced problem back to d columns with zeros so shapes stay square
    W0s = np.zeros_like(W0); W0s[..., cols] = W0[..., cols]
    vs = np.zeros_like(v); vs[..., cols] = v[..., cols]
    zs, Ws = oracle.linear(q, k, vs, W0s, b=4)
    np.testing.assert_allclose(zs[..., cols], z[..., cols], atol=1e-12)
    np.testing.assert_allclose(Ws[..., cols], Wf[..., cols], atol=1e-12)


def test_linear_split_run_continues():
    """Passing W_final back as W0 continues the sequence (chunked prefill) when the
    split point is a multiple of b."""
    B, H, T, d, b = 2, 2, 48, 8, 8
    q, k, v = _qkv(B, H, T, d)
    W0 = rng.standard_normal((B, H, d, d)) * 0.1
    z, Wf = oracle.linear(q, k, v, W0, b=b)
    z1, W1 = oracle.linear(q[:, :, :24], k[:, :, :24], v[:, :, :24], W0, b=b)
    z2, W2 = oracle.linear(q[:, :, 24:], k[:, :, 24:], v[:, :, 24:], W1, b=b)
    np.testing.assert_allclose(np.concatenate([z1, z2], 2), z, atol=1e-12)
    np.testing.assert_allclose(W2, Wf, atol=1e-12)


def test_linear_shared_vs_per_batch_w0():
    B, H, T, d = 3, 2, 10, 4
    q, k, v = _qkv(B, H, T, d)
    W0 = rng.standard_normal((H, d, d))
    z1, W1 = oracle.linear(q, k, v, W0, b=3)
    z2, W2 = oracle.linear(q, k, v, np.broadcast_to(W0, (B, H, d, d)).copy(), b=3)
    np.testing.assert_array_equal(z1, z2)
    np.testing.assert_array_equal(W1, W2)


# ------------------------------------------------------------------ TTT-MLP


@pytest.mark.parametrize("activation", ["silu", "gelu"])
def test_mlp_gradient_matches_finite_differences(activation):
    """One mini-batch step: W_out = W0 - grad(sum_s eta_s l_s)(W0) with the hand
    gradient inside the oracle; compare every parameter entry with central finite
    differences of the plain forward loss (h = 1e-6).  SiLU (ViT3 article) and the
    walkthrough's GELU, h * Phi(h)."""
    from scipy.special import erf
    B, H, T, d, m = 1, 1, 3, 4, 16
    q, k, v = _qkv(B, H, T, d)
    W1, c1, W2, c2 = _mlp_params(H, d, m)
    eta = np.array([[[0.3, 0.7, 1.1]]])
    _, W1o, c1o, W2o, c2o = oracle.mlp(q, k, v, W1, c1, W2, c2, b=T, causal=True, eta=eta,
                                       activation=activation)
    if activation == "silu":
        act = lambda x: x / (1 + np.exp(-x))
    else:
        act = lambda x: x * 0.5 * (1 + erf(x / np.sqrt(2)))

    def loss(P):
        a, ca, bm, cb = P
        tot = 0.0
        for s in range(T):
            h = k[0, 0, s] @ a + ca
            out = act(h) @ bm + cb
            tot += eta[0, 0, s] * 0.5 * np.sum((out - v[0, 0, s]) ** 2)
        return tot

    P = [W1[0].copy(), c1[0].copy(), W2[0].copy(), c2[0].copy()]
    got = [W1[0] - W1o[0, 0], c1[0] - c1o[0, 0], W2[0] - W2o[0, 0], c2[0] - c2o[0, 0]]
    hstep = 1e-6
    for pi in range(4):
        fd = np.zeros_like(P[pi])
        for idx in np.ndindex(P[pi].shape):
            Pp = [p.copy() for p in P]; Pm = [p.copy() for p in P]
            Pp[pi][idx] += hstep; Pm[pi][idx] -= hstep
            fd[idx] = (loss(Pp) - loss(Pm)) / (2 * hstep)
        np.testing.assert_allclose(got[pi], fd, rtol=1e-7, atol=1e-9)


@pytest.mark.parametrize("activation", ["silu", "gelu"])
@pytest.mark.parametrize("T,b,causal", [(7, 1, True), (7, 3, True), (8, 4, False),
                                        (7, 7, False), (6, 10, True)])
def test_mlp_matches_definition_autograd(T, b, causal, activation):
    B, H, d, m = 1, 1, 3, 8
    q, k, v = _qkv(B, H, T, d)
    W1, c1, W2, c2 = _mlp_params(H, d, m)
    eta = rng.uniform(0.1, 1.0, (B, H, T))
    z, W1o, c1o, W2o, c2o = oracle.mlp(q, k, v, W1, c1, W2, c2, b=b, causal=causal, eta=eta,
                                       activation=activation)
    t = lambda a: torch.tensor(a)
    f = _defs.f_mlp if activation == "silu" else _defs.f_mlp_gelu
    zr, Pr = _defs.definition_autograd(f, [t(W1[0]), t(c1[0]), t(W2[0]), t(c2[0])],
                                       t(q[0, 0]), t(k[0, 0]), t(v[0, 0]), t(eta[0, 0]), b, causal)
    # the plain inner GD can grow large at eta ~ 1 (GELU more so): compare relative
    # to the values' size, at fp64 rounding level
    np.testing.assert_allclose(z[0, 0], zr.numpy(), rtol=1e-11, atol=1e-12)
    for got, ref in zip([W1o, c1o, W2o, c2o], Pr):
        np.testing.assert_allclose(got[0, 0], ref.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("activation", ["silu", "gelu"])
@pytest.mark.parametrize("b,causal", [(1, True), (16, True), (6, True), (16, False), (40, False)])
def test_mlp_dual_form_equals_primal(b, causal, activation):
    B, H, T, d, m = 1, 2, 41, 8, 32
    q, k, v = _qkv(B, H, T, d)
    W1, c1, W2, c2 = _mlp_params(H, d, m, scale=0.2)
    eta = rng.uniform(0.02, 0.15, (B, H, T))   # keeps the inner dynamics bounded
    z, W1o, c1o, W2o, c2o = oracle.mlp(q, k, v, W1, c1, W2, c2, b=b, causal=causal, eta=eta,
                                       activation=activation)
    for h in range(H):
        zr, (a, ca, bm, cb) = _defs.dual_mlp(q[0, h], k[0, h], v[0, h], W1[h], c1[h], W2[h],
                                             c2[h], eta[0, h], b, causal, activation)
        np.testing.assert_allclose(z[0, h], zr, atol=1e-11)
        for got, ref in zip([W1o, c1o, W2o, c2o], [a, ca, bm, cb]):
            np.testing.assert_allclose(got[0, h], ref, atol=1e-11)


def test_mlp_full_batch_is_one_gd_step():
    B, H, T, d, m = 2, 1, 9, 4, 16
    q, k, v = _qkv(B, H, T, d)
    W1, c1, W2, c2 = _mlp_params(H, d, m)
    z, W1o, c1o, W2o, c2o = oracle.mlp(q, k, v, W1, c1, W2, c2, b=T, causal=False,
                                       eta_scalar=1.0)
    for bi in range(B):
        P = [torch.tensor(p[0], requires_grad=True) for p in (W1, c1, W2, c2)]
        K, V, Q = (torch.tensor(x[bi, 0]) for x in (k, v, q))
        L = 0.5 * ((_defs.f_mlp(K, P) - V) ** 2).sum()
        gs = torch.autograd.grad(L, P)
        P1 = [(p - g).detach() for p, g in zip(P, gs)]
        for got, ref in zip([W1o, c1o, W2o, c2o], P1):
            np.testing.assert_allclose(got[bi, 0], ref.numpy(), atol=1e-12)
        np.testing.assert_allclose(z[bi, 0], _defs.f_mlp(Q, P1).numpy(), atol=1e-12)


def test_mlp_eta_zero_is_identity():
    B, H, T, d, m = 1, 1, 5, 4, 8
    q, k, v = _qkv(B, H, T, d)
    W1, c1, W2, c2 = _mlp_params(H, d, m)
    z, W1o, *_ = oracle.mlp(q, k, v, W1, c1, W2, c2, b=2, eta_scalar=0.0)
    np.testing.assert_array_equal(W1o[0], W1)
    P = [torch.tensor(p[0]) for p in (W1, c1, W2, c2)]
    np.testing.assert_allclose(z[0, 0], _defs.f_mlp(torch.tensor(q[0, 0]), P).numpy(), atol=1e-13)


def test_empty_sequence():
    q = np.zeros((1, 1, 0, 4))
    W0 = rng.standard_normal((1, 4, 4))
    z, Wf = oracle.linear(q, q, q, W0, b=4)
    assert z.shape == (1, 1, 0, 4)
    np.testing.assert_array_equal(Wf[0], W0)


# ------------------------------------------------ depthwise convolution inner model


def _dw_torch(x, W, hh, ww):
    """Depthwise 3x3 'same' cross-correlation of a [N,d] token map (row-major grid)
    with taps W [9,d], by torch.nn.functional.conv2d (groups = d)."""
    N, d = x.shape
    img = x.T.reshape(1, d, hh, ww)
    w = W.T.reshape(d, 1, 3, 3)
    return torch.nn.functional.conv2d(img, w, padding=1, groups=d).reshape(d, N).T


@pytest.mark.parametrize("epochs", [1, 2])
@pytest.mark.parametrize("hh,ww", [(4, 5), (3, 3), (1, 6)])
def test_dwconv_full_batch_steps_by_autograd(hh, ww, epochs):
    """Depthwise-convolution inner model (ViT3 article, observation 6), full-batch
    MSE steps: W_{e+1} = W_e - grad(sum_p eta_p 1/2 ||f(K)_p - v_p||^2) by autograd
    through torch's grouped conv2d; every query reads the last W."""
    B, H, d = 1, 2, 3
    N = hh * ww
    q, k, v = _qkv(B, H, N, d)
    eta = rng.uniform(0.2, 1.0, (B, H, N))
    W0 = rng.standard_normal((H, 9, d)) * 0.3
    z, Wf = oracle.dwconv(q, k, v, W0, hh, ww, eta=eta, epochs=epochs)
    for h in range(H):
        W = torch.tensor(W0[h])
        K, V, Q = (torch.tensor(x[0, h]) for x in (k, v, q))
        for _ in range(epochs):
            Wg = W.clone().requires_grad_(True)
            L = (torch.tensor(eta[0, h])[:, None] * 0.5 * (_dw_torch(K, Wg, hh, ww) - V) ** 2).sum()
            (g,) = torch.autograd.grad(L, Wg)
            W = (Wg - g).detach()
        np.testing.assert_allclose(Wf[0, h], W.numpy(), atol=1e-12)
        np.testing.assert_allclose(z[0, h], _dw_torch(Q, W, hh, ww).numpy(), atol=1e-12)


def test_dwconv_dot_loss_closed_form():
    """Dot loss: W1[o][c] = W0[o][c] + eta sum_p v_p[c] K[p + o][c], written here with
    explicit zero padding of the grid."""
    B, H, hh, ww, d = 2, 1, 3, 4, 2
    q, k, v = _qkv(B, H, hh * ww, d, unit=False)
    W0 = rng.standard_normal((H, 9, d))
    z, Wf = oracle.dwconv(q, k, v, W0, hh, ww, eta_scalar=0.5, loss="dot")
    for bi in range(B):
        Kp = np.zeros((hh + 2, ww + 2, d))
        Kp[1:-1, 1:-1] = k[bi, 0].reshape(hh, ww, d)
        V = v[bi, 0].reshape(hh, ww, d)
        W = W0[0].copy()
        for o in range(9):
            di, dj = o // 3, o % 3
            W[o] += 0.5 * (V * Kp[di:di + hh, dj:dj + ww]).sum((0, 1))
        np.testing.assert_allclose(Wf[bi, 0], W, atol=1e-12)
        Qp = np.zeros((hh + 2, ww + 2, d))
        Qp[1:-1, 1:-1] = q[bi, 0].reshape(hh, ww, d)
        Z = sum(Qp[o // 3:o // 3 + hh, o % 3:o % 3 + ww] * W[o] for o in range(9))
        np.testing.assert_allclose(z[bi, 0], Z.reshape(hh * ww, d), atol=1e-12)


# ---------------------------------------------- inner layer norm + residual (Linear)


@pytest.mark.parametrize("T,b,causal", [(11, 1, True), (11, 4, True), (12, 4, False), (9, 9, False),
                                        (10, 16, True)])
def test_linear_layer_norm_residual_matches_definition_autograd(T, b, causal):
    """f(x; W) = x + LN(x W) (the walkthrough's TTT-Linear, section 2.2.1): the
    oracle's hand LN backward equals the layer's definition evaluated with torch's
    layer_norm and autograd, every mini-batch size, both masks."""
    B, H, d = 1, 2, 6
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.1, 1.0, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.3
    gam = rng.uniform(0.5, 1.5, (H, d))
    bet = rng.standard_normal((H, d)) * 0.1
    z, Wf = oracle.linear(q, k, v, W0, b, causal=causal, eta=eta, ln_gamma=gam, ln_beta=bet)
    t = lambda a: torch.tensor(a)
    for h in range(H):
        f = _defs.make_f_linear_ln(t(gam[h]), t(bet[h]))
        zr, (Wr,) = _defs.definition_autograd(f, [t(W0[h])], t(q[0, h]), t(k[0, h]), t(v[0, h]),
                                              t(eta[0, h]), b, causal)
        np.testing.assert_allclose(z[0, h], zr.numpy(), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(Wf[0, h], Wr.numpy(), rtol=1e-10, atol=1e-11)


def test_linear_layer_norm_needs_mse():
    q, k, v = _qkv(1, 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.linear(q, k, v, np.zeros((1, 4, 4)), 2, loss="dot", ln_gamma=np.ones((1, 4)),
                      ln_beta=np.zeros((1, 4)))


# ------------------------------------------------- input-dependent learning rate

def _logit(eta, eta_base):
    p = eta / eta_base
    return np.log(p) - np.log1p(-p)


def test_eta_gate_zero_vector_is_half_the_base_rate():
    """theta = 0: sigma(0) = 1/2 for every token, exactly."""
    x = rng.standard_normal((2, 7, 24))
    eta = oracle.eta_gate(x, np.zeros((3, 24)), eta_base=0.1)
    assert eta.shape == (2, 3, 7)
    assert np.all(eta == 0.05)


def test_eta_gate_one_hot_vectors_read_one_feature_per_head():
    """theta[h] = c_h e_{j_h}: the logit of eta[b,h,t] / eta_base is c_h x[b,t,j_h]
    (pins which axis of x is the feature axis and which row of theta each head uses)."""
    B, T, dm, H = 3, 11, 40, 4
    x = rng.standard_normal((B, T, dm))
    js, cs = [3, 17, 0, 39], [0.5, -1.25, 2.0, 0.75]
    theta = np.zeros((H, dm))
    for h in range(H):
        theta[h, js[h]] = cs[h]
    eta = oracle.eta_gate(x, theta, eta_base=1.0)
    for h in range(H):
        np.testing.assert_allclose(_logit(eta[:, h, :], 1.0), cs[h] * x[:, :, js[h]], rtol=1e-10, atol=1e-12)


def test_eta_gate_logit_is_linear_in_the_vector():
    """logit(eta(theta1 + theta2)) = logit(eta(theta1)) + logit(eta(theta2)): the gate's
    argument is a full dot product (no dropped or repeated feature)."""
    B, T, dm, H = 2, 9, 72, 3
    x = rng.standard_normal((B, T, dm))
    t1, t2 = 0.05 * rng.standard_normal((H, dm)), 0.05 * rng.standard_normal((H, dm))
    e1, e2, e12 = (oracle.eta_gate(x, t, 1.0) for t in (t1, t2, t1 + t2))
    np.testing.assert_allclose(_logit(e12, 1.0), _logit(e1, 1.0) + _logit(e2, 1.0), rtol=1e-9, atol=1e-12)


def test_eta_gate_symmetry_and_saturation():
    """sigma(a) + sigma(-a) = 1, so eta(theta) + eta(-theta) = eta_base; a large
    argument gives the base rate (sigma(40) rounds to 1 in double precision)."""
    x = rng.standard_normal((2, 6, 16))
    th = rng.standard_normal((5, 16))
    np.testing.assert_allclose(oracle.eta_gate(x, th, 0.1) + oracle.eta_gate(x, -th, 0.1), 0.1, rtol=1e-14)
    ones = np.ones((1, 3, 4))
    assert np.all(oracle.eta_gate(ones, np.full((1, 4), 10.0), 1.0) == 1.0)
    assert np.all(oracle.eta_gate(ones, np.full((1, 4), -10.0), 1.0) < 1e-17)


# ------------------------------------------------ inner layer norm + residual (MLP)


@pytest.mark.parametrize("activation", ["silu", "gelu"])
@pytest.mark.parametrize("T,b,causal", [(11, 1, True), (11, 4, True), (12, 4, False), (9, 9, False),
                                        (10, 16, True)])
def test_mlp_layer_norm_residual_matches_definition_autograd(T, b, causal, activation):
    """f(x) = x + LN(act(x W1 + c1) W2 + c2) (the walkthrough's TTT-MLP, section 2.2.1):
    the oracle's hand LN backward, fed into the MLP's backward, equals the layer's
    definition with torch's layer_norm and autograd, every mini-batch size, both masks."""
    B, H, d, m = 1, 2, 6, 16
    q, k, v = _qkv(B, H, T, d)
    W1, c1, W2, c2 = _mlp_params(H, d, m)
    eta = rng.uniform(0.1, 1.0, (B, H, T))
    gam = rng.uniform(0.5, 1.5, (H, d))
    bet = rng.standard_normal((H, d)) * 0.1
    out = oracle.mlp(q, k, v, W1, c1, W2, c2, b=b, causal=causal, eta=eta, activation=activation,
                     ln_gamma=gam, ln_beta=bet)
    t = lambda a: torch.tensor(a)
    for h in range(H):
        f = _defs.make_f_mlp_ln(t(gam[h]), t(bet[h]), activation)
        zr, Pr = _defs.definition_autograd(f, [t(W1[h]), t(c1[h]), t(W2[h]), t(c2[h])], t(q[0, h]),
                                           t(k[0, h]), t(v[0, h]), t(eta[0, h]), b, causal)
        np.testing.assert_allclose(out[0][0, h], zr.numpy(), rtol=1e-10, atol=1e-11)
        for got, ref in zip(out[1:], Pr):
            np.testing.assert_allclose(got[0, h], ref.numpy(), rtol=1e-10, atol=1e-11)


# ------------------------------------------- block (several mini-batches) form


@pytest.mark.parametrize("T,b,nb", [(64, 16, 4), (70, 16, 4), (45, 4, 3), (33, 8, 1), (50, 5, 10)])
def test_linear_block_form_equals_token_loop(T, b, nb):
    """Causal TTT-Linear rewritten per block of nb mini-batches as one affine state map
    (a block-unit-triangular solve for the steps, then W <- (I + K^T P) W + K^T C): equal
    to the oracle's token loop to fp64 rounding, ragged tails included."""
    B, H, d = 1, 2, 8
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.1, 1.0, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.3
    z, Wf = oracle.linear(q, k, v, W0, b, causal=True, eta=eta)
    for h in range(H):
        zb, Wb = _defs.block_form_linear(q[0, h], k[0, h], v[0, h], W0[h], eta[0, h], b, nb)
        np.testing.assert_allclose(zb, z[0, h], rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(Wb, Wf[0, h], rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("T,C", [(16, 16), (48, 16), (57, 16), (5, 16), (40, 8)])
def test_chunked_delta_rule_equals_token_loop(T, C):
    """The delta rule (b = 1) in chunks of C tokens, as the chunked kernel computes it: the
    residuals at the chunk's start weights, a forward substitution through the strictly
    lower (k_t . k_s) eta_s, then the mini-batch output and update with the solved
    residuals; equal to the oracle's token loop to fp64 rounding, ragged tails included."""
    B, H, d = 1, 2, 8
    q, k, v = _qkv(B, H, T, d)
    eta = rng.uniform(0.1, 1.0, (B, H, T))
    W0 = rng.standard_normal((H, d, d)) * 0.3
    z, Wf = oracle.linear(q, k, v, W0, 1, causal=True, eta=eta)
    for h in range(H):
        zc, Wc = _defs.chunked_delta_rule(q[0, h], k[0, h], v[0, h], W0[h], eta[0, h], C)
        np.testing.assert_allclose(zc, z[0, h], rtol=1e-9, atol=1e-10)
        np.testing.assert_allclose(Wc, Wf[0, h], rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("nb", [1, 2, 4])
def test_block_form_triangular_factor_is_a_finite_series(nb):
    """L is block-strictly-lower over nb mini-batches, so L^nb = 0 and (I + L)^-1 is the
    finite series I - L + L^2 - ... (Horner: I - L(I - L(...))): no solve on chip."""
    b, d = 16, 8
    n = b * nb
    K = _unit(rng.standard_normal((n, d)))
    et = rng.uniform(0.1, 1.0, n)
    mb = np.arange(n) // b
    L = (mb[:, None] > mb[None, :]) * (et[:, None] * (K @ K.T))
    assert np.abs(np.linalg.matrix_power(L, nb)).max() == 0.0
    T = np.eye(n)
    for _ in range(nb - 1):
        T = np.eye(n) - L @ T
    np.testing.assert_allclose(T, np.linalg.inv(np.eye(n) + L), rtol=1e-12, atol=1e-13)


def _norm_full_batch_spread(eta):
    """max |z(W) - z(bf16(W))| / max |z| of the fp64 full-batch TTT-MLP with the inner
    norm on the GPU tests' B2 H8 T150 inputs: only the start weights are rounded."""
    import torch
    from test_sequence_layers_gb300 import synth
    B, H, T, seed = 2, 8, 150, 452
    inp = synth.make("mlp", B=B, H=H, T=T, d=64, m=256, b=T, causal=False, eta=eta, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    inp.params["c1"] = torch.randn(inp.params["c1"].shape, generator=g) * 0.1
    inp.params["c2"] = torch.randn(inp.params["c2"].shape, generator=g) * 0.1
    g = torch.Generator().manual_seed(seed + 1)
    gam = 1.0 + 0.1 * torch.randn((H, 64), generator=g)
    bet = 0.1 * torch.randn((H, 64), generator=g)
    P = [inp.params[n] for n in ("W1", "c1", "W2", "c2")]
    z0, *_ = oracle.mlp(inp.q, inp.k, inp.v, *P, T, False, eta_scalar=eta, ln_gamma=gam, ln_beta=bet)
    Pb = [x.to(torch.bfloat16).float() for x in P]
    z1, *_ = oracle.mlp(inp.q, inp.k, inp.v, *Pb, T, False, eta_scalar=eta, ln_gamma=gam, ln_beta=bet)
    return np.abs(z1 - z0).max() / np.abs(z0).max()


def test_mlp_norm_full_batch_conditioning():
    """The inner norm divides by each output row's spread, so at a large inner step z
    carries bf16 rounding of the weights on amplified (the reason the full-batch norm
    GPU tests run at eta = 0.1): > 1 % at eta = 0.2, < 0.5 % at eta = 0.1."""
    assert _norm_full_batch_spread(0.2) > 0.01
    assert _norm_full_batch_spread(0.1) < 0.005
