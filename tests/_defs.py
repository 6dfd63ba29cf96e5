"""Independent restatements used to pin the oracle (test-side only).

Nothing here is shared with the oracle or with the CUDA path.  Each helper is a
different route to a value the pages fix: autograd instead of hand gradients,
the column-convention delta rule as printed, brute-force attention sums, and the
matrix ("dual") form of a mini-batch step.
"""
import numpy as np
import torch


def silu_t(x):
    return x * torch.sigmoid(x)


def f_linear(x, P):
    return x @ P[0]


def f_mlp(x, P):
    W1, c1, W2, c2 = P
    return silu_t(x @ W1 + c1) @ W2 + c2


def make_f_linear_ln(gamma, beta, eps=1e-6):
    """f(x; W) = x + LN(x W) with fixed scale / shift (torch's layer_norm)."""
    def f(x, P):
        y = x @ P[0]
        return x + torch.nn.functional.layer_norm(y, (y.shape[-1],), gamma, beta, eps)
    return f


def make_f_mlp_ln(gamma, beta, activation="silu", eps=1e-6):
    """f(x) = x + LN(act(x W1 + c1) W2 + c2) with fixed scale / shift (torch's layer_norm)."""
    act = silu_t if activation == "silu" else torch.nn.functional.gelu

    def f(x, P):
        W1, c1, W2, c2 = P
        y = act(x @ W1 + c1) @ W2 + c2
        return x + torch.nn.functional.layer_norm(y, (y.shape[-1],), gamma, beta, eps)
    return f


def f_mlp_gelu(x, P):
    W1, c1, W2, c2 = P
    return torch.nn.functional.gelu(x @ W1 + c1) @ W2 + c2


def definition_autograd(f, P0, q, k, v, eta, b, causal):
    """The layer exactly as defined, one chain, fp64 torch, gradients by autograd.

    W_t = W_start - grad_W( sum_{s in block, s <= t} eta_s * 1/2 ||f(k_s;W) - v_s||^2 )
    evaluated at the block's start weights; z_t = f(q_t; W_t) (causal) or
    f(q_t; W_end of the block) (non-causal).  q,k,v: [T,d]; eta: [T]."""
    T = q.shape[0]
    P = [p.clone() for p in P0]
    z = torch.zeros(T, v.shape[1], dtype=torch.float64)

    def step(Ps, lo, hi):
        Ps = [p.detach().clone().requires_grad_(True) for p in Ps]
        L = sum(eta[s] * 0.5 * ((f(k[s:s + 1], Ps) - v[s:s + 1]) ** 2).sum()
                for s in range(lo, hi))
        gs = torch.autograd.grad(L, Ps)
        return [(p - g).detach() for p, g in zip(Ps, gs)]

    for n0 in range(0, T, b):
        n1 = min(n0 + b, T)
        if causal:
            for t in range(n0, n1):
                Pt = step(P, n0, t + 1)
                z[t] = f(q[t:t + 1], Pt)[0]
        P_end = step(P, n0, n1)
        if not causal:
            for t in range(n0, n1):
                z[t] = f(q[t:t + 1], P_end)[0]
        P = P_end
    return z, P


def dual_linear(q, k, v, W0, eta, b, causal):
    """Mini-batch step in matrix form, numpy fp64, one chain (q,k,v [T,d], eta [T]).
    E = K W - V;  Z = Q W - M.(Q K^T) diag(eta) E;  W <- W - K^T diag(eta) E."""
    T, d = q.shape
    W = W0.copy()
    z = np.zeros((T, d))
    for n0 in range(0, T, b):
        n1 = min(n0 + b, T)
        Q, K, V, et = q[n0:n1], k[n0:n1], v[n0:n1], eta[n0:n1]
        M = np.tril(np.ones((n1 - n0, n1 - n0))) if causal else np.ones((n1 - n0, n1 - n0))
        E = K @ W - V
        Et = et[:, None] * E
        z[n0:n1] = Q @ W - (M * (Q @ K.T)) @ Et
        W = W - K.T @ Et
    return z, W


def block_form_linear(q, k, v, W0, eta, b, nb):
    """Causal TTT-Linear over blocks of nb mini-batches of b tokens each, numpy fp64, one
    chain (q,k,v [T,d], eta [T]); the state moves once per block by a dense affine map.

    With U_i = -diag(eta_i) (K_i W_i - V_i) the step of mini-batch i and W_i = W + sum_{j<i}
    K_j^T U_j (W the block's start state), the steps of a block solve the block-unit-
    lower-triangular system (I + L) U = -diag(eta) (K W - V), L_ij = diag(eta_i) K_i K_j^T
    for j < i.  With T = (I + L)^-1:  U = P W + C, P = -T diag(eta) K, C = T diag(eta) V,
        W_next = (I + K^T P) W + K^T C                   (the only serial product)
        Z      = (Q + M.(Q K^T) P) W + M.(Q K^T) C       (M: key s <= query t)
    so everything but one d x d product per block is independent of the state."""
    T, d = q.shape
    W = W0.copy()
    z = np.zeros((T, d))
    L = b * nb
    for s0 in range(0, T, L):
        s1 = min(s0 + L, T)
        n = s1 - s0
        Q, K, V, et = q[s0:s1], k[s0:s1], v[s0:s1], eta[s0:s1]
        mb = np.arange(n) // b                           # mini-batch of each token
        Lm = (mb[:, None] > mb[None, :]) * (et[:, None] * (K @ K.T))
        Tinv = np.linalg.solve(np.eye(n) + Lm, np.eye(n))
        P = -Tinv @ (et[:, None] * K)
        C = Tinv @ (et[:, None] * V)
        M = np.tril(np.ones((n, n)))
        S = M * (Q @ K.T)
        z[s0:s1] = (Q + S @ P) @ W + S @ C
        W = (np.eye(d) + K.T @ P) @ W + K.T @ C
    return z, W


def chunked_delta_rule(q, k, v, W0, eta, C=16):
    """The delta rule (mini-batches of one token) in chunks of C tokens, numpy fp64, one
    chain (q,k,v [T,d], eta [T]), in the order of the chunked kernel's steps.  With W the
    chunk's start weights and R = K W - V, token t's residual at its own weights is
    e_t = r_t - sum_{s<t} eta_s (k_t . k_s) e_s, i.e. (I + A) E = R with A strictly lower,
    A_ts = (k_t . k_s) eta_s, solved by forward substitution (after e_s is final, every
    later row loses A_ts e_s).  Then, as in a mini-batch step with the solved E,
        Z = Q W - tril(Q K^T) diag(eta) E      (tril keeps key s <= query t)
        W <- W - K^T diag(eta) E."""
    T, d = q.shape
    W = W0.copy()
    z = np.zeros((T, d))
    for n0 in range(0, T, C):
        n1 = min(n0 + C, T)
        n = n1 - n0
        Q, K, V, et = q[n0:n1], k[n0:n1], v[n0:n1], eta[n0:n1]
        E = K @ W - V
        A = np.tril(K @ K.T, -1) * et[None, :]
        for s in range(n - 1):
            E[s + 1:] -= A[s + 1:, s:s + 1] * E[s:s + 1]
        Et = et[:, None] * E
        z[n0:n1] = Q @ W - (np.tril(np.ones((n, n))) * (Q @ K.T)) @ Et
        W = W - K.T @ Et
    return z, W


def dual_mlp(q, k, v, W1, c1, W2, c2, eta, b, causal, activation="silu"):
    """TTT-MLP mini-batch step in matrix form (numpy fp64, one chain).  The "+1"
    terms carry the bias writes: c_t = c - sum_{s<=t} eta_s * grad_c l_s."""
    from scipy.special import erf
    sig = lambda x: 1.0 / (1.0 + np.exp(-x))
    if activation == "silu":
        act = lambda x: x * sig(x)
        dact = lambda x: sig(x) * (1 + x * (1 - sig(x)))
    else:
        Phi = lambda x: 0.5 * (1 + erf(x / np.sqrt(2)))
        act = lambda x: x * Phi(x)
        dact = lambda x: Phi(x) + x * np.exp(-0.5 * x * x) / np.sqrt(2 * np.pi)
    T, d = q.shape
    W1, c1, W2, c2 = W1.copy(), c1.copy(), W2.copy(), c2.copy()
    z = np.zeros((T, d))
    for n0 in range(0, T, b):
        n1 = min(n0 + b, T)
        Q, K, V, et = q[n0:n1], k[n0:n1], v[n0:n1], eta[n0:n1][:, None]
        n = n1 - n0
        M = np.tril(np.ones((n, n))) if causal else np.ones((n, n))
        Hk = K @ W1 + c1
        Ak = act(Hk)
        E = Ak @ W2 + c2 - V
        D = (E @ W2.T) * dact(Hk)
        Et, Dt = et * E, et * D
        Hq = Q @ W1 + c1 - (M * (Q @ K.T + 1)) @ Dt
        Aq = act(Hq)
        z[n0:n1] = Aq @ W2 + c2 - (M * (Aq @ Ak.T + 1)) @ Et
        W2 = W2 - Ak.T @ Et
        c2 = c2 - Et.sum(0)
        W1 = W1 - K.T @ Dt
        c1 = c1 - Dt.sum(0)
    return z, (W1, c1, W2, c2)
