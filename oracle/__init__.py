"""fp64 CPU oracle for the TTT layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product path.

The arithmetic lives in ``ttt_oracle.c`` (a plain token-by-token loop in double
precision; see the header of that file for the definition it follows and the
passages of the pages it cites).  This module only compiles it with gcc, marshals
arrays to contiguous float64 and calls it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ttt_oracle.c")
_LIB = os.path.join(_HERE, "libttt_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library in place (plain -O2, no tuning)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i, d, ll = ctypes.c_int, ctypes.c_double, ctypes.c_longlong
        lib.ttt_oracle_linear.argtypes = [i, i, i, i, i, i, i, i, dp, dp, dp, dp, d, dp, ll, dp, dp, i,
                                          dp, dp, d]
        lib.ttt_oracle_linear.restype = i
        lib.ttt_oracle_mlp.argtypes = [i, i, i, i, i, i, i, dp, dp, dp, dp, d,
                                       dp, dp, dp, dp, i, dp, dp, dp, dp, dp, i, i, dp, dp, d]
        lib.ttt_oracle_mlp.restype = i
        lib.ttt_oracle_dwconv.argtypes = [i, i, i, i, i, i, i, dp, dp, dp, dp, d, dp, ll, dp, dp, i]
        lib.ttt_oracle_dwconv.restype = i
        lib.ttt_oracle_eta_gate.argtypes = [i, i, i, i, dp, dp, d, dp]
        lib.ttt_oracle_eta_gate.restype = i
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: upcast exactly on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return os.cpu_count() or 1


def linear(q, k, v, W0, b, causal=True, eta=None, eta_scalar=1.0, loss="mse",
           threads=None, epochs=1, ln_gamma=None, ln_beta=None, ln_eps=1e-6):
    """TTT-Linear forward, fp64.  q,k,v: [B,H,T,d]; W0: [H,d,d] (shared over the
    batch) or [B,H,d,d]; eta: [B,H,T] or None (then eta_scalar for every token);
    loss "mse" or "dot"; epochs > 1 only with causal=False and b >= T (repeated
    full-batch steps); ln_gamma, ln_beta [H,d]: inner model x + LN(x W) (MSE only).  Returns (z [B,H,T,d], W_final [B,H,d,d]) as float64 numpy
    arrays."""
    q, k, v, W0, eta = _f64(q), _f64(k), _f64(v), _f64(W0), _f64(eta)
    B, H, T, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    if W0.ndim == 3:
        assert W0.shape == (H, d, d)
        w0_bstride = 0
    else:
        assert W0.shape == (B, H, d, d)
        w0_bstride = H * d * d
    if eta is not None:
        assert eta.shape == (B, H, T)
    z = np.zeros((B, H, T, d))
    Wf = np.zeros((B, H, d, d))
    gam, bet = _f64(ln_gamma), _f64(ln_beta)
    if gam is not None:
        assert gam.shape == (H, d) and bet.shape == (H, d)
    rc = _load().ttt_oracle_linear(B, H, T, d, int(b), 1 if causal else 0,
                                   {"mse": 0, "dot": 1}[loss], int(epochs),
                                   _ptr(q), _ptr(k), _ptr(v), _ptr(eta), float(eta_scalar),
                                   _ptr(W0), w0_bstride, _ptr(z), _ptr(Wf),
                                   threads or default_threads(), _ptr(gam), _ptr(bet), float(ln_eps))
    if rc != 0:
        raise ValueError("ttt_oracle_linear rejected its arguments")
    return z, Wf


def mlp(q, k, v, W1, c1, W2, c2, b, causal=True, eta=None, eta_scalar=0.1, threads=None,
        activation="silu", ln_gamma=None, ln_beta=None, ln_eps=1e-6):
    """TTT-MLP forward, fp64, f(x) = act(x W1 + c1) W2 + c2, act "silu" or "gelu"
    (erf form); with ln_gamma, ln_beta [H,d]: f(x) = x + LN(act(x W1 + c1) W2 + c2).
    Parameters are given per head ([H,...], shared over the batch) or per (batch,
    head) ([B,H,...]).  Returns (z, W1_final, c1_final, W2_final, c2_final)."""
    q, k, v, eta = _f64(q), _f64(k), _f64(v), _f64(eta)
    W1, c1, W2, c2 = _f64(W1), _f64(c1), _f64(W2), _f64(c2)
    B, H, T, d = q.shape
    m = W1.shape[-1]
    per_batch = 1 if W1.ndim == 4 else 0
    lead = (B, H) if per_batch else (H,)
    assert W1.shape == lead + (d, m) and c1.shape == lead + (m,)
    assert W2.shape == lead + (m, d) and c2.shape == lead + (d,)
    if eta is not None:
        assert eta.shape == (B, H, T)
    gam, bet = _f64(ln_gamma), _f64(ln_beta)
    if gam is not None:
        assert gam.shape == (H, d) and bet.shape == (H, d)
    z = np.zeros((B, H, T, d))
    W1o, c1o = np.zeros((B, H, d, m)), np.zeros((B, H, m))
    W2o, c2o = np.zeros((B, H, m, d)), np.zeros((B, H, d))
    rc = _load().ttt_oracle_mlp(B, H, T, d, m, int(b), 1 if causal else 0,
                                _ptr(q), _ptr(k), _ptr(v), _ptr(eta), float(eta_scalar),
                                _ptr(W1), _ptr(c1), _ptr(W2), _ptr(c2), per_batch,
                                _ptr(z), _ptr(W1o), _ptr(c1o), _ptr(W2o), _ptr(c2o),
                                threads or default_threads(), {"silu": 0, "gelu": 1}[activation],
                                _ptr(gam), _ptr(bet), float(ln_eps))
    if rc != 0:
        raise ValueError("ttt_oracle_mlp rejected its arguments")
    return z, W1o, c1o, W2o, c2o


def dwconv(q, k, v, W0, height, width, eta=None, eta_scalar=1.0, loss="mse", epochs=1,
           threads=None):
    """Depthwise 3x3 convolution inner model, full-batch inner GD (non-causal), fp64.
    q,k,v: [B,H,N,d] with N = height*width tokens in row-major grid order; W0:
    [H,9,d] (shared over the batch) or [B,H,9,d], tap o = (di+1)*3 + (dj+1).
    Returns (z [B,H,N,d], W_final [B,H,9,d])."""
    q, k, v, W0, eta = _f64(q), _f64(k), _f64(v), _f64(W0), _f64(eta)
    B, H, N, d = q.shape
    assert N == height * width and k.shape == q.shape and v.shape == q.shape
    if W0.ndim == 3:
        assert W0.shape == (H, 9, d)
        w0_bstride = 0
    else:
        assert W0.shape == (B, H, 9, d)
        w0_bstride = H * 9 * d
    z = np.zeros((B, H, N, d))
    Wf = np.zeros((B, H, 9, d))
    rc = _load().ttt_oracle_dwconv(B, H, height, width, d, {"mse": 0, "dot": 1}[loss], int(epochs),
                                   _ptr(q), _ptr(k), _ptr(v), _ptr(eta), float(eta_scalar),
                                   _ptr(W0), w0_bstride, _ptr(z), _ptr(Wf),
                                   threads or default_threads())
    if rc != 0:
        raise ValueError("ttt_oracle_dwconv rejected its arguments")
    return z, Wf


def eta_gate(x, theta, eta_base=1.0):
    """Input-dependent inner learning rate, fp64: eta[b,h,t] = eta_base *
    sigma(theta[h] . x[b,t]).  x: [B,T,dm] (the layer's input tokens); theta: [H,dm]
    (one learnable vector per head).  Returns eta [B,H,T] as a float64 numpy array."""
    x, theta = _f64(x), _f64(theta)
    B, T, dm = x.shape
    H = theta.shape[0]
    assert theta.shape == (H, dm)
    eta = np.zeros((B, H, T))
    rc = _load().ttt_oracle_eta_gate(B, T, H, dm, _ptr(x), _ptr(theta), float(eta_base), _ptr(eta))
    if rc != 0:
        raise ValueError("ttt_oracle_eta_gate rejected its arguments")
    return eta
