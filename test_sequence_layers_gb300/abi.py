"""ctypes binding of libttt (include/ttt.h): argument marshalling only.

Every step of the layer runs in the CUDA library; this module checks shapes and
dtypes, allocates outputs with PyTorch (device memory and streams are PyTorch's
job here) and passes raw pointers.  There is no fallback: if the library is
missing or a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libttt.so")

TTT_F32, TTT_BF16 = 0, 1
STATUS = {0: "TTT_OK", -1: "TTT_ERR_ARG", -2: "TTT_ERR_UNSUPPORTED", -3: "TTT_ERR_ALIGN",
          -4: "TTT_ERR_LAUNCH", -5: "TTT_ERR_TIMEOUT", -6: "TTT_ERR_SCRATCH"}

# every symbol include/ttt.h declares
EXPORTS = ("ttt_linear_fwd", "ttt_linear_seqpar_workspace", "ttt_linear_fwd_seqpar",
           "ttt_linear_fwd_seqpar_noalloc", "ttt_dwconv_fwd", "ttt_eta_gate",
           "ttt_mlp_fwd", "ttt_sync_status", "ttt_status_str", "ttt_launch_count",
           "ttt_debug_wait_limit")


class LinearDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("d", ctypes.c_int), ("mini_batch", ctypes.c_int), ("causal", ctypes.c_int),
                ("io_dtype", ctypes.c_int), ("w0_batch_stride", ctypes.c_longlong),
                ("loss", ctypes.c_int), ("epochs", ctypes.c_int),
                ("ln_gamma", ctypes.c_void_p), ("ln_beta", ctypes.c_void_p), ("ln_eps", ctypes.c_float)]

LOSSES = {"mse": 0, "dot": 1}


class DwconvDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("height", ctypes.c_int),
                ("width", ctypes.c_int), ("d", ctypes.c_int), ("io_dtype", ctypes.c_int),
                ("loss", ctypes.c_int), ("epochs", ctypes.c_int),
                ("w0_batch_stride", ctypes.c_longlong)]


class MlpDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("d", ctypes.c_int), ("m", ctypes.c_int), ("mini_batch", ctypes.c_int),
                ("causal", ctypes.c_int), ("io_dtype", ctypes.c_int),
                ("params_per_batch", ctypes.c_int), ("activation", ctypes.c_int),
                ("ln_gamma", ctypes.c_void_p), ("ln_beta", ctypes.c_void_p), ("ln_eps", ctypes.c_float)]

ACTIVATIONS = {"silu": 0, "gelu": 1}


class GateDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("dm", ctypes.c_int)]


class TTTError(RuntimeError):
    def __init__(self, fn, rc):
        self.code = rc
        super().__init__(f"{fn} returned {STATUS.get(rc, rc)}: {status_str(rc)}")


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libttt.so is missing ({LIB_PATH}); run "
                               "`python -m test_sequence_layers_gb300.build` first")
        L = ctypes.CDLL(LIB_PATH)
        vp, fp, f = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float
        L.ttt_linear_fwd.argtypes = [ctypes.POINTER(LinearDesc), vp, vp, vp, fp, f, fp, vp, fp, vp]
        L.ttt_linear_fwd.restype = ctypes.c_int
        L.ttt_linear_seqpar_workspace.argtypes = [ctypes.POINTER(LinearDesc)]
        L.ttt_linear_seqpar_workspace.restype = ctypes.c_size_t
        L.ttt_linear_fwd_seqpar.argtypes = [ctypes.POINTER(LinearDesc), vp, vp, vp, fp, f, fp, vp, fp,
                                            vp, ctypes.c_size_t, vp]
        L.ttt_linear_fwd_seqpar.restype = ctypes.c_int
        L.ttt_linear_fwd_seqpar_noalloc.argtypes = [ctypes.POINTER(LinearDesc), vp, vp, vp, fp, f, fp, vp,
                                                    fp, vp]
        L.ttt_linear_fwd_seqpar_noalloc.restype = ctypes.c_int
        L.ttt_dwconv_fwd.argtypes = [ctypes.POINTER(DwconvDesc), vp, vp, vp, fp, f, fp, vp, fp, vp]
        L.ttt_dwconv_fwd.restype = ctypes.c_int
        L.ttt_mlp_fwd.argtypes = [ctypes.POINTER(MlpDesc), vp, vp, vp, fp, f, fp, fp, fp, fp,
                                  vp, fp, fp, fp, fp, vp]
        L.ttt_mlp_fwd.restype = ctypes.c_int
        L.ttt_eta_gate.argtypes = [ctypes.POINTER(GateDesc), vp, vp, f, fp, vp]
        L.ttt_eta_gate.restype = ctypes.c_int
        L.ttt_sync_status.argtypes = [vp]
        L.ttt_sync_status.restype = ctypes.c_int
        L.ttt_status_str.argtypes = [ctypes.c_int]
        L.ttt_status_str.restype = ctypes.c_char_p
        L.ttt_launch_count.argtypes = []
        L.ttt_launch_count.restype = ctypes.c_ulonglong
        L.ttt_debug_wait_limit.argtypes = [ctypes.c_ulonglong]
        L.ttt_debug_wait_limit.restype = None
        _lib = L
    return _lib


def status_str(rc: int) -> str:
    return lib().ttt_status_str(rc).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tokens(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B,H,T,d] tensor")
    if not (q.shape == k.shape == v.shape and q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share shape and dtype")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q, k, v must be bfloat16 or float32")
    return TTT_BF16 if q.dtype == torch.bfloat16 else TTT_F32


def _f32(t, name):
    if t is None:
        return None
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    return t


def _check_call(dev, stream, tensors, shapes):
    """Every tensor of a call lives on `dev` (the library launches on the current
    device, which the call makes `dev`), the stream belongs to it, and every given
    tensor has its expected shape.  Raises ValueError before anything is queued."""
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device} but q on {dev}: one device per call")
    for name, (t, shape) in shapes.items():
        if t is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if stream is not None and stream.device != dev:
        raise ValueError(f"the stream is on {stream.device} but the tensors on {dev}")


def _out_like_q(z, q):
    if z is not None and (z.dtype != q.dtype or not z.is_contiguous()):
        raise ValueError("z must be a contiguous tensor of q's dtype")


def _w0_stride(W0, B, H, d):
    if W0.shape == (H, d, d):
        return 0
    if W0.shape == (B, H, d, d):
        return H * d * d
    raise ValueError("W0 must be [H,d,d] or [B,H,d,d]")


def _linear_prologue(q, k, v, W0, eta, z, W_out, stream, ln_gamma=None, ln_beta=None):
    """Checks of every TTT-Linear wrapper; returns (io dtype, W0 batch stride)."""
    io = _check_tokens(q, k, v)
    B, H, T, d = q.shape
    for t, n in ((W0, "W0"), (eta, "eta"), (W_out, "W_out"), (ln_gamma, "ln_gamma"), (ln_beta, "ln_beta")):
        _f32(t, n)
    _check_call(q.device, stream,
                {"W0": W0, "eta": eta, "z": z, "W_out": W_out, "ln_gamma": ln_gamma, "ln_beta": ln_beta},
                {"eta": (eta, (B, H, T)), "z": (z, (B, H, T, d)), "W_out": (W_out, (B, H, d, d)),
                 "ln_gamma": (ln_gamma, (H, d)), "ln_beta": (ln_beta, (H, d))})
    _out_like_q(z, q)
    return io, _w0_stride(W0, B, H, d)


def ttt_linear_fwd(q, k, v, W0, mini_batch, causal=True, eta=None, eta_scalar=1.0,
                   z=None, W_out=None, want_W=True, stream=None, loss="mse", epochs=1,
                   ln_gamma=None, ln_beta=None, ln_eps=1e-6):
    """TTT-Linear forward.  q,k,v: [B,H,T,d] bf16 or fp32 CUDA tensors; W0: fp32
    [H,d,d] (shared over the batch) or [B,H,d,d]; eta: fp32 [B,H,T] or None;
    loss "mse" or "dot"; epochs > 1: repeated full-batch steps (causal=False,
    mini_batch >= T); ln_gamma, ln_beta: fp32 [H,d] for the inner model
    x + LN(x W).  Returns (z, W_final or None)."""
    io, w0s = _linear_prologue(q, k, v, W0, eta, z, W_out, stream, ln_gamma, ln_beta)
    B, H, T, d = q.shape
    with torch.cuda.device(q.device):
        if z is None:
            z = torch.empty_like(q)
        if W_out is None and want_W:
            W_out = torch.empty((B, H, d, d), device=q.device, dtype=torch.float32)
        desc = LinearDesc(B, H, T, d, int(mini_batch), 1 if causal else 0, io, w0s, LOSSES[loss],
                          int(epochs), _ptr(ln_gamma), _ptr(ln_beta), float(ln_eps))
        rc = lib().ttt_linear_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(eta),
                                  float(eta_scalar), _ptr(W0), _ptr(z), _ptr(W_out), _stream(stream))
    if rc != 0:
        raise TTTError("ttt_linear_fwd", rc)
    return z, W_out


def ttt_linear_seqpar_workspace(B, H, T, d, mini_batch, causal=True, dtype=torch.bfloat16,
                                loss="mse") -> int:
    """Workspace bytes ttt_linear_fwd_seqpar needs on the current device (0: the
    problem is not split)."""
    io = TTT_BF16 if dtype == torch.bfloat16 else TTT_F32
    desc = LinearDesc(B, H, T, d, int(mini_batch), 1 if causal else 0, io, 0, LOSSES[loss], 1)
    return int(lib().ttt_linear_seqpar_workspace(ctypes.byref(desc)))


def ttt_linear_fwd_seqpar(q, k, v, W0, mini_batch, causal=True, eta=None, eta_scalar=1.0,
                          z=None, W_out=None, want_W=True, workspace=None, stream=None, loss="mse"):
    """Sequence-parallel TTT-Linear forward (same arguments as ttt_linear_fwd).
    workspace: a CUDA uint8 tensor of at least ttt_linear_seqpar_workspace(...) bytes,
    allocated here when None.  Returns (z, W_final or None)."""
    io, w0s = _linear_prologue(q, k, v, W0, eta, z, W_out, stream)
    _check_call(q.device, None, {"workspace": workspace}, {})
    if workspace is not None and not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    B, H, T, d = q.shape
    with torch.cuda.device(q.device):
        if z is None:
            z = torch.empty_like(q)
        if W_out is None and want_W:
            W_out = torch.empty((B, H, d, d), device=q.device, dtype=torch.float32)
        desc = LinearDesc(B, H, T, d, int(mini_batch), 1 if causal else 0, io, w0s, LOSSES[loss], 1)
        need = int(lib().ttt_linear_seqpar_workspace(ctypes.byref(desc)))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        rc = lib().ttt_linear_fwd_seqpar(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(eta),
                                         float(eta_scalar), _ptr(W0), _ptr(z), _ptr(W_out),
                                         _ptr(workspace), nbytes, _stream(stream))
    if rc != 0:
        raise TTTError("ttt_linear_fwd_seqpar", rc)
    return z, W_out


def ttt_linear_fwd_seqpar_noalloc(q, k, v, W0, z, W_out, mini_batch, causal=True, eta=None,
                                  eta_scalar=1.0, stream=None, loss="mse"):
    """The sequence-parallel forward on the library's fixed scratch (no workspace,
    no allocation inside the call): z and W_out are the caller's output tensors."""
    if z is None:
        raise ValueError("z must be given (this entry point allocates nothing)")
    io, w0s = _linear_prologue(q, k, v, W0, eta, z, W_out, stream)
    B, H, T, d = q.shape
    with torch.cuda.device(q.device):
        desc = LinearDesc(B, H, T, d, int(mini_batch), 1 if causal else 0, io, w0s, LOSSES[loss], 1)
        rc = lib().ttt_linear_fwd_seqpar_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(eta),
                                                 float(eta_scalar), _ptr(W0), _ptr(z), _ptr(W_out),
                                                 _stream(stream))
    if rc != 0:
        raise TTTError("ttt_linear_fwd_seqpar_noalloc", rc)
    return z, W_out


def ttt_dwconv_fwd(q, k, v, W0, height, width, eta=None, eta_scalar=1.0, loss="mse", epochs=1,
                   z=None, W_out=None, want_W=True, stream=None):
    """Depthwise 3x3 convolution inner model, full-batch inner GD.  q,k,v: [B,H,N,d]
    with N = height*width tokens in row-major grid order; W0: fp32 taps [H,9,d] or
    [B,H,9,d].  Returns (z, W_final [B,H,9,d] or None)."""
    io = _check_tokens(q, k, v)
    B, H, N, d = q.shape
    if N != height * width:
        raise ValueError("q has N tokens, the grid height*width")
    for t, n in ((W0, "W0"), (eta, "eta"), (W_out, "W_out")):
        _f32(t, n)
    _check_call(q.device, stream, {"W0": W0, "eta": eta, "z": z, "W_out": W_out},
                {"eta": (eta, (B, H, N)), "z": (z, (B, H, N, d)), "W_out": (W_out, (B, H, 9, d))})
    _out_like_q(z, q)
    if W0.shape == (H, 9, d):
        w0s = 0
    elif W0.shape == (B, H, 9, d):
        w0s = H * 9 * d
    else:
        raise ValueError("W0 must be [H,9,d] or [B,H,9,d]")
    with torch.cuda.device(q.device):
        if z is None:
            z = torch.empty_like(q)
        if W_out is None and want_W:
            W_out = torch.empty((B, H, 9, d), device=q.device, dtype=torch.float32)
        desc = DwconvDesc(B, H, height, width, d, io, LOSSES[loss], int(epochs), w0s)
        rc = lib().ttt_dwconv_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(eta),
                                  float(eta_scalar), _ptr(W0), _ptr(z), _ptr(W_out), _stream(stream))
    if rc != 0:
        raise TTTError("ttt_dwconv_fwd", rc)
    return z, W_out


def ttt_mlp_fwd(q, k, v, W1, c1, W2, c2, mini_batch, causal=True, eta=None, eta_scalar=0.1,
                z=None, outs=None, want_W=True, stream=None, activation="silu", ln_gamma=None,
                ln_beta=None, ln_eps=1e-6):
    """TTT-MLP forward, f(x) = act(x W1 + c1) W2 + c2, activation "silu" or "gelu"; with
    ln_gamma, ln_beta (fp32 [H,d]): f(x) = x + LN(act(x W1 + c1) W2 + c2).
    Parameters fp32, per head ([H,...]) or per (batch, head) ([B,H,...]).  outs: the
    final-weight tensors (W1, c1, W2, c2), each [B,H,...] fp32 or None.  Returns
    (z, (W1,c1,W2,c2) final or None)."""
    io = _check_tokens(q, k, v)
    B, H, T, d = q.shape
    W1, c1, W2, c2 = (_f32(t, n) for t, n in ((W1, "W1"), (c1, "c1"), (W2, "W2"), (c2, "c2")))
    eta = _f32(eta, "eta")
    ln_gamma, ln_beta = _f32(ln_gamma, "ln_gamma"), _f32(ln_beta, "ln_beta")
    m = W1.shape[-1]
    per_batch = 1 if W1.dim() == 4 else 0
    lead = (B, H) if per_batch else (H,)
    if (W1.shape != lead + (d, m) or c1.shape != lead + (m,) or W2.shape != lead + (m, d)
            or c2.shape != lead + (d,)):
        raise ValueError("inner weights must be W1 [..,d,m], c1 [..,m], W2 [..,m,d], c2 [..,d]")
    if outs is not None:
        if len(outs) != 4:
            raise ValueError("outs must be (W1, c1, W2, c2) final-weight tensors")
        for t, n in zip(outs, ("W1_out", "c1_out", "W2_out", "c2_out")):
            _f32(t, n)
    o = outs if outs is not None else (None, None, None, None)
    shapes = {"eta": (eta, (B, H, T)), "z": (z, (B, H, T, d)), "ln_gamma": (ln_gamma, (H, d)),
              "ln_beta": (ln_beta, (H, d))}
    for t, n, sh in zip(o, ("W1_out", "c1_out", "W2_out", "c2_out"), ((d, m), (m,), (m, d), (d,))):
        shapes[n] = (t, (B, H) + sh)
    _check_call(q.device, stream, {"W1": W1, "c1": c1, "W2": W2, "c2": c2, "eta": eta, "z": z,
                                   "ln_gamma": ln_gamma, "ln_beta": ln_beta,
                                   **dict(zip(("W1_out", "c1_out", "W2_out", "c2_out"), o))}, shapes)
    _out_like_q(z, q)
    with torch.cuda.device(q.device):
        if z is None:
            z = torch.empty_like(q)
        if outs is None and want_W:
            dev = q.device
            outs = (torch.empty((B, H, d, m), device=dev), torch.empty((B, H, m), device=dev),
                    torch.empty((B, H, m, d), device=dev), torch.empty((B, H, d), device=dev))
        o = outs if outs is not None else (None, None, None, None)
        desc = MlpDesc(B, H, T, d, m, int(mini_batch), 1 if causal else 0, io, per_batch,
                       ACTIVATIONS[activation], None if ln_gamma is None else ln_gamma.data_ptr(),
                       None if ln_beta is None else ln_beta.data_ptr(), float(ln_eps))
        rc = lib().ttt_mlp_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(eta),
                               float(eta_scalar), _ptr(W1), _ptr(c1), _ptr(W2), _ptr(c2), _ptr(z),
                               *(_ptr(t) for t in o), _stream(stream))
    if rc != 0:
        raise TTTError("ttt_mlp_fwd", rc)
    return z, outs


def ttt_eta_gate(x, theta, eta_base=1.0, eta=None, stream=None):
    """Input-dependent inner learning rate eta[b,h,t] = eta_base * sigmoid(theta[h] .
    x[b,t]).  x: bf16 [B,T,dm] (the layer's input tokens); theta: bf16 [H,dm] (one
    vector per head).  Returns eta, fp32 [B,H,T] (the layout the TTT entry points
    read)."""
    for name, t in (("x", x), ("theta", theta)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor (no CPU path)")
    if x.dim() != 3 or theta.dim() != 2 or theta.shape[1] != x.shape[2]:
        raise ValueError("x must be [B,T,dm] and theta [H,dm]")
    B, T, dm = x.shape
    H = theta.shape[0]
    eta = _f32(eta, "eta")
    _check_call(x.device, stream, {"theta": theta, "eta": eta}, {"eta": (eta, (B, H, T))})
    with torch.cuda.device(x.device):
        if eta is None:
            eta = torch.empty((B, H, T), device=x.device, dtype=torch.float32)
        desc = GateDesc(B, T, H, dm)
        rc = lib().ttt_eta_gate(ctypes.byref(desc), _ptr(x), _ptr(theta), float(eta_base), _ptr(eta),
                                _stream(stream))
    if rc != 0:
        raise TTTError("ttt_eta_gate", rc)
    return eta


def ttt_sync_status(stream=None):
    """Waits for the stream; raises TTTError if a kernel wait timed out."""
    rc = lib().ttt_sync_status(_stream(stream))
    if rc != 0:
        raise TTTError("ttt_sync_status", rc)


def ttt_launch_count() -> int:
    return int(lib().ttt_launch_count())


def ttt_debug_wait_limit(ns: int) -> None:
    """Test hook of the timeout path: ns > 0 makes the first consumer wait of the
    b = 16 and full-batch TTT-Linear kernels run out after ns nanoseconds (see
    include/ttt.h); 0 restores normal operation."""
    lib().ttt_debug_wait_limit(int(ns))
