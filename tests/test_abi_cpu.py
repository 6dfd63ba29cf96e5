"""The C-ABI library without a GPU: it loads, exports every function include/ttt.h
declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

from test_sequence_layers_gb300 import abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return abi.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "ttt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ttt_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(abi.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings(L):
    for rc in (0, -1, -2, -3, -4, -5):
        assert abi.status_str(rc)
    assert abi.status_str(7) == "unknown status"


FAKE = 1 << 20  # an aligned address that is never dereferenced (validation fails first)


def _lin(**kw):
    d = dict(B=1, H=1, T=32, d=64, mini_batch=16, causal=1, io_dtype=abi.TTT_BF16,
             w0_batch_stride=0, loss=0, epochs=1)
    d.update(kw)
    return abi.LinearDesc(**d)


def _call_lin(L, desc, q=FAKE, k=FAKE, v=FAKE, eta=None, W0=FAKE, z=FAKE, Wout=None):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.ttt_linear_fwd(ctypes.byref(desc) if desc is not None else None, vp(q), vp(k), vp(v),
                            vp(eta), 1.0, vp(W0), vp(z), vp(Wout), None)


def test_linear_rejects_bad_arguments(L):
    assert L.ttt_linear_fwd(None, None, None, None, None, 1.0, None, None, None, None) == -1
    assert _call_lin(L, _lin(B=0)) == -1
    assert _call_lin(L, _lin(T=-1)) == -1
    assert _call_lin(L, _lin(mini_batch=0)) == -1
    assert _call_lin(L, _lin(causal=2)) == -1
    assert _call_lin(L, _lin(io_dtype=5)) == -1
    assert _call_lin(L, _lin(), q=None) == -1
    assert _call_lin(L, _lin(), W0=None) == -1
    assert _call_lin(L, _lin(w0_batch_stride=7)) == -1
    assert _call_lin(L, _lin(d=48)) == -2
    assert _call_lin(L, _lin(loss=2)) == -1
    assert _call_lin(L, _lin(epochs=-1)) == -1
    assert _call_lin(L, _lin(epochs=2)) == -2                     # causal
    assert _call_lin(L, _lin(epochs=2, causal=0, mini_batch=16)) == -2  # b < T
    g = ctypes.c_void_p(FAKE)
    assert _call_lin(L, _lin(ln_gamma=g)) == -1                          # scale without shift
    assert _call_lin(L, _lin(ln_gamma=g, ln_beta=g, ln_eps=0.0)) == -1
    assert _call_lin(L, _lin(ln_gamma=g, ln_beta=g, ln_eps=1e-6, loss=1)) == -1
    assert _call_lin(L, _lin(ln_gamma=g, ln_beta=g, ln_eps=1e-6, causal=0, mini_batch=32,
                             epochs=2)) == -2
    assert _call_lin(L, _lin(d=256)) == -2
    assert _call_lin(L, _lin(), q=FAKE + 8) == -3
    assert _call_lin(L, _lin(), z=FAKE + 2) == -3
    assert _call_lin(L, _lin(), eta=FAKE + 2) == -3
    # final weights may not overlap weights shared over the batch
    assert _call_lin(L, _lin(B=2), W0=FAKE, Wout=FAKE + 64) == -1


def _mlp(**kw):
    d = dict(B=1, H=1, T=32, d=64, m=256, mini_batch=16, causal=1, io_dtype=abi.TTT_BF16,
             params_per_batch=0, activation=0)
    d.update(kw)
    return abi.MlpDesc(**d)


def _call_mlp(L, desc, q=FAKE, W1=FAKE, c1=FAKE, W2=FAKE, c2=FAKE, W1o=None):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return L.ttt_mlp_fwd(ctypes.byref(desc), vp(q), vp(q), vp(q), None, 0.1, vp(W1), vp(c1),
                         vp(W2), vp(c2), vp(FAKE), vp(W1o), None, None, None, None)


def test_mlp_rejects_bad_arguments(L):
    assert _call_mlp(L, _mlp(m=0)) == -1
    assert _call_mlp(L, _mlp(), c1=None) == -1
    assert _call_mlp(L, _mlp(params_per_batch=3)) == -1
    assert _call_mlp(L, _mlp(activation=2)) == -1
    assert _call_mlp(L, _mlp(d=128)) == -2
    assert _call_mlp(L, _mlp(m=40)) == -2
    assert _call_mlp(L, _mlp(), q=FAKE + 4) == -3
    assert _call_mlp(L, _mlp(), W2=FAKE + 1) == -3
    assert _call_mlp(L, _mlp(B=2), W1=FAKE, W1o=FAKE) == -1
    g = FAKE + (1 << 24)
    assert _call_mlp(L, _mlp(ln_gamma=g, ln_eps=1e-6)) == -1               # beta missing
    assert _call_mlp(L, _mlp(io_dtype=abi.TTT_F32, ln_gamma=g, ln_beta=g, ln_eps=0.0)) == -1
    assert _call_mlp(L, _mlp(d=32, ln_gamma=g, ln_beta=g, ln_eps=1e-6)) == -2  # bf16 inner norm: d = 64 only
    # bf16 inner norm: mini-batches of <= 16 tokens or one non-causal full batch
    assert _call_mlp(L, _mlp(mini_batch=32, ln_gamma=g, ln_beta=g, ln_eps=1e-6)) == -2
    assert _call_mlp(L, _mlp(T=64, mini_batch=32, causal=0, ln_gamma=g, ln_beta=g, ln_eps=1e-6)) == -2
    assert _call_mlp(L, _mlp(T=64, mini_batch=64, causal=1, ln_gamma=g, ln_beta=g, ln_eps=1e-6)) == -2
    assert _call_mlp(L, _mlp(io_dtype=abi.TTT_F32, ln_gamma=g + 2, ln_beta=g, ln_eps=1e-6)) == -3


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 4, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        abi.ttt_linear_fwd(q, q, q, torch.zeros(1, 16, 16), 4)


def test_seqpar_rejects_bad_arguments_and_reports_no_workspace_without_gpu(L):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    assert L.ttt_linear_fwd_seqpar(None, None, None, None, None, 1.0, None, None, None, None, 0,
                                   None) == -1
    for bad in (_lin(B=0), _lin(T=-1), _lin(mini_batch=0), _lin(causal=2)):
        assert L.ttt_linear_fwd_seqpar(ctypes.byref(bad), vp(FAKE), vp(FAKE), vp(FAKE), None, 1.0,
                                       vp(FAKE), vp(FAKE), None, None, 0, None) == -1
    assert L.ttt_linear_fwd_seqpar(ctypes.byref(_lin(d=48)), vp(FAKE), vp(FAKE), vp(FAKE), None,
                                   1.0, vp(FAKE), vp(FAKE), None, None, 0, None) == -2
    assert L.ttt_linear_seqpar_workspace(None) == 0
    # no device visible: the call would not split, so no workspace is needed
    assert L.ttt_linear_seqpar_workspace(ctypes.byref(_lin(T=4096))) == 0


def test_dwconv_rejects_bad_arguments(L):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)

    def call(**kw):
        d = dict(B=1, H=1, height=14, width=14, d=64, io_dtype=abi.TTT_BF16, loss=0, epochs=1,
                 w0_batch_stride=0)
        d.update(kw)
        desc = abi.DwconvDesc(**d)
        return L.ttt_dwconv_fwd(ctypes.byref(desc), vp(FAKE), vp(FAKE), vp(FAKE), None, 1.0,
                                vp(FAKE), vp(FAKE), None, None)

    assert L.ttt_dwconv_fwd(None, None, None, None, None, 1.0, None, None, None, None) == -1
    assert call(B=0) == -1
    assert call(epochs=0) == -1
    assert call(loss=3) == -1
    assert call(io_dtype=7) == -1
    assert call(w0_batch_stride=5) == -1
    assert call(d=12) == -2                      # channels must be a multiple of 8
    assert call(height=64, width=64) == -2       # the sequence does not fit on chip


def test_eta_gate_rejects_bad_arguments(L):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)

    def call(x=FAKE, theta=FAKE, eta=FAKE + (1 << 26), **kw):
        d = dict(B=2, T=100, H=32, dm=2048)
        d.update(kw)
        desc = abi.GateDesc(**d)
        return L.ttt_eta_gate(ctypes.byref(desc), vp(x), vp(theta), 1.0, vp(eta), None)

    assert L.ttt_eta_gate(None, None, None, 1.0, None, None) == -1
    assert call(B=-1) == -1
    assert call(H=0) == -1
    assert call(dm=0) == -1
    assert call(B=0) == 0 and call(T=0, x=None) == 0   # nothing to queue
    assert call(x=None) == -1
    assert call(H=65) == -2                             # heads past 64
    assert call(dm=100) == -2                           # width not a multiple of 8
    assert call(x=FAKE + 8) == -3
    assert call(theta=FAKE + 2) == -3
    assert call(eta=FAKE + (1 << 26) + 2) == -3
    assert call(eta=FAKE + 64) == -1                    # eta overlaps x


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library the binding raises; there is no CPU fallback."""
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from test_sequence_layers_gb300 import abi\n"
            "abi.LIB_PATH = %r\n"
            "try:\n    abi.lib()\nexcept RuntimeError as e:\n    print('raised', e)\n" % (ROOT, str(tmp_path / "libttt.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("raised"), (r.stdout, r.stderr)


class _Dev:
    """Stand-in for a CUDA tensor (this machine has none): the attributes the binding
    reads before it touches the library or the device."""

    def __init__(self, shape, dtype=None, index=0, cuda=True):
        import torch
        self.shape = torch.Size(shape)
        self.dtype = torch.float32 if dtype is None else dtype
        self.device = torch.device("cuda", index) if cuda else torch.device("cpu")
        self.is_cuda = cuda

    def dim(self):
        return len(self.shape)

    def is_contiguous(self):
        return True

    def data_ptr(self):
        raise AssertionError("the binding reached the library with a bad argument")


def _lin_args(B=2, H=3, T=40, d=64, **over):
    import torch
    bf = torch.bfloat16
    a = dict(q=_Dev((B, H, T, d), bf), k=_Dev((B, H, T, d), bf), v=_Dev((B, H, T, d), bf),
             W0=_Dev((H, d, d)), eta=_Dev((B, H, T)), z=_Dev((B, H, T, d), bf), W_out=_Dev((B, H, d, d)))
    a.update(over)
    return a


@pytest.mark.parametrize("bad", [
    dict(z=_Dev((2, 3, 40, 64), None, cuda=False)),            # CPU output
    dict(z=_Dev((2, 3, 39, 64))),                              # wrong shape (and dtype)
    dict(W_out=_Dev((2, 3, 64, 32))),                          # undersized final weights
    dict(W_out=_Dev((3, 64, 64))),                             # final weights must be [B,H,d,d]
    dict(eta=_Dev((2, 3, 39))),                                # undersized per-token rates
    dict(eta=_Dev((3, 40))),
    dict(W0=_Dev((3, 64, 64), index=1)),                       # another device
    dict(z=_Dev((2, 3, 40, 64), None, index=1)),
    dict(eta=_Dev((2, 3, 40), index=1)),
    dict(k=_Dev((2, 3, 40, 64), None, index=1)),
])
def test_linear_wrappers_reject_bad_tensors_before_any_launch(bad):
    a = _lin_args(**bad)
    for fn in (abi.ttt_linear_fwd, abi.ttt_linear_fwd_seqpar):
        with pytest.raises(ValueError):
            fn(a["q"], a["k"], a["v"], a["W0"], 16, eta=a["eta"], z=a["z"], W_out=a["W_out"])
    with pytest.raises(ValueError):
        abi.ttt_linear_fwd_seqpar_noalloc(a["q"], a["k"], a["v"], a["W0"], a["z"], a["W_out"], 16,
                                          eta=a["eta"])


def test_linear_wrapper_rejects_inner_norm_of_wrong_shape():
    a = _lin_args()
    with pytest.raises(ValueError):
        abi.ttt_linear_fwd(a["q"], a["k"], a["v"], a["W0"], 16, z=a["z"], W_out=a["W_out"],
                           ln_gamma=_Dev((3, 32)), ln_beta=_Dev((3, 64)))


def _mlp_args(B=2, H=3, T=40, d=64, m=256):
    import torch
    bf = torch.bfloat16
    return dict(q=_Dev((B, H, T, d), bf), W1=_Dev((H, d, m)), c1=_Dev((H, m)), W2=_Dev((H, m, d)),
                c2=_Dev((H, d)), z=_Dev((B, H, T, d), bf),
                outs=(_Dev((B, H, d, m)), _Dev((B, H, m)), _Dev((B, H, m, d)), _Dev((B, H, d))))


@pytest.mark.parametrize("which", ["W1_out_shape", "c2_out_shape", "W2_device", "z_shape", "eta_shape",
                                   "outs_cpu"])
def test_mlp_wrapper_rejects_bad_tensors_before_any_launch(which):
    a = _mlp_args()
    outs, eta, z, W2 = list(a["outs"]), None, a["z"], a["W2"]
    if which == "W1_out_shape":
        outs[0] = _Dev((2, 3, 64, 128))
    elif which == "c2_out_shape":
        outs[3] = _Dev((3, 64))
    elif which == "W2_device":
        W2 = _Dev((3, 256, 64), index=1)
    elif which == "z_shape":
        z = _Dev((2, 3, 40, 32))
    elif which == "eta_shape":
        eta = _Dev((2, 3, 41))
    elif which == "outs_cpu":
        outs[1] = _Dev((2, 3, 256), cuda=False)
    q = a["q"]
    with pytest.raises(ValueError):
        abi.ttt_mlp_fwd(q, q, q, a["W1"], a["c1"], W2, a["c2"], 16, eta=eta, z=z, outs=tuple(outs))


def test_gate_and_dwconv_wrappers_reject_bad_tensors():
    import torch
    x, th = _Dev((2, 50, 256), torch.bfloat16), _Dev((4, 256), torch.bfloat16)
    with pytest.raises(ValueError):
        abi.ttt_eta_gate(x, th, eta=_Dev((2, 4, 49)))
    with pytest.raises(ValueError):
        abi.ttt_eta_gate(x, _Dev((4, 256), torch.bfloat16, index=1))
    q = _Dev((1, 2, 196, 64), torch.bfloat16)
    with pytest.raises(ValueError):
        abi.ttt_dwconv_fwd(q, q, q, _Dev((2, 9, 64)), 14, 14, z=q, W_out=_Dev((1, 2, 9, 32)))
    with pytest.raises(ValueError):
        abi.ttt_dwconv_fwd(q, q, q, _Dev((2, 9, 64), index=2), 14, 14, z=q, W_out=_Dev((1, 2, 9, 64)))


def test_stream_on_another_device_is_rejected():
    import torch

    class _S:
        device = torch.device("cuda", 1)
    a = _lin_args()
    with pytest.raises(ValueError):
        abi.ttt_linear_fwd(a["q"], a["k"], a["v"], a["W0"], 16, eta=a["eta"], z=a["z"], W_out=a["W_out"],
                           stream=_S())
