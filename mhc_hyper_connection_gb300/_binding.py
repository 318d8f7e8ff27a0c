"""ctypes binding of include/mhc_pre.h -- argument marshalling only.

Every function of the C ABI is exposed under its own name.  ``MhcPre`` wraps
a handle and turns torch tensors into the pointer struct; all computation
happens in the CUDA library.  If the library has not been built this module
raises on first use: there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

MHC_OK = 0
MHC_ERR_NULLPTR = 161001
MHC_ERR_PARAM_INVALID = 161002
MHC_ERR_RUNTIME = 361001
MHC_IMPL_FP32 = 0
MHC_IMPL_TF32 = 1
MHC_DTYPE_BF16 = 0
MHC_DTYPE_FP16 = 1
MHC_KERNEL_AUTO = 0
MHC_KERNEL_CLUSTER = 1
MHC_KERNEL_GRID = 2
MHC_KERNEL_RESIDENT = 3

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmhc_pre.so")


class MhcPreConfig(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("D", ctypes.c_int64), ("alpha_len", ctypes.c_int32),
                ("num_iters", ctypes.c_int32), ("norm_eps", ctypes.c_double),
                ("hc_eps", ctypes.c_double), ("impl_mode", ctypes.c_int32),
                ("need_backward", ctypes.c_int32), ("batch_consistent", ctypes.c_int32),
                ("x_dtype", ctypes.c_int32), ("kernel", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("x_stages", ctypes.c_int32), ("w_stages", ctypes.c_int32), ("gw_groups", ctypes.c_int32),
                ("gw_x_stages", ctypes.c_int32), ("gw_x_lead", ctypes.c_int32), ("tm_buffers", ctypes.c_int32)]

# Launch-choice fields of MhcPreConfig (0 = automatic); MhcPre takes them as
# keyword arguments.
LAUNCH_FIELDS = ("kernel", "cluster", "x_stages", "w_stages", "gw_groups", "gw_x_stages", "gw_x_lead", "tm_buffers")


_P = ctypes.c_void_p


class MhcPreArgs(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("x", _P), ("phi", _P), ("alpha", _P), ("bias", _P),
                ("gamma", _P), ("pre_mix", _P), ("y", _P), ("h_post", _P), ("h_res", _P),
                ("h_pre", _P), ("inv_rms", _P), ("h_mix", _P), ("sum_out", _P),
                ("norm_out", _P), ("workspace", _P), ("workspace_bytes", ctypes.c_size_t), ("weights", _P)]


class MhcPreBwdArgs(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("x", _P), ("phi", _P), ("alpha", _P), ("gamma", _P),
                ("grad_h_in", _P), ("grad_h_post", _P), ("grad_h_res", _P), ("inv_rms", _P),
                ("h_mix", _P), ("h_pre", _P), ("h_post", _P), ("sum_out", _P), ("norm_out", _P),
                ("grad_x_post", _P), ("grad_x", _P), ("grad_phi", _P), ("grad_alpha", _P),
                ("grad_bias", _P), ("grad_gamma", _P), ("workspace", _P),
                ("workspace_bytes", ctypes.c_size_t)]


class MhcError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})"
                         + (f": {detail}" if detail else ""))


_lib = None
_lock = threading.Lock()


def library() -> ctypes.CDLL:
    """Load libmhc_pre.so (built in-tree).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m mhc_hyper_connection_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            lib.mhc_pre_config_default.argtypes = [ctypes.POINTER(MhcPreConfig)]
            lib.mhc_pre_config_default.restype = None
            lib.mhc_pre_create.argtypes = [ctypes.POINTER(_P), ctypes.POINTER(MhcPreConfig)]
            lib.mhc_pre_create.restype = ctypes.c_int32
            lib.mhc_pre_workspace_size.argtypes = [_P, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)]
            lib.mhc_pre_workspace_size.restype = ctypes.c_int32
            lib.mhc_pre_run.argtypes = [_P, ctypes.POINTER(MhcPreArgs), _P]
            lib.mhc_pre_run.restype = ctypes.c_int32
            lib.mhc_pre_run_noalloc.argtypes = [_P, ctypes.POINTER(MhcPreArgs), _P]
            lib.mhc_pre_run_noalloc.restype = ctypes.c_int32
            lib.mhc_pre_status.argtypes = [_P, _P, _P]
            lib.mhc_pre_status.restype = ctypes.c_int32
            lib.mhc_pre_weights_size.argtypes = [_P, ctypes.POINTER(ctypes.c_size_t)]
            lib.mhc_pre_weights_size.restype = ctypes.c_int32
            lib.mhc_pre_prepare_weights.argtypes = [_P, _P, _P, _P, ctypes.c_size_t, _P]
            lib.mhc_pre_prepare_weights.restype = ctypes.c_int32
            lib.mhc_pre_set_wait_test.argtypes = [_P, ctypes.c_uint32, ctypes.c_int32]
            lib.mhc_pre_set_wait_test.restype = ctypes.c_int32
            lib.mhc_pre_set_profile_events.argtypes = [_P, _P, _P]
            lib.mhc_pre_set_profile_events.restype = ctypes.c_int32
            I32P = ctypes.POINTER(ctypes.c_int32)
            lib.mhc_pre_last_launch.argtypes = [_P, I32P, I32P, I32P, I32P]
            lib.mhc_pre_last_launch.restype = ctypes.c_int32
            lib.mhc_post_run.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P, _P, _P]
            lib.mhc_post_run.restype = ctypes.c_int32
            lib.mhc_pre_backward_workspace_size.argtypes = [_P, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)]
            lib.mhc_pre_backward_workspace_size.restype = ctypes.c_int32
            lib.mhc_pre_backward_run.argtypes = [_P, ctypes.POINTER(MhcPreBwdArgs), _P]
            lib.mhc_pre_backward_run.restype = ctypes.c_int32
            lib.mhc_pre_inv_rms_run.argtypes = [_P, ctypes.c_int64, _P, _P, _P]
            lib.mhc_pre_inv_rms_run.restype = ctypes.c_int32
            lib.mhc_pre_mixes_run.argtypes = [_P, ctypes.c_int64, _P, _P, _P, _P, _P]
            lib.mhc_pre_mixes_run.restype = ctypes.c_int32
            lib.mhc_pre_sinkhorn_run.argtypes = [_P, ctypes.POINTER(MhcPreArgs), _P, _P, _P]
            lib.mhc_pre_sinkhorn_run.restype = ctypes.c_int32
            lib.mhc_pre_last_kernel.argtypes = [_P]
            lib.mhc_pre_last_kernel.restype = ctypes.c_char_p
            lib.mhc_pre_destroy.argtypes = [_P]
            lib.mhc_pre_destroy.restype = None
            lib.mhc_pre_status_string.argtypes = [ctypes.c_int32]
            lib.mhc_pre_status_string.restype = ctypes.c_char_p
            lib.mhc_pre_last_error.argtypes = []
            lib.mhc_pre_last_error.restype = ctypes.c_char_p
            _lib = lib
    return _lib


# ----------------------------------------------------------- raw C entry points

def mhc_pre_config_default() -> MhcPreConfig:
    c = MhcPreConfig()
    library().mhc_pre_config_default(ctypes.byref(c))
    return c


def mhc_pre_create(cfg: MhcPreConfig):
    """Returns (status, handle-or-None)."""
    h = _P()
    st = library().mhc_pre_create(ctypes.byref(h), ctypes.byref(cfg))
    return st, (h if st == MHC_OK else None)


def mhc_pre_workspace_size(handle, T: int):
    n = ctypes.c_size_t(0)
    st = library().mhc_pre_workspace_size(handle, int(T), ctypes.byref(n))
    return st, n.value


def mhc_pre_run(handle, args: MhcPreArgs, stream: int = 0) -> int:
    return library().mhc_pre_run(handle, ctypes.byref(args), _P(stream or None))


def mhc_pre_run_noalloc(handle, args: MhcPreArgs, stream: int = 0) -> int:
    """The forward on the library's fixed scratch array (no workspace)."""
    return library().mhc_pre_run_noalloc(handle, ctypes.byref(args), _P(stream or None))


def mhc_pre_status(handle, workspace: int = 0, stream: int = 0) -> int:
    return library().mhc_pre_status(handle, _P(workspace or None), _P(stream or None))


def mhc_pre_weights_size(handle):
    """Returns (status, bytes of the prepared-weights form)."""
    n = ctypes.c_size_t(0)
    st = library().mhc_pre_weights_size(handle, ctypes.byref(n))
    return st, n.value


def mhc_pre_prepare_weights(handle, phi: int, gamma: int, weights: int, weights_bytes: int, stream: int = 0) -> int:
    return library().mhc_pre_prepare_weights(handle, phi, gamma, weights, weights_bytes, stream)


def mhc_pre_set_wait_test(handle, wait_limit_us: int = 0, withhold_last_x_copy: int = 0) -> int:
    return library().mhc_pre_set_wait_test(handle, int(wait_limit_us), int(withhold_last_x_copy))


def mhc_pre_set_profile_events(handle, before: int = 0, after: int = 0) -> int:
    return library().mhc_pre_set_profile_events(handle, _P(before or None), _P(after or None))


def mhc_pre_last_launch(handle):
    """(status, {cluster, grid, stages, ystages}) of the last run on this handle."""
    v = [ctypes.c_int32(0) for _ in range(4)]
    st = library().mhc_pre_last_launch(handle, *[ctypes.byref(x) for x in v])
    return st, dict(zip(("cluster", "grid", "stages", "ystages"), (x.value for x in v)))


def mhc_pre_last_kernel(handle) -> str:
    """Name of the fused kernel the last run on this handle launched."""
    return library().mhc_pre_last_kernel(handle).decode()


def mhc_post_run(T: int, n: int, D: int, x: int, residual: int, post: int, comb: int, out: int,
                 stream: int = 0) -> int:
    """The post-mapping (include/mhc_post.h) on raw device pointers."""
    return library().mhc_post_run(int(T), int(n), int(D), _P(x or None), _P(residual or None), _P(post or None),
                                  _P(comb or None), _P(out or None), _P(stream or None))


def hc_post(x, residual, post, comb, out=None, stream=None):
    """out[t, j, d] = post[t, j] x[t, d] + sum_i comb[t, i, j] residual[t, i, d]
    on torch tensors (x bf16 [T, D], residual bf16 [T, n, D], post fp32 [T, n],
    comb fp32 [T, n, n]; or the BSND layout with leading dims (B, S) in place
    of T); returns out (bf16, shaped like residual).  Raises MhcError on a
    host-side rejection."""
    import torch
    n, D = residual.shape[-2:]
    T = _tokens(residual.shape[:-2])
    if out is None:
        out = torch.empty(residual.shape, dtype=torch.bfloat16, device=residual.device)
    if stream is None:
        stream = torch.cuda.current_stream(residual.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    st = mhc_post_run(T, n, D, _ptr(x), _ptr(residual), _ptr(post), _ptr(comb), _ptr(out), int(stream))
    if st != MHC_OK:
        raise MhcError(st, "mhc_post_run", last_error())
    return out


def mhc_pre_backward_workspace_size(handle, T: int):
    n = ctypes.c_size_t(0)
    st = library().mhc_pre_backward_workspace_size(handle, int(T), ctypes.byref(n))
    return st, n.value


def mhc_pre_backward_run(handle, args: MhcPreBwdArgs, stream: int = 0) -> int:
    return library().mhc_pre_backward_run(handle, ctypes.byref(args), _P(stream or None))


def mhc_pre_inv_rms_run(handle, T: int, x: int, inv_rms: int, stream: int = 0) -> int:
    return library().mhc_pre_inv_rms_run(handle, int(T), _P(x or None), _P(inv_rms or None), _P(stream or None))


def mhc_pre_mixes_run(handle, T: int, x: int, phi: int, gamma: int, mixes: int, stream: int = 0) -> int:
    return library().mhc_pre_mixes_run(handle, int(T), _P(x or None), _P(phi or None), _P(gamma or None),
                                       _P(mixes or None), _P(stream or None))


def mhc_pre_sinkhorn_run(handle, args: MhcPreArgs, mixes: int, inv_rms: int, stream: int = 0) -> int:
    return library().mhc_pre_sinkhorn_run(handle, ctypes.byref(args), _P(mixes or None), _P(inv_rms or None),
                                          _P(stream or None))


def mhc_pre_destroy(handle) -> None:
    library().mhc_pre_destroy(handle)


def status_string(status: int) -> str:
    return library().mhc_pre_status_string(int(status)).decode()


def last_error() -> str:
    return library().mhc_pre_last_error().decode()


# ------------------------------------------------------------- torch marshalling

def _ptr(t) -> Optional[int]:
    """Device address of a tensor; the library takes contiguous tensors only
    (the pages do not support non-contiguous inputs), so anything else is
    refused here rather than misread."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the mHC library must be contiguous")
    return int(t.data_ptr())


def _tokens(lead) -> int:
    """Token count of the leading dims: (T,) in TND layout or (B, S) in BSND."""
    lead = tuple(int(v) for v in lead)
    if len(lead) not in (1, 2):
        raise ValueError("leading dims must be (T,) or (B, S)")
    return lead[0] * (lead[1] if len(lead) == 2 else 1)


class MhcPre:
    """One configured forward (n, D, alpha_len, num_iters, eps, mode, backward).

    Launch-choice keywords (kernel, cluster, x_stages, w_stages, gw_groups,
    gw_x_stages, gw_x_lead; 0 = automatic) go to the matching
    mhc_pre_config fields."""

    def __init__(self, n: int, D: int, *, alpha_len: int = 3, num_iters: int = 20,
                 norm_eps: float = 1e-6, hc_eps: float = 1e-6, impl_mode: int = MHC_IMPL_FP32,
                 need_backward: bool = False, batch_consistent: bool = False,
                 x_dtype: int = MHC_DTYPE_BF16, **launch):
        cfg = mhc_pre_config_default()
        cfg.n, cfg.D, cfg.alpha_len, cfg.num_iters = n, D, alpha_len, num_iters
        cfg.norm_eps, cfg.hc_eps = norm_eps, hc_eps
        cfg.impl_mode, cfg.need_backward = impl_mode, int(bool(need_backward))
        cfg.batch_consistent, cfg.x_dtype = int(bool(batch_consistent)), int(x_dtype)
        for k, v in launch.items():
            if k not in LAUNCH_FIELDS:
                raise TypeError(f"MhcPre() got an unexpected keyword argument {k!r}")
            setattr(cfg, k, int(v))
        st, h = mhc_pre_create(cfg)
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_create", last_error())
        self.handle = h
        self.n, self.D, self.alpha_len, self.num_iters = n, D, alpha_len, num_iters
        self.need_backward = bool(need_backward)
        self.x_dtype = int(x_dtype)
        self.R = n * n + 2 * n if alpha_len == 3 else 2 * n

    def close(self):
        if self.handle is not None:
            mhc_pre_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_size(self, T: int) -> int:
        st, n = mhc_pre_workspace_size(self.handle, T)
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_workspace_size", last_error())
        return n

    def allocate(self, T, device, *, h_res: bool = True, h_pre: bool = True):
        """Output and workspace tensors (torch supplies the memory) for T
        tokens, or for a (B, S) batch in the BSND layout: outputs then carry
        the leading dims (B, S) (hIn [B, S, D], hPost [B, S, n], ...), the
        same memory as T = B * S tokens."""
        import torch
        lead = (T,) if isinstance(T, int) else tuple(T)
        T = _tokens(lead)
        n, D, R, I = self.n, self.D, self.R, self.num_iters
        f32 = dict(dtype=torch.float32, device=device)
        ydt = torch.float16 if self.x_dtype == MHC_DTYPE_FP16 else torch.bfloat16
        out = {"y": torch.empty(lead + (D,), dtype=ydt, device=device),
               "h_post": torch.empty(lead + (n,), **f32),
               "h_res": torch.empty(lead + (n, n), **f32) if (h_res or self.alpha_len == 3) else None,
               "h_pre": torch.empty(lead + (n,), **f32) if (h_pre or self.need_backward) else None,
               "inv_rms": None, "h_mix": None, "sum_out": None, "norm_out": None}
        if self.need_backward:
            out["inv_rms"] = torch.empty(lead, **f32)
            out["h_mix"] = torch.empty(lead + (R,), **f32)
            if self.alpha_len == 3:
                out["sum_out"] = torch.empty((2 * I,) + lead + (n,), **f32)
                out["norm_out"] = torch.empty((2 * I,) + lead + (n, n), **f32)
        ws = self.workspace_size(T)
        # At least the 256-byte header, zeroed, so a status read is defined even for T = 0.
        out["workspace"] = torch.zeros((max(ws, 256),), dtype=torch.uint8, device=device)
        return out

    def prepare_weights(self, phi, gamma=None, stream=None):
        """phi (.) gamma in the form a run takes as `weights` (a uint8 tensor on
        phi's device), for repeated calls with the same weights."""
        import torch
        st, nbytes = mhc_pre_weights_size(self.handle)
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_weights_size", last_error())
        w = torch.empty((nbytes,), dtype=torch.uint8, device=phi.device)
        if stream is None:
            stream = torch.cuda.current_stream(phi.device).cuda_stream
        elif hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        st = mhc_pre_prepare_weights(self.handle, _ptr(phi), _ptr(gamma), _ptr(w), nbytes, int(stream))
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_prepare_weights", last_error())
        return w

    def make_args(self, x, phi, alpha, bias, out, gamma=None, pre_mix=None, weights=None) -> MhcPreArgs:
        a = MhcPreArgs()
        a.T = _tokens(x.shape[:-2]) if x is not None else 0
        a.x, a.phi, a.alpha, a.bias = _ptr(x), _ptr(phi), _ptr(alpha), _ptr(bias)
        a.gamma, a.pre_mix = _ptr(gamma), _ptr(pre_mix)
        for k in ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix", "sum_out", "norm_out"):
            setattr(a, k, _ptr(out.get(k)))
        ws = out.get("workspace")
        a.workspace = _ptr(ws)
        a.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
        a.weights = _ptr(weights)
        return a

    def run(self, x, phi, alpha, bias, out, gamma=None, pre_mix=None, stream=None, weights=None):
        """Enqueue the forward on `stream` (torch stream or raw handle; default:
        torch's current stream).  `weights` (from prepare_weights) replaces
        phi and gamma.  Raises MhcError on a host-side rejection."""
        args = self.make_args(x, phi, alpha, bias, out, gamma, pre_mix, weights)
        if stream is None:
            import torch
            stream = torch.cuda.current_stream(x.device).cuda_stream
        elif hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        st = mhc_pre_run(self.handle, args, int(stream))
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_run", last_error())
        return out

    def backward_workspace_size(self, T: int) -> int:
        st, n = mhc_pre_backward_workspace_size(self.handle, T)
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_backward_workspace_size", last_error())
        return n

    def allocate_backward(self, T, device, *, gamma: bool = False):
        """Gradient outputs and workspace for T tokens, or a (B, S) batch in
        the BSND layout (torch supplies the memory)."""
        import torch
        lead = (T,) if isinstance(T, int) else tuple(T)
        T = _tokens(lead)
        n, D, R = self.n, self.D, self.R
        f32 = dict(dtype=torch.float32, device=device)
        return {"grad_x": torch.empty(lead + (n, D), dtype=torch.bfloat16, device=device),
                "grad_phi": torch.empty((R, n * D), **f32),
                "grad_alpha": torch.empty((3,), **f32),
                "grad_bias": torch.empty((R,), **f32),
                "grad_gamma": torch.empty((n, D), **f32) if gamma else None,
                "workspace": torch.zeros((max(self.backward_workspace_size(T), 256),),
                                         dtype=torch.uint8, device=device)}

    def make_backward_args(self, x, phi, alpha, gamma, grad_h_in, grad_h_post, grad_h_res, saved,
                           grads, grad_x_post=None) -> MhcPreBwdArgs:
        """saved: the forward's outputs (inv_rms, h_mix, h_pre, h_post and,
        for the Sinkhorn form, sum_out / norm_out -- None selects the logit
        form); grads: from allocate_backward."""
        a = MhcPreBwdArgs()
        a.T = _tokens(x.shape[:-2])
        a.x, a.phi, a.alpha, a.gamma = _ptr(x), _ptr(phi), _ptr(alpha), _ptr(gamma)
        a.grad_h_in, a.grad_h_post, a.grad_h_res = _ptr(grad_h_in), _ptr(grad_h_post), _ptr(grad_h_res)
        for k in ("inv_rms", "h_mix", "h_pre", "h_post", "sum_out", "norm_out"):
            setattr(a, k, _ptr(saved.get(k)))
        a.grad_x_post = _ptr(grad_x_post)
        for k in ("grad_x", "grad_phi", "grad_alpha", "grad_bias", "grad_gamma"):
            setattr(a, k, _ptr(grads.get(k)))
        ws = grads.get("workspace")
        a.workspace = _ptr(ws)
        a.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()
        return a

    def backward(self, x, phi, alpha, gamma, grad_h_in, grad_h_post, grad_h_res, saved, grads,
                 grad_x_post=None, stream=None):
        """Enqueue the backward on `stream` (default: torch's current stream).
        Raises MhcError on a host-side rejection."""
        args = self.make_backward_args(x, phi, alpha, gamma, grad_h_in, grad_h_post, grad_h_res, saved,
                                       grads, grad_x_post)
        if stream is None:
            import torch
            stream = torch.cuda.current_stream(x.device).cuda_stream
        elif hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        st = mhc_pre_backward_run(self.handle, args, int(stream))
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_backward_run", last_error())
        return grads

    def run_composite(self, x, phi, alpha, bias, out, gamma=None, pre_mix=None, stream=None):
        """The composite route (include/mhc_pre_stages.h): invRms, the mixes,
        then gates + Sinkhorn + y, as three launches on `stream`; fills the
        same outputs as run().  A debug aid: slower than the fused run()."""
        import torch
        T = _tokens(x.shape[:-2])
        if stream is None:
            stream = torch.cuda.current_stream(x.device).cuda_stream
        elif hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        ir = out.get("inv_rms")
        ir = ir if ir is not None else torch.empty((T,), dtype=torch.float32, device=x.device)
        mx = out.get("h_mix")
        mx = mx if mx is not None else torch.empty((T, self.R), dtype=torch.float32, device=x.device)
        st = mhc_pre_inv_rms_run(self.handle, T, _ptr(x), _ptr(ir), int(stream))
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_inv_rms_run", last_error())
        st = mhc_pre_mixes_run(self.handle, T, _ptr(x), _ptr(phi), _ptr(gamma), _ptr(mx), int(stream))
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_mixes_run", last_error())
        args = self.make_args(x, phi, alpha, bias, out, gamma, pre_mix)
        st = mhc_pre_sinkhorn_run(self.handle, args, _ptr(mx), _ptr(ir), int(stream))
        if st != MHC_OK:
            raise MhcError(st, "mhc_pre_sinkhorn_run", last_error())
        return out

    def status(self, out=None, stream=None) -> int:
        ws = None if out is None else out.get("workspace")
        if stream is None:
            stream = 0
        elif hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        return mhc_pre_status(self.handle, _ptr(ws) or 0, int(stream))
