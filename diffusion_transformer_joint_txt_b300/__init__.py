"""B300-native joint text/image attention for FLUX-style diffusion transformers.

Python binding of the C ABI declared in ``include/flux_attn.h``.  It does
argument marshalling only -- torch tensors become device pointers, the current
torch CUDA stream becomes the ``cudaStream_t`` -- and every step of the path
runs in the kernels of ``libflux_attn.so``.  There is no fallback: the first
call into the package without the built library raises ImportError (the
library is loaded on first use so that the build module itself can be
imported before it exists).

Entry points keep the C names (``flux_attn_create``, ``flux_attn_forward``,
``flux_attn_prologue``, ``flux_attn_attend``, ``flux_attn_sync_status``,
``flux_attn_destroy`` ...); ``FluxAttention`` wraps a handle for convenience.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflux_attn.so")

FLUX_ATTN_OK = 0
FLUX_ATTN_ERR_INVALID_ARG = 1
FLUX_ATTN_ERR_UNSUPPORTED = 2
FLUX_ATTN_ERR_OOM = 3
FLUX_ATTN_ERR_CUDA = 4
FLUX_ATTN_ERR_DEVICE_TIMEOUT = 5
FLUX_ATTN_BF16 = 0
FLUX_ATTN_FP8_E4M3 = 1
FLUX_ATTN_DEBUG_FORCE_TIMEOUT = 1

HEAD_DIM = 128


class flux_attn_config(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("max_tokens", ctypes.c_int),
        ("axes_dim", ctypes.c_int * 3),
        ("rope_theta", ctypes.c_float),
        ("rms_eps", ctypes.c_float),
        ("precision", ctypes.c_int),
        ("debug_flags", ctypes.c_int),
        ("vc_repair_budget", ctypes.c_float),
        ("sol_tau", ctypes.c_float),
        ("sol_disabled_until_timestep", ctypes.c_float),
    ]


class FluxAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("flux_attn status %d (%s): %s" % (status, _status_string(status), message))
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libflux_attn.so is not built; run `python -m diffusion_transformer_joint_txt_b300.build` "
                          "(expected at %s)" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "flux_attn_create": (I, [ctypes.POINTER(flux_attn_config), ctypes.POINTER(P)]),
        "flux_attn_destroy": (I, [P]),
        "flux_attn_forward": (I, [P, P, P, P, I, I, I, I, I, P, P, P, P, P]),
        "flux_attn_prologue": (I, [P, P, P, I, I, I, I, I, P, P, P, P, P, P]),
        "flux_attn_attend": (I, [P, P, P, P, I, P, P]),
        "flux_attn_prologue_fp8": (I, [P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, P, P]),
        "flux_attn_attend_fp8": (I, [P, P, P, P, P, I, P, P]),
        "flux_attn_prologue_fp8_vc": (I, [P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P]),
        "flux_attn_attend_fp8_vc": (I, [P, P, P, P, P, P, P, I, P, P]),
        "flux_attn_vc_repair_count": (I, [P, I]),
        "flux_attn_forward_sol": (I, [P, P, P, P, I, I, I, I, I, P, P, P, ctypes.c_float, P, P]),
        "flux_attn_sol_mask": (I, [P, P, P, I, P, P]),
        "flux_attn_attend_sol": (I, [P, P, P, P, P, I, P, P]),
        "flux_attn_qkv": (I, [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P]),
        "flux_attn_forward_hidden": (I, [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P]),
        "flux_attn_qkv_fp8": (I, [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P]),
        "flux_attn_forward_noalloc": (I, [ctypes.POINTER(flux_attn_config), P, P, P, I, I, I, I, I, P, P, P, P,
                                          P, P]),
        "flux_attn_sync_status": (I, [P, P]),
        "flux_attn_workspace_bytes": (Z, [P]),
        "flux_attn_launches_per_forward": (I, [P, I]),
        "flux_attn_status_string": (ctypes.c_char_p, [I]),
        "flux_attn_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib_handle = [None]


def _L() -> ctypes.CDLL:
    """The loaded library; raises ImportError when it has not been built."""
    if _lib_handle[0] is None:
        _lib_handle[0] = _load()
    return _lib_handle[0]


def _status_string(status: int) -> str:
    return _L().flux_attn_status_string(status).decode()


def _check(status: int) -> int:
    if status != FLUX_ATTN_OK:
        raise FluxAttnError(status, _L().flux_attn_last_error().decode())
    return status


def _ptr(t) -> Optional[int]:
    """Device pointer of a tensor (or a raw integer address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def library_path() -> str:
    return LIB_PATH


# ------------------------------------------------------------ C-named calls

def flux_attn_create(batch: int, num_heads: int, max_tokens: int, head_dim: int = HEAD_DIM,
                     axes_dim: Sequence[int] = (16, 56, 56), rope_theta: float = 10000.0,
                     rms_eps: float = 1e-6, precision: int = FLUX_ATTN_BF16, debug_flags: int = 0,
                     vc_repair_budget: float = 0.0, sol_tau: float = 0.0,
                     sol_disabled_until_timestep: float = 0.96) -> int:
    cfg = flux_attn_config(batch, num_heads, head_dim, max_tokens, (ctypes.c_int * 3)(*axes_dim),
                           rope_theta, rms_eps, precision, debug_flags, vc_repair_budget, sol_tau,
                           sol_disabled_until_timestep)
    h = ctypes.c_void_p()
    _check(_L().flux_attn_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def flux_attn_destroy(h: int) -> None:
    _check(_L().flux_attn_destroy(h))


def flux_attn_forward(h, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                      out, stream=None) -> None:
    _check(_L().flux_attn_forward(h, _ptr(q), _ptr(k), _ptr(v), txt_len, img_h, img_w, ref_h, ref_w,
                                  _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out), _stream(stream)))


def flux_attn_prologue(h, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                       qn, kn, stream=None) -> None:
    _check(_L().flux_attn_prologue(h, _ptr(q), _ptr(k), txt_len, img_h, img_w, ref_h, ref_w, _ptr(pos_ids),
                                   _ptr(q_norm_w), _ptr(k_norm_w), _ptr(qn), _ptr(kn), _stream(stream)))


def flux_attn_attend(h, qn, kn, v, n_tokens, out, stream=None) -> None:
    _check(_L().flux_attn_attend(h, _ptr(qn), _ptr(kn), _ptr(v), n_tokens, _ptr(out), _stream(stream)))


def flux_attn_prologue_fp8(h, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                           q8, k8, v8t, scales, stream=None) -> None:
    _check(_L().flux_attn_prologue_fp8(h, _ptr(q), _ptr(k), _ptr(v), txt_len, img_h, img_w, ref_h, ref_w,
                                       _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(q8), _ptr(k8),
                                       _ptr(v8t), _ptr(scales), _stream(stream)))


def flux_attn_attend_fp8(h, q8, k8, v8t, scales, n_tokens, out, stream=None) -> None:
    _check(_L().flux_attn_attend_fp8(h, _ptr(q8), _ptr(k8), _ptr(v8t), _ptr(scales), n_tokens, _ptr(out),
                                     _stream(stream)))


def flux_attn_prologue_fp8_vc(h, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                              q8, k8, v8t, scales, repair_idx, k_rep, v_rep, stream=None) -> None:
    _check(_L().flux_attn_prologue_fp8_vc(h, _ptr(q), _ptr(k), _ptr(v), txt_len, img_h, img_w, ref_h, ref_w,
                                          _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(q8), _ptr(k8),
                                          _ptr(v8t), _ptr(scales), _ptr(repair_idx), _ptr(k_rep), _ptr(v_rep),
                                          _stream(stream)))


def flux_attn_attend_fp8_vc(h, q8, k8, v8t, scales, k_rep, v_rep, n_tokens, out, stream=None) -> None:
    _check(_L().flux_attn_attend_fp8_vc(h, _ptr(q8), _ptr(k8), _ptr(v8t), _ptr(scales), _ptr(k_rep), _ptr(v_rep),
                                        n_tokens, _ptr(out), _stream(stream)))


def flux_attn_vc_repair_count(h, n_tokens: int) -> int:
    return int(_L().flux_attn_vc_repair_count(h, n_tokens))


def flux_attn_forward_sol(h, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w, timestep,
                          out, stream=None) -> None:
    _check(_L().flux_attn_forward_sol(h, _ptr(q), _ptr(k), _ptr(v), txt_len, img_h, img_w, ref_h, ref_w,
                                      _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), float(timestep), _ptr(out),
                                      _stream(stream)))


def flux_attn_sol_mask(h, qn, kn, n_tokens, keep, stream=None) -> None:
    _check(_L().flux_attn_sol_mask(h, _ptr(qn), _ptr(kn), n_tokens, _ptr(keep), _stream(stream)))


def flux_attn_attend_sol(h, qn, kn, v, keep, n_tokens, out, stream=None) -> None:
    _check(_L().flux_attn_attend_sol(h, _ptr(qn), _ptr(kn), _ptr(v), _ptr(keep), n_tokens, _ptr(out),
                                     _stream(stream)))


def flux_attn_qkv(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                  qn, kn, v, stream=None) -> None:
    _check(_L().flux_attn_qkv(h, _ptr(x), _ptr(w_qkv), _ptr(b_qkv), d_model, txt_len, img_h, img_w, ref_h, ref_w,
                              _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(qn), _ptr(kn), _ptr(v),
                              _stream(stream)))


def flux_attn_qkv_fp8(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w,
                      k_norm_w, q8, k8, v8t, scales, stream=None) -> None:
    _check(_L().flux_attn_qkv_fp8(h, _ptr(x), _ptr(w_qkv), _ptr(b_qkv), d_model, txt_len, img_h, img_w, ref_h, ref_w,
                                  _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(q8), _ptr(k8), _ptr(v8t),
                                  _ptr(scales), _stream(stream)))


def flux_attn_forward_hidden(h, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w, pos_ids,
                             q_norm_w, k_norm_w, out, stream=None) -> None:
    _check(_L().flux_attn_forward_hidden(h, _ptr(x), _ptr(w_qkv), _ptr(b_qkv), d_model, txt_len, img_h, img_w,
                                         ref_h, ref_w, _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out),
                                         _stream(stream)))


def make_config(batch: int, num_heads: int, max_tokens: int, head_dim: int = HEAD_DIM,
                axes_dim: Sequence[int] = (16, 56, 56), rope_theta: float = 10000.0, rms_eps: float = 1e-6,
                precision: int = FLUX_ATTN_BF16, debug_flags: int = 0,
                vc_repair_budget: float = 0.0, sol_tau: float = 0.0,
                sol_disabled_until_timestep: float = 0.96) -> flux_attn_config:
    return flux_attn_config(batch, num_heads, head_dim, max_tokens, (ctypes.c_int * 3)(*axes_dim),
                            rope_theta, rms_eps, precision, debug_flags, vc_repair_budget, sol_tau,
                            sol_disabled_until_timestep)


def flux_attn_forward_noalloc(cfg: flux_attn_config, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids,
                              q_norm_w, k_norm_w, out, device_error=None, stream=None) -> None:
    """The allocation-free forward: same result as flux_attn_forward without a
    handle and without any device allocation (for callers that reserve all
    device memory up front).  Its scratch is one array shared by every call on
    a device, so calls must not overlap on the GPU; the limit is
    batch * num_heads * N <= 32768."""
    _check(_L().flux_attn_forward_noalloc(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), txt_len, img_h, img_w,
                                          ref_h, ref_w, _ptr(pos_ids), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(out),
                                          _ptr(device_error), _stream(stream)))


def flux_attn_sync_status(h, stream=None) -> int:
    """Synchronise the stream and return the device status (no exception)."""
    return int(_L().flux_attn_sync_status(h, _stream(stream)))


def flux_attn_workspace_bytes(h) -> int:
    return int(_L().flux_attn_workspace_bytes(h))


def flux_attn_launches_per_forward(h, n_tokens: int) -> int:
    return int(_L().flux_attn_launches_per_forward(h, n_tokens))


def flux_attn_status_string(status: int) -> str:
    return _status_string(status)


def flux_attn_last_error() -> str:
    return _L().flux_attn_last_error().decode()


# ---------------------------------------------------------------- wrapper

def pad16(n: int) -> int:
    """Row length of the transposed FP8 V: N rounded up to a multiple of 16."""
    return (n + 15) // 16 * 16


def _require(t, dtype, shape, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be a contiguous CUDA %s tensor of shape %s (got %s %s %s)"
                         % (name, dtype, tuple(shape), t.dtype, t.device, tuple(t.shape)))


class FluxAttention:
    """One library handle: joint attention with the QK-RMSNorm + RoPE prologue.

    Tensors are torch CUDA tensors on the handle's device: q, k, v, out bf16
    [B, N, H, 128]; q_norm_w, k_norm_w fp32 [128]; pos_ids int32 [N, 3] or
    None (positions derived from the text/image/reference geometry).
    """

    def __init__(self, batch: int, num_heads: int, max_tokens: int, precision: str = "bf16",
                 axes_dim: Sequence[int] = (16, 56, 56), rope_theta: float = 10000.0,
                 rms_eps: float = 1e-6, debug_flags: int = 0, vc_repair_budget: float = 0.0,
                 sol_tau: float = 0.0, sol_disabled_until_timestep: float = 0.96):
        """precision "bf16" or "fp8"; vc_repair_budget > 0 (FP8 only) turns on
        the VC-Attention repair of the ceil(rho N) worst-quantised key tokens;
        sol_tau > 0 (BF16 only) enables the block-sparse Sol-Attention calls."""
        self.batch, self.num_heads, self.max_tokens = batch, num_heads, max_tokens
        self.precision = precision
        prec = {"bf16": FLUX_ATTN_BF16, "fp8": FLUX_ATTN_FP8_E4M3}[precision]
        self.handle = flux_attn_create(batch, num_heads, max_tokens, HEAD_DIM, axes_dim, rope_theta, rms_eps,
                                       prec, debug_flags, vc_repair_budget, sol_tau, sol_disabled_until_timestep)

    def close(self) -> None:
        if getattr(self, "handle", None):
            flux_attn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _shape(self, n: int) -> Tuple[int, int, int, int]:
        return (self.batch, n, self.num_heads, HEAD_DIM)

    def forward(self, q, k, v, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                q_norm_w=None, k_norm_w=None, pos_ids=None, out=None, stream=None):
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        for t, name in ((q, "q"), (k, "k"), (v, "v")):
            _require(t, torch.bfloat16, self._shape(n), name)
        _require(q_norm_w, torch.float32, (HEAD_DIM,), "q_norm_w")
        _require(k_norm_w, torch.float32, (HEAD_DIM,), "k_norm_w")
        if pos_ids is not None:
            _require(pos_ids, torch.int32, (n, 3), "pos_ids")
        if out is None:
            out = torch.empty_like(q)
        _require(out, torch.bfloat16, self._shape(n), "out")
        flux_attn_forward(self.handle, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w,
                          k_norm_w, out, stream)
        return out

    def prologue(self, q, k, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                 q_norm_w=None, k_norm_w=None, pos_ids=None, qn=None, kn=None, stream=None):
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        _require(q, torch.bfloat16, self._shape(n), "q")
        _require(k, torch.bfloat16, self._shape(n), "k")
        _require(q_norm_w, torch.float32, (HEAD_DIM,), "q_norm_w")
        _require(k_norm_w, torch.float32, (HEAD_DIM,), "k_norm_w")
        hm = (self.batch, self.num_heads, n, HEAD_DIM)
        qn = torch.empty(hm, dtype=torch.bfloat16, device=q.device) if qn is None else qn
        kn = torch.empty(hm, dtype=torch.bfloat16, device=q.device) if kn is None else kn
        _require(qn, torch.bfloat16, hm, "qn")
        _require(kn, torch.bfloat16, hm, "kn")
        flux_attn_prologue(self.handle, q, k, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                           qn, kn, stream)
        return qn, kn

    def attend(self, qn, kn, v, out=None, stream=None):
        import torch
        n = qn.shape[2]
        hm = (self.batch, self.num_heads, n, HEAD_DIM)
        _require(qn, torch.bfloat16, hm, "qn")
        _require(kn, torch.bfloat16, hm, "kn")
        _require(v, torch.bfloat16, self._shape(n), "v")
        out = torch.empty_like(v) if out is None else out
        _require(out, torch.bfloat16, self._shape(n), "out")
        flux_attn_attend(self.handle, qn, kn, v, n, out, stream)
        return out

    def qkv(self, x, w_qkv, b_qkv, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
            q_norm_w=None, k_norm_w=None, pos_ids=None, qn=None, kn=None, v=None, stream=None):
        """QKV projection with the fused QK-norm + RoPE epilogue: x bf16
        [B, N, d_model] (or [B*N, d_model]), w_qkv bf16 [3 H 128, d_model],
        b_qkv fp32 [3 H 128] or None.  Returns (qn, kn, v): bf16
        [B, H, N, 128], [B, H, N, 128], [B, N, H, 128]."""
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        B, H = self.batch, self.num_heads
        d_model = x.shape[-1]
        if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.numel() != B * n * d_model:
            raise ValueError("x must be a contiguous CUDA bf16 tensor of B * N * d_model elements")
        _require(w_qkv, torch.bfloat16, (3 * H * HEAD_DIM, d_model), "w_qkv")
        if b_qkv is not None:
            _require(b_qkv, torch.float32, (3 * H * HEAD_DIM,), "b_qkv")
        _require(q_norm_w, torch.float32, (HEAD_DIM,), "q_norm_w")
        _require(k_norm_w, torch.float32, (HEAD_DIM,), "k_norm_w")
        if pos_ids is not None:
            _require(pos_ids, torch.int32, (n, 3), "pos_ids")
        hm = (B, H, n, HEAD_DIM)
        qn = torch.empty(hm, dtype=torch.bfloat16, device=x.device) if qn is None else qn
        kn = torch.empty(hm, dtype=torch.bfloat16, device=x.device) if kn is None else kn
        v = torch.empty(self._shape(n), dtype=torch.bfloat16, device=x.device) if v is None else v
        _require(qn, torch.bfloat16, hm, "qn")
        _require(kn, torch.bfloat16, hm, "kn")
        _require(v, torch.bfloat16, self._shape(n), "v")
        flux_attn_qkv(self.handle, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w, pos_ids,
                      q_norm_w, k_norm_w, qn, kn, v, stream)
        return qn, kn, v

    def qkv_fp8(self, x, w_qkv, b_qkv, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                q_norm_w=None, k_norm_w=None, pos_ids=None, stream=None):
        """FP8 handles: the QKV projection (fused QK-norm + RoPE) to E4M3 codes;
        returns (q8, k8, v8t, scales) as prologue_fp8 does."""
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        B, H = self.batch, self.num_heads
        new = lambda shape, dt: torch.empty(shape, dtype=dt, device=x.device)
        q8, k8 = new((B, H, n, HEAD_DIM), torch.uint8), new((B, H, n, HEAD_DIM), torch.uint8)
        v8t, scales = new((B, H, HEAD_DIM, pad16(n)), torch.uint8), new((B, H, 3), torch.float32)
        flux_attn_qkv_fp8(self.handle, x, w_qkv, b_qkv, x.shape[-1], txt_len, img_h, img_w, ref_h, ref_w, pos_ids,
                          q_norm_w, k_norm_w, q8, k8, v8t, scales, stream)
        return q8, k8, v8t, scales

    def forward_hidden(self, x, w_qkv, b_qkv, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                       q_norm_w=None, k_norm_w=None, pos_ids=None, out=None, stream=None):
        """QKV projection (fused QK-norm + RoPE) and joint attention in one call;
        returns out bf16 [B, N, H, 128]."""
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        d_model = x.shape[-1]
        if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or \
                x.numel() != self.batch * n * d_model:
            raise ValueError("x must be a contiguous CUDA bf16 tensor of B * N * d_model elements")
        _require(w_qkv, torch.bfloat16, (3 * self.num_heads * HEAD_DIM, d_model), "w_qkv")
        if b_qkv is not None:
            _require(b_qkv, torch.float32, (3 * self.num_heads * HEAD_DIM,), "b_qkv")
        _require(q_norm_w, torch.float32, (HEAD_DIM,), "q_norm_w")
        _require(k_norm_w, torch.float32, (HEAD_DIM,), "k_norm_w")
        if pos_ids is not None:
            _require(pos_ids, torch.int32, (n, 3), "pos_ids")
        out = torch.empty(self._shape(n), dtype=torch.bfloat16, device=x.device) if out is None else out
        _require(out, torch.bfloat16, self._shape(n), "out")
        flux_attn_forward_hidden(self.handle, x, w_qkv, b_qkv, d_model, txt_len, img_h, img_w, ref_h, ref_w,
                                 pos_ids, q_norm_w, k_norm_w, out, stream)
        return out

    def prologue_fp8(self, q, k, v, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                     q_norm_w=None, k_norm_w=None, pos_ids=None, q8=None, k8=None, v8t=None, scales=None,
                     stream=None):
        """FP8 handles: E4M3 codes q8, k8 [B, H, N, 128], v8t [B, H, 128, pad16(N)]
        (uint8 tensors; v8t holds the keys of every 8 columns in the order
        0 2 4 6 1 3 5 7 that attend_fp8 reads) and scales [B, H, 3] (fp32), into
        the given tensors or new ones."""
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        for t, name in ((q, "q"), (k, "k"), (v, "v")):
            _require(t, torch.bfloat16, self._shape(n), name)
        _require(q_norm_w, torch.float32, (HEAD_DIM,), "q_norm_w")
        _require(k_norm_w, torch.float32, (HEAD_DIM,), "k_norm_w")
        if pos_ids is not None:
            _require(pos_ids, torch.int32, (n, 3), "pos_ids")
        B, H = self.batch, self.num_heads
        new = lambda shape, dt: torch.empty(shape, dtype=dt, device=q.device)
        q8 = new((B, H, n, HEAD_DIM), torch.uint8) if q8 is None else q8
        k8 = new((B, H, n, HEAD_DIM), torch.uint8) if k8 is None else k8
        v8t = new((B, H, HEAD_DIM, pad16(n)), torch.uint8) if v8t is None else v8t
        scales = new((B, H, 3), torch.float32) if scales is None else scales
        _require(q8, torch.uint8, (B, H, n, HEAD_DIM), "q8")
        _require(k8, torch.uint8, (B, H, n, HEAD_DIM), "k8")
        _require(v8t, torch.uint8, (B, H, HEAD_DIM, pad16(n)), "v8t")
        _require(scales, torch.float32, (B, H, 3), "scales")
        flux_attn_prologue_fp8(self.handle, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w,
                               k_norm_w, q8, k8, v8t, scales, stream)
        return q8, k8, v8t, scales

    def attend_fp8(self, q8, k8, v8t, scales, out=None, stream=None):
        import torch
        B, H, n = self.batch, self.num_heads, q8.shape[2]
        _require(q8, torch.uint8, (B, H, n, HEAD_DIM), "q8")
        _require(k8, torch.uint8, (B, H, n, HEAD_DIM), "k8")
        _require(v8t, torch.uint8, (B, H, HEAD_DIM, pad16(n)), "v8t")
        _require(scales, torch.float32, (B, H, 3), "scales")
        out = torch.empty((B, n, H, HEAD_DIM), dtype=torch.bfloat16, device=q8.device) if out is None else out
        _require(out, torch.bfloat16, self._shape(n), "out")
        flux_attn_attend_fp8(self.handle, q8, k8, v8t, scales, n, out, stream)
        return out

    def vc_repair_count(self, n_tokens: int) -> int:
        return flux_attn_vc_repair_count(self.handle, n_tokens)

    def prologue_fp8_vc(self, q, k, v, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                        q_norm_w=None, k_norm_w=None, pos_ids=None, stream=None):
        """VC-Attention handles: (q8, k8, v8t, scales, repair_idx, k_rep, v_rep) -- the
        E4M3 codes with the repaired tokens moved out of the first N - R key
        positions, the repaired tokens int32 [B, H, R] ascending, and their rows
        k' / s_k, v / s_v bf16 [B, H, R, 128]."""
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        for t, name in ((q, "q"), (k, "k"), (v, "v")):
            _require(t, torch.bfloat16, self._shape(n), name)
        _require(q_norm_w, torch.float32, (HEAD_DIM,), "q_norm_w")
        _require(k_norm_w, torch.float32, (HEAD_DIM,), "k_norm_w")
        if pos_ids is not None:
            _require(pos_ids, torch.int32, (n, 3), "pos_ids")
        B, H, R = self.batch, self.num_heads, self.vc_repair_count(n)
        new = lambda shape, dt: torch.empty(shape, dtype=dt, device=q.device)
        q8, k8 = new((B, H, n, HEAD_DIM), torch.uint8), new((B, H, n, HEAD_DIM), torch.uint8)
        v8t, scales = new((B, H, HEAD_DIM, pad16(n)), torch.uint8), new((B, H, 3), torch.float32)
        idx = new((B, H, max(R, 1)), torch.int32)
        k_rep, v_rep = new((B, H, max(R, 1), HEAD_DIM), torch.bfloat16), new((B, H, max(R, 1), HEAD_DIM),
                                                                             torch.bfloat16)
        flux_attn_prologue_fp8_vc(self.handle, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w,
                                  k_norm_w, q8, k8, v8t, scales, idx, k_rep, v_rep, stream)
        return q8, k8, v8t, scales, idx, k_rep, v_rep

    def attend_fp8_vc(self, q8, k8, v8t, scales, k_rep, v_rep, out=None, stream=None):
        import torch
        B, H, n = self.batch, self.num_heads, q8.shape[2]
        out = torch.empty((B, n, H, HEAD_DIM), dtype=torch.bfloat16, device=q8.device) if out is None else out
        _require(out, torch.bfloat16, self._shape(n), "out")
        flux_attn_attend_fp8_vc(self.handle, q8, k8, v8t, scales, k_rep, v_rep, n, out, stream)
        return out

    def forward_sol(self, q, k, v, txt_len: int, img_h: int, img_w: int, ref_h: int = 0, ref_w: int = 0,
                    q_norm_w=None, k_norm_w=None, pos_ids=None, timestep: float = 0.0, out=None, stream=None):
        """Sol-Attention forward (dense while timestep > sol_disabled_until_timestep)."""
        import torch
        n = txt_len + img_h * img_w + ref_h * ref_w
        for t, name in ((q, "q"), (k, "k"), (v, "v")):
            _require(t, torch.bfloat16, self._shape(n), name)
        out = torch.empty_like(q) if out is None else out
        _require(out, torch.bfloat16, self._shape(n), "out")
        flux_attn_forward_sol(self.handle, q, k, v, txt_len, img_h, img_w, ref_h, ref_w, pos_ids, q_norm_w, k_norm_w,
                              timestep, out, stream)
        return out

    def sol_mask(self, qn, kn, stream=None):
        """Block mask uint8 [B, H, nb, nb] of Q', K' bf16 [B, H, N, 128]."""
        import torch
        n = qn.shape[2]
        nb = (n + 127) // 128
        keep = torch.empty((self.batch, self.num_heads, nb, nb), dtype=torch.uint8, device=qn.device)
        flux_attn_sol_mask(self.handle, qn, kn, n, keep, stream)
        return keep

    def attend_sol(self, qn, kn, v, keep, out=None, stream=None):
        import torch
        n = qn.shape[2]
        out = torch.empty_like(v) if out is None else out
        _require(out, torch.bfloat16, self._shape(n), "out")
        flux_attn_attend_sol(self.handle, qn, kn, v, keep, n, out, stream)
        return out

    def sync_status(self, stream=None) -> int:
        return flux_attn_sync_status(self.handle, stream)

    def workspace_bytes(self) -> int:
        return flux_attn_workspace_bytes(self.handle)

    def launches_per_forward(self, n_tokens: int) -> int:
        return flux_attn_launches_per_forward(self.handle, n_tokens)
