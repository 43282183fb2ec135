"""fp64 CPU oracle for the joint text/image attention path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library and its Python
binding never import it, and it imports nothing from them.

The arithmetic lives in ``flux_attn_oracle.c`` (plain C, fp64, OpenMP over
rows); this file only compiles it with gcc and marshals numpy arrays.  The
header comment of the C file lists the passages it follows and the readings
taken where the pages are silent.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, library routines in fp64, brute force on tiny
inputs, exhaustive E4M3 round trip).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flux_attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_libs = {}

AXES_DEFAULT = (16, 56, 56)


def compile_source(src: str, out: str) -> str:
    """gcc the oracle source (fp64, no fast-math, no FMA contraction)."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the in-tree oracle library if it is missing or stale."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


_active = [None]


def use_library(path: Optional[str]) -> None:
    """Point the module functions at another build of the oracle source
    (the mutation tests load deliberately broken copies); None restores the
    in-tree build."""
    _active[0] = path


def _load():
    path = _active[0]
    if path is None:
        path = build()
    if path not in _libs:
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        L = ctypes.c_int64
        lib.oracle_max_threads.restype = I
        lib.oracle_e4m3_decode.restype = D
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [D]
        for name in ("oracle_prologue_bf16", "oracle_prologue_f64"):
            f = getattr(lib, name)
            f.restype = I
            f.argtypes = [P, I, I, I, I, P, P, D, D, P, P, I]
        for name in ("oracle_attention_rows_bf16", "oracle_attention_rows_f64"):
            f = getattr(lib, name)
            f.restype = I
            f.argtypes = [P, P, P, I, I, I, I, P, P, P, D, D, P, I, P, L, P, I]
        lib.oracle_qkv_rows.restype = I
        lib.oracle_qkv_rows.argtypes = [P, P, P, I, I, I, I, I, P, P, P, D, D, P, P, L, P, P, P, I]
        lib.oracle_vc_attention_rows_bf16.restype = I
        lib.oracle_vc_attention_rows_bf16.argtypes = [P, P, P, I, I, I, I, P, P, P, D, D, P, D, P, L, P, I]
        lib.oracle_vc_select_head_bf16.restype = L
        lib.oracle_vc_select_head_bf16.argtypes = [P, P, P, I, I, I, I, P, P, P, D, D, P, D, I, I, P, P, I]
        lib.oracle_sol_mask_bf16.restype = L
        lib.oracle_sol_mask_bf16.argtypes = [P, P, I, I, I, I, P, P, P, D, D, P, D, I, I, P, P, I]
        lib.oracle_sol_attention_rows_bf16.restype = I
        lib.oracle_sol_attention_rows_bf16.argtypes = [P, P, P, I, I, I, I, P, P, P, D, D, P, D, P, L, P, I]
        lib.oracle_fp8_quantize_values.restype = D
        lib.oracle_fp8_quantize_values.argtypes = [P, L, P]
        lib.oracle_vc_repair_count.restype = L
        lib.oracle_vc_repair_count.argtypes = [D, L]
        lib.oracle_fp8_quantize_head_bf16.restype = I
        lib.oracle_fp8_quantize_head_bf16.argtypes = [P, P, P, I, I, I, I, P, P, P, D, D, P, I, I,
                                                      P, P, P, P, I]
        _libs[path] = lib
    return _libs[path]


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_encode(x) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    return np.array([lib.oracle_e4m3_encode(float(t)) for t in x.ravel()], np.uint8).reshape(x.shape)


def e4m3_decode(c) -> np.ndarray:
    lib = _load()
    c = np.asarray(c, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(t)) for t in c.ravel()], np.float64).reshape(c.shape)


def _axes(axes: Sequence[int]) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(axes, dtype=np.int32))


def prologue(x: np.ndarray, pos: np.ndarray, w: np.ndarray, eps: float = 1e-6,
             theta: float = 10000.0, axes: Sequence[int] = AXES_DEFAULT, nthreads: int = 0) -> np.ndarray:
    """RMSNorm then RoPE of every [B, N, H, d] row.

    ``x`` is uint16 bf16 bits (weights float32) or float64 (weights float64).
    Returns float64 [B, N, H, d].
    """
    lib = _load()
    B, N, H, d = x.shape
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    assert pos.shape == (N, 3)
    out = np.empty((B, N, H, d), np.float64)
    ax = _axes(axes)
    if x.dtype == np.uint16:
        x = np.ascontiguousarray(x)
        wf = np.ascontiguousarray(w, dtype=np.float32)
        rc = lib.oracle_prologue_bf16(_ptr(x), B, N, H, d, _ptr(pos), _ptr(wf), eps, theta,
                                      _ptr(ax), _ptr(out), nthreads)
    else:
        x = np.ascontiguousarray(x, dtype=np.float64)
        wd = np.ascontiguousarray(w, dtype=np.float64)
        rc = lib.oracle_prologue_f64(_ptr(x), B, N, H, d, _ptr(pos), _ptr(wd), eps, theta,
                                     _ptr(ax), _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle_prologue failed: %d" % rc)
    return out


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, pos: np.ndarray,
                   w_q: np.ndarray, w_k: np.ndarray, rows: Optional[np.ndarray] = None,
                   eps: float = 1e-6, theta: float = 10000.0, axes: Sequence[int] = AXES_DEFAULT,
                   fp8: bool = False, nthreads: int = 0) -> np.ndarray:
    """Joint attention output rows.

    q, k, v: [B, N, H, d], all uint16 bf16 bits (weights float32) or all
    float64 (weights float64).  rows: int64 [R, 3] of (b, h, n); None means
    every row, returned as [B, N, H, d]; otherwise [R, d].
    """
    lib = _load()
    B, N, H, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    full = rows is None
    if full:
        bb, hh, nn = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), indexing="ij")
        rows = np.stack([bb.ravel(), hh.ravel(), nn.ravel()], 1)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.empty((R, d), np.float64)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    assert pos.shape == (N, 3)
    ax = _axes(axes)
    if q.dtype == np.uint16:
        q, k, v = (np.ascontiguousarray(t) for t in (q, k, v))
        wq = np.ascontiguousarray(w_q, dtype=np.float32)
        wk = np.ascontiguousarray(w_k, dtype=np.float32)
        fn = lib.oracle_attention_rows_bf16
    else:
        q, k, v = (np.ascontiguousarray(t, dtype=np.float64) for t in (q, k, v))
        wq = np.ascontiguousarray(w_q, dtype=np.float64)
        wk = np.ascontiguousarray(w_k, dtype=np.float64)
        fn = lib.oracle_attention_rows_f64
    rc = fn(_ptr(q), _ptr(k), _ptr(v), B, N, H, d, _ptr(pos), _ptr(wq), _ptr(wk), eps, theta,
            _ptr(ax), int(bool(fp8)), _ptr(rows), R, _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle_attention_rows failed: %d" % rc)
    if full:
        # rows were ordered (b, h, n); return [B, N, H, d]
        return out.reshape(B, H, N, d).transpose(0, 2, 1, 3).copy()
    return out


def fp8_quantize_head(q, k, v, pos, w_q, w_k, b: int, h: int, eps: float = 1e-6,
                      theta: float = 10000.0, axes: Sequence[int] = AXES_DEFAULT, nthreads: int = 0):
    """E4M3 codes [N, d] of Q', K', V for head (b, h) and their scales (q, k, v)."""
    lib = _load()
    B, N, H, d = q.shape
    q, k, v = (np.ascontiguousarray(t, dtype=np.uint16) for t in (q, k, v))
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    wq = np.ascontiguousarray(w_q, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    q8 = np.empty((N, d), np.uint8)
    k8 = np.empty((N, d), np.uint8)
    v8 = np.empty((N, d), np.uint8)
    sc = np.empty(3, np.float64)
    rc = lib.oracle_fp8_quantize_head_bf16(_ptr(q), _ptr(k), _ptr(v), B, N, H, d, _ptr(pos),
                                           _ptr(wq), _ptr(wk), eps, theta, _ptr(_axes(axes)),
                                           b, h, _ptr(q8), _ptr(k8), _ptr(v8), _ptr(sc), nthreads)
    if rc != 0:
        raise ValueError("oracle_fp8_quantize_head failed: %d" % rc)
    return q8, k8, v8, sc


def fp8_quantize(x: np.ndarray):
    """Reading R5 on an array: (E4M3 codes uint8 of x's shape, scale = amax / 448
    of the whole array, 1 when it is all zero)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    codes = np.empty(x.shape, np.uint8)
    scale = _load().oracle_fp8_quantize_values(_ptr(x), x.size, _ptr(codes))
    return codes, float(scale)


def vc_repair_count(rho: float, n_tokens: int) -> int:
    """R = ceil(rho N), clamped to [0, N]: how many key tokens a head repairs."""
    return int(_load().oracle_vc_repair_count(float(rho), int(n_tokens)))


def vc_attention_rows(q, k, v, pos, w_q, w_k, rho: float, rows: Optional[np.ndarray] = None,
                      eps: float = 1e-6, theta: float = 10000.0, axes: Sequence[int] = AXES_DEFAULT,
                      nthreads: int = 0) -> np.ndarray:
    """VC-Attention FP8 rows (reading R7 of the C source): FP8 attention over the
    dequantised Q', K', V with the ceil(rho N) worst-quantised key tokens of
    every head taking part with their exact K', V.  Arguments and result as
    attention_rows with bf16 inputs."""
    lib = _load()
    B, N, H, d = q.shape
    full = rows is None
    if full:
        bb, hh, nn = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), indexing="ij")
        rows = np.stack([bb.ravel(), hh.ravel(), nn.ravel()], 1)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.empty((R, d), np.float64)
    q, k, v = (np.ascontiguousarray(t, dtype=np.uint16) for t in (q, k, v))
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    wq = np.ascontiguousarray(w_q, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    rc = lib.oracle_vc_attention_rows_bf16(_ptr(q), _ptr(k), _ptr(v), B, N, H, d, _ptr(pos), _ptr(wq), _ptr(wk),
                                           eps, theta, _ptr(_axes(axes)), float(rho), _ptr(rows), R, _ptr(out),
                                           nthreads)
    if rc != 0:
        raise ValueError("oracle_vc_attention_rows failed: %d" % rc)
    if full:
        return out.reshape(B, H, N, d).transpose(0, 2, 1, 3).copy()
    return out


def vc_select_head(q, k, v, pos, w_q, w_k, rho: float, b: int, h: int, eps: float = 1e-6,
                   theta: float = 10000.0, axes: Sequence[int] = AXES_DEFAULT, nthreads: int = 0):
    """Reading R7 for head (b, h): (selected token indices ascending, int64 [R];
    the quantisation error e_m of every key token, float64 [N])."""
    lib = _load()
    B, N, H, d = q.shape
    q, k, v = (np.ascontiguousarray(t, dtype=np.uint16) for t in (q, k, v))
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    wq = np.ascontiguousarray(w_q, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    sel = np.empty(N, np.int64)
    err = np.empty(N, np.float64)
    R = lib.oracle_vc_select_head_bf16(_ptr(q), _ptr(k), _ptr(v), B, N, H, d, _ptr(pos), _ptr(wq), _ptr(wk), eps,
                                       theta, _ptr(_axes(axes)), float(rho), b, h, _ptr(sel), _ptr(err), nthreads)
    if R < 0:
        raise ValueError("oracle_vc_select_head failed: %d" % R)
    return sel[:R].copy(), err


def sol_mask(q, k, pos, w_q, w_k, tau: float, b: int, h: int, eps: float = 1e-6, theta: float = 10000.0,
             axes: Sequence[int] = AXES_DEFAULT, nthreads: int = 0):
    """Reading R8 for head (b, h): (keep bool [nb, nb], mass float64 [nb, nb]) --
    query block i keeps key block j, and the pooled mass mu_ij."""
    lib = _load()
    B, N, H, d = q.shape
    nb = (N + 127) // 128
    q, k = (np.ascontiguousarray(t, dtype=np.uint16) for t in (q, k))
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    wq = np.ascontiguousarray(w_q, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    keep = np.empty((nb, nb), np.uint8)
    mass = np.empty((nb, nb), np.float64)
    r = lib.oracle_sol_mask_bf16(_ptr(q), _ptr(k), B, N, H, d, _ptr(pos), _ptr(wq), _ptr(wk), eps, theta,
                                 _ptr(_axes(axes)), float(tau), b, h, _ptr(keep), _ptr(mass), nthreads)
    if r != nb:
        raise ValueError("oracle_sol_mask failed: %d" % r)
    return keep.astype(bool), mass


def sol_attention_rows(q, k, v, pos, w_q, w_k, tau: float, rows: Optional[np.ndarray] = None, eps: float = 1e-6,
                       theta: float = 10000.0, axes: Sequence[int] = AXES_DEFAULT, nthreads: int = 0) -> np.ndarray:
    """Sol-Attention rows (reading R8 of the C source): each query attends to
    the keys of the 128-token key blocks its query block keeps.  Arguments
    and result as attention_rows with bf16 inputs."""
    lib = _load()
    B, N, H, d = q.shape
    full = rows is None
    if full:
        bb, hh, nn = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), indexing="ij")
        rows = np.stack([bb.ravel(), hh.ravel(), nn.ravel()], 1)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.empty((R, d), np.float64)
    q, k, v = (np.ascontiguousarray(t, dtype=np.uint16) for t in (q, k, v))
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    wq = np.ascontiguousarray(w_q, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    rc = lib.oracle_sol_attention_rows_bf16(_ptr(q), _ptr(k), _ptr(v), B, N, H, d, _ptr(pos), _ptr(wq), _ptr(wk),
                                            eps, theta, _ptr(_axes(axes)), float(tau), _ptr(rows), R, _ptr(out),
                                            nthreads)
    if rc != 0:
        raise ValueError("oracle_sol_attention_rows failed: %d" % rc)
    if full:
        return out.reshape(B, H, N, d).transpose(0, 2, 1, 3).copy()
    return out


def qkv_rows(x: np.ndarray, w: np.ndarray, bias: Optional[np.ndarray], n_tokens: int, pos: np.ndarray,
             w_q: np.ndarray, w_k: np.ndarray, heads: int, rows: Optional[np.ndarray] = None,
             eps: float = 1e-6, theta: float = 10000.0, axes: Sequence[int] = AXES_DEFAULT, nthreads: int = 0):
    """QKV projection y = x W^T (+ bias) of the requested token rows, split into
    heads, with RMSNorm + RoPE on Q and K (reading R6 of the C source).

    x: uint16 bf16 bits [M, D] (M = B * N); w: uint16 bf16 bits [3 H d, D];
    bias: float32 [3 H d] or None.  Returns (q, k, v), each float64
    [R, H, d] for rows (int64 token indices; None = all M rows).
    """
    lib = _load()
    M, D = x.shape
    F = w.shape[0]
    d = F // (3 * heads)
    assert w.shape == (3 * heads * d, D) and M % n_tokens == 0
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = [np.empty((R, heads, d), np.float64) for _ in range(3)]
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    assert pos.shape == (n_tokens, 3)
    wq = np.ascontiguousarray(w_q, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    rc = lib.oracle_qkv_rows(_ptr(x), _ptr(w), None if b is None else _ptr(b), M, D, heads, d, n_tokens,
                             _ptr(pos), _ptr(wq), _ptr(wk), eps, theta, _ptr(_axes(axes)), _ptr(rows), R,
                             _ptr(out[0]), _ptr(out[1]), _ptr(out[2]), nthreads)
    if rc != 0:
        raise ValueError("oracle_qkv_rows failed: %d" % rc)
    return tuple(out)
