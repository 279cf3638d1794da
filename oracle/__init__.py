"""fp64 CPU oracle for the exact-attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, two passes per row); this
module only builds it with gcc and marshals arrays.  What it computes, per query row i of head
(b, hq), is the dense definition that the tiled online-softmax method reaches up to rounding order
("Attention Kernel 实现与正确性验证", walkerchi.com, section 1.1 and 1.2; "Triton-CUDA Attention",
skillmd.com, GQA and causal variants; "Flash Attention 与 Kernel 优化", fangpin.github.io,
"输出与保存状态"):

    h_kv = hq * Hkv // Hq ;  J(i) = causal ? {0..i} : {0..N-1}
    s_j  = sm_scale * <Q[b,hq,i,:], K[b,h_kv,j,:]>
    O    = sum_j exp(s_j - m) V[b,h_kv,j,:] / sum_j exp(s_j - m),   m = max_j s_j
    LSE  = m + ln sum_j exp(s_j - m)

``attn_bwd_ref`` gives the gradients of the same definition (the pages' backward by recompute).
``mla_decode_ref`` (``mla_oracle.c``) is absorbed MLA decode in the compressed space ("Attention
Kernel 实现与正确性验证", walkerchi.com, sections 2.1 and 2.2).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "mla_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``oracle/_build/liboracle.so`` (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and all(
        os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src) for src in _SRCS)
    if fresh and not force:
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f64p = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int32)
            c_int = ctypes.c_int
            lib.oracle_attn_fwd_f64.argtypes = [u16p, u16p, u16p, c_int, c_int, c_int, c_int, c_int,
                                                c_int, ctypes.c_double, i32p, c_int, f64p, f64p,
                                                c_int]
            lib.oracle_attn_fwd_f64.restype = c_int
            lib.oracle_attn_probs_f64.argtypes = [u16p, u16p, u16p, c_int, c_int, c_int, c_int,
                                                  c_int, c_int, ctypes.c_double, f64p, f64p, f64p,
                                                  c_int]
            lib.oracle_attn_probs_f64.restype = c_int
            lib.oracle_attn_bwd_f64.argtypes = [u16p, u16p, u16p, u16p, c_int, c_int, c_int,
                                                c_int, c_int, c_int, ctypes.c_double, f64p, f64p,
                                                f64p, c_int]
            lib.oracle_attn_bwd_f64.restype = c_int
            lib.oracle_mla_decode_f64.argtypes = [f64p, f64p, c_int, c_int, c_int, c_int, c_int,
                                                  ctypes.c_double, f64p, f64p, c_int]
            lib.oracle_mla_decode_f64.restype = c_int
            lib.oracle_default_threads.argtypes = []
            lib.oracle_default_threads.restype = c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    """Cores the oracle uses when ``n_threads <= 0``."""
    return int(_load().oracle_default_threads())


def _bf16_bits(x) -> np.ndarray:
    """Raw bf16 bit patterns (uint16, C-contiguous) of a torch bf16 tensor or a uint16 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch

    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected a bf16 tensor, got {x.dtype}")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, Hq, N, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != D:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return B, Hq, k.shape[1], N, D


def attn_ref(q, k, v, causal: bool, sm_scale: float, rows=None, n_threads: int = 0):
    """Oracle output and LSE in float64.

    ``q`` [B,Hq,N,D], ``k``/``v`` [B,Hkv,N,D]: torch bf16 tensors or uint16 bf16-bit arrays.
    ``rows``: None for every row (returns O [B,Hq,N,D], LSE [B,Hq,N]); or an int array
    [B, Hq, R] of query rows per head (returns O [B,Hq,R,D], LSE [B,Hq,R]).
    """
    lib = _load()
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    B, Hq, Hkv, N, D = _shapes(qb, kb, vb)
    if rows is None:
        R = N
        rows_arr = None
        rp = ctypes.POINTER(ctypes.c_int32)()
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        if rows_arr.ndim != 3 or rows_arr.shape[:2] != (B, Hq):
            raise ValueError(f"rows must be [B={B}, Hq={Hq}, R], got {rows_arr.shape}")
        R = rows_arr.shape[2]
        rp = _ptr(rows_arr, ctypes.c_int32)
    out = np.zeros((B, Hq, R, D), dtype=np.float64)
    lse = np.zeros((B, Hq, R), dtype=np.float64)
    st = lib.oracle_attn_fwd_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                 _ptr(vb, ctypes.c_uint16), B, Hq, Hkv, N, D, int(bool(causal)),
                                 float(sm_scale), rp, R, _ptr(out, ctypes.c_double),
                                 _ptr(lse, ctypes.c_double), int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_attn_fwd_f64 rejected its arguments (status {st})")
    return out, lse


def attn_probs(q, k, v, causal: bool, sm_scale: float, n_threads: int = 0):
    """Oracle O, LSE and the probability matrix P [B,Hq,N,N] (tiny N only), all float64."""
    lib = _load()
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    B, Hq, Hkv, N, D = _shapes(qb, kb, vb)
    out = np.zeros((B, Hq, N, D), dtype=np.float64)
    lse = np.zeros((B, Hq, N), dtype=np.float64)
    probs = np.zeros((B, Hq, N, N), dtype=np.float64)
    st = lib.oracle_attn_probs_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                   _ptr(vb, ctypes.c_uint16), B, Hq, Hkv, N, D,
                                   int(bool(causal)), float(sm_scale), _ptr(out, ctypes.c_double),
                                   _ptr(lse, ctypes.c_double), _ptr(probs, ctypes.c_double),
                                   int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_attn_probs_f64 rejected its arguments (status {st})")
    return out, lse, probs


def attn_bwd_ref(q, k, v, dout, causal: bool, sm_scale: float, n_threads: int = 0):
    """Oracle gradients (dq [B,Hq,N,D], dk, dv [B,Hkv,N,D], float64) of the forward above for the
    output gradient ``dout`` [B,Hq,N,D] (bf16).  Scores and probabilities are recomputed from the
    definition (the pages' backward by recompute), written out densely."""
    lib = _load()
    qb, kb, vb, gb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v), _bf16_bits(dout)
    B, Hq, Hkv, N, D = _shapes(qb, kb, vb)
    if gb.shape != qb.shape:
        raise ValueError("dout must have q's shape")
    dq = np.zeros((B, Hq, N, D), dtype=np.float64)
    dk = np.zeros((B, Hkv, N, D), dtype=np.float64)
    dv = np.zeros((B, Hkv, N, D), dtype=np.float64)
    st = lib.oracle_attn_bwd_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                 _ptr(vb, ctypes.c_uint16), _ptr(gb, ctypes.c_uint16), B, Hq, Hkv,
                                 N, D, int(bool(causal)), float(sm_scale),
                                 _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                 _ptr(dv, ctypes.c_double), int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_attn_bwd_f64 rejected its arguments (status {st})")
    return dq, dk, dv


def _f64(x) -> np.ndarray:
    """float64 C-contiguous copy of a torch tensor (any float dtype) or a numpy array."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    return np.ascontiguousarray(x.detach().cpu().double().numpy())


def mla_decode_ref(q, kv, d_c: int, sm_scale: float, n_threads: int = 0):
    """Absorbed MLA decode oracle (``mla_oracle.c``), float64.

    ``q`` [B, H, d_c + d_r] holds q_abs (the query with W_uk folded in) then q_pe; ``kv``
    [B, T, d_c + d_r] holds c_kv then k_pe.  Returns out_c [B, H, d_c] (compressed space) and
    LSE [B, H].  Any float dtype; bf16 inputs are widened exactly."""
    lib = _load()
    qd, kvd = _f64(q), _f64(kv)
    if qd.ndim != 3 or kvd.ndim != 3 or qd.shape[0] != kvd.shape[0] or qd.shape[2] != kvd.shape[2]:
        raise ValueError(f"q must be [B,H,dq] and kv [B,T,dq]: {qd.shape} {kvd.shape}")
    B, H, dq = qd.shape
    T = kvd.shape[1]
    d_r = dq - d_c
    out = np.zeros((B, H, d_c), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    st = lib.oracle_mla_decode_f64(_ptr(qd, ctypes.c_double), _ptr(kvd, ctypes.c_double), B, H, T,
                                   d_c, d_r, float(sm_scale), _ptr(out, ctypes.c_double),
                                   _ptr(lse, ctypes.c_double), int(n_threads))
    if st != 0:
        raise ValueError(f"oracle_mla_decode_f64 rejected its arguments (status {st})")
    return out, lse
