"""GB300 (sm_103a) fused exact-attention forward.

``attn_fwd(q, k, v, causal=False, sm_scale=None)`` returns ``(out, lse)`` for
q [B,Hq,N,D] and k, v [B,Hkv,N,D] (bf16, CUDA, contiguous): out = softmax(sm_scale QK^T
[+ causal mask]) V in bf16 and the natural-log LSE of each row in fp32.  All arithmetic runs in
the hand-written CUDA kernels behind the C ABI (``include/attn.h``); this module only allocates
outputs with PyTorch and marshals pointers, sizes and the current stream.
"""
from __future__ import annotations

import ctypes
import math

from . import _lib

ATTN_OK = 0
STATUS_NAMES = {
    0: "ATTN_OK", -1: "ATTN_ERR_NULL", -2: "ATTN_ERR_SHAPE", -3: "ATTN_ERR_HEADS",
    -4: "ATTN_ERR_HEADDIM", -5: "ATTN_ERR_ALIGN", -6: "ATTN_ERR_SCALE", -7: "ATTN_ERR_ARCH",
    -8: "ATTN_ERR_CUDA", -9: "ATTN_ERR_TIMEOUT", -10: "ATTN_ERR_MEMORY", -11: "ATTN_ERR_ALIAS",
    -12: "ATTN_ERR_SPLITS", -13: "ATTN_ERR_WORKSPACE", -14: "ATTN_ERR_SCRATCH",
    -15: "ATTN_ERR_STRIDE",
}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str = "attn_fwd"):
        lib = _lib.load()
        msg = lib.attn_status_string(status).decode()
        extra = ""
        if status == -8:
            extra = f" (cudaError {lib.attn_last_cuda_error()})"
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}{extra}")
        self.status = status


def _stream_handle(device):
    import torch

    return torch.cuda.current_stream(device).cuda_stream


def _check_inputs(q, k, v, allow_strided=False):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise ValueError(f"{name} must be a 4-D torch tensor [B, H, N, D]")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bf16, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if allow_strided:
            if t.stride(-1) != 1:
                raise ValueError(f"{name}: the D axis must be contiguous (stride 1)")
        elif not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous ([B, H, N, D] row-major); call "
                             ".contiguous() first")
    B, Hq, N, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != D:
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on the same device")
    return B, Hq, k.shape[1], N, D


def _outputs(q, out, lse, allow_strided=False):
    import torch

    B, Hq, N, _ = q.shape
    if out is None:
        out = torch.empty_like(q)  # keeps q's layout when q is dense
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    ok_layout = out.stride(-1) == 1 if allow_strided else out.is_contiguous()
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not ok_layout:
        raise ValueError("out must be a bf16 tensor shaped like q (contiguous, or with a "
                         "contiguous D axis for strided inputs)")
    if lse.shape != (B, Hq, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, Hq, N]")
    return out, lse


def attn_fwd(q, k, v, causal: bool = False, sm_scale: float | None = None, out=None, lse=None):
    """Fused attention forward on the current CUDA stream of ``q``'s device.

    Returns ``(out, lse)``: out bf16 [B,Hq,N,D], lse fp32 [B,Hq,N].  ``out``/``lse`` may be passed
    preallocated (right shape and dtype).  q, k, v, out may be strided views (e.g. [B, N, H, D]
    memory seen as [B, H, N, D]) as long as D is contiguous and the other strides are multiples of
    8 elements; those go through ``attn_fwd_strided`` without a copy.  Problems whose query tiles
    leave SMs idle over a long key axis may be split along the keys by the library itself
    (``fwd_num_splits`` says how many ways; the result equals the single pass up to rounding).
    Raises ``AttnError`` on a nonzero status.
    """
    import torch

    B, Hq, Hkv, N, D = _check_inputs(q, k, v, allow_strided=True)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    out, lse = _outputs(q, out, lse, allow_strided=True)
    lib = _lib.load()
    with torch.cuda.device(q.device):
        if all(t.is_contiguous() for t in (q, k, v, out)):
            st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, Hq, Hkv, N, D, int(bool(causal)),
                              float(sm_scale), _stream_handle(q.device))
        else:
            arrs = [(ctypes.c_longlong * 3)(t.stride(0), t.stride(1), t.stride(2))
                    for t in (q, k, v, out)]
            st = lib.attn_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      lse.data_ptr(), B, Hq, Hkv, N, D, int(bool(causal)),
                                      float(sm_scale), *[ctypes.cast(a, ctypes.c_void_p)
                                                         for a in arrs],
                                      _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st)
    return out, lse


def fwd_num_splits(B: int, Hq: int, N: int, D: int, causal: bool = False) -> int:
    """Key-axis splits ``attn_fwd`` itself uses for these sizes on the current device (1: single
    pass; more: the splits of each work item merge inside a thread-block cluster)."""
    return int(_lib.load().attn_fwd_num_splits(B, Hq, N, D, int(bool(causal))))


def splitkv_num_splits(B: int, Hq: int, N: int, D: int, causal: bool = False) -> int:
    """Split count the library suggests for these sizes on the current device."""
    return int(_lib.load().attn_fwd_splitkv_num_splits(B, Hq, N, D, int(bool(causal))))


def splitkv_workspace_bytes(B: int, Hq: int, N: int, D: int, num_splits: int = 0) -> int:
    """Workspace bytes ``attn_fwd_splitkv`` needs (0 when the call resolves to one split)."""
    return int(_lib.load().attn_fwd_splitkv_workspace_bytes(B, Hq, N, D, int(num_splits)))


def attn_fwd_splitkv(q, k, v, causal: bool = False, sm_scale: float | None = None,
                     num_splits: int = 0, workspace=None, out=None, lse=None):
    """Split-KV forward (partials over key-axis splits + merge); same result as ``attn_fwd`` up
    to rounding.  ``workspace``: optional CUDA tensor of at least ``splitkv_workspace_bytes(...)``
    bytes (allocated here when omitted; left untouched when 2-4 splits merge inside clusters).
    ``num_splits=1`` runs the single pass."""
    import torch

    B, Hq, Hkv, N, D = _check_inputs(q, k, v)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    out, lse = _outputs(q, out, lse)
    lib = _lib.load()
    with torch.cuda.device(q.device):
        need = splitkv_workspace_bytes(B, Hq, N, D, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        st = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, Hq, Hkv, N, D, int(bool(causal)),
                                  float(sm_scale), int(num_splits), ws_ptr, ws_bytes,
                                  _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv")
    return out, lse


MLA_D_C = 512
MLA_D_R = 64


def mla_decode_num_splits(B: int, H: int, T: int) -> int:
    """Token-axis splits ``mla_decode`` picks by default."""
    return int(_lib.load().attn_mla_decode_num_splits(B, H, T))


def mla_decode_workspace_bytes(B: int, H: int, T: int, num_splits: int = 0) -> int:
    return int(_lib.load().attn_mla_decode_workspace_bytes(B, H, T, num_splits))


def mla_decode(q, kv, sm_scale: float, num_splits: int = 0, workspace=None, out=None, lse=None):
    """Absorbed MLA decode: q [B, H, 576] (q_abs | q_pe), kv [B, T, 576] (c_kv | k_pe), bf16 CUDA
    tensors.  Returns out_c [B, H, 512] (bf16, compressed space) and LSE [B, H] (fp32).
    ``sm_scale`` is the un-absorbed one, 1/sqrt(d_nope + d_r)."""
    import torch

    for t in (q, kv):
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
            raise TypeError("q and kv must be CUDA tensors")
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 3:
            raise ValueError("q and kv must be contiguous 3-D bf16 tensors")
    if q.device != kv.device:
        raise ValueError("q and kv must be on the same device")
    B, H, dq = q.shape
    if kv.shape[0] != B or kv.shape[2] != dq:
        raise ValueError(f"kv must be [B, T, {dq}], got {tuple(kv.shape)}")
    T = kv.shape[1]
    if out is None:
        out = torch.empty(B, H, MLA_D_C, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    lib = _lib.load()
    with torch.cuda.device(q.device):
        need = mla_decode_workspace_bytes(B, H, T, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        st = lib.attn_mla_decode(q.data_ptr(), kv.data_ptr(), out.data_ptr(), lse.data_ptr(), B,
                                 H, T, MLA_D_C, dq - MLA_D_C, float(sm_scale), int(num_splits),
                                 ws_ptr, ws_bytes, _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_mla_decode")
    return out, lse


def attn_bwd(q, k, v, out, lse, dout, causal: bool = False, sm_scale: float | None = None,
             dq=None, dk=None, dv=None, workspace=None):
    """Gradients (dq, dk, dv) of ``attn_fwd`` by recompute from its ``out`` and ``lse``, for the
    output gradient ``dout`` (all contiguous CUDA tensors; dq like q, dk/dv like k)."""
    import torch

    B, Hq, Hkv, N, D = _check_inputs(q, k, v)
    for name, t, like in (("out", out, q), ("dout", dout, q)):
        if t.shape != like.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, Hq, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, Hq, N]")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    lib = _lib.load()
    with torch.cuda.device(q.device):
        need = int(lib.attn_bwd_workspace_bytes(B, Hq, N))
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                          dv.data_ptr(), B, Hq, Hkv, N, D, int(bool(causal)), float(sm_scale),
                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def _autograd_function():
    import torch

    class FlashAttention(torch.autograd.Function):
        """``FlashAttention.apply(q, k, v, is_causal=False)``: the pages' autograd interface
        ("Flash Attention 与 Kernel 优化": inputs already projected, [.., N, D] per head), here
        for q [B,Hq,N,D] and k, v [B,Hkv,N,D]; forward and backward both run the CUDA kernels,
        and the forward saves q, k, v, O and LSE for the backward's recompute."""

        @staticmethod
        def forward(ctx, q, k, v, is_causal=False, sm_scale=None):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            out, lse = attn_fwd(q, k, v, causal=is_causal, sm_scale=sm_scale)
            ctx.save_for_backward(q, k, v, out, lse)
            ctx.is_causal, ctx.sm_scale = is_causal, sm_scale
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            dq, dk, dv = attn_bwd(q, k, v, out, lse, dout.contiguous(), causal=ctx.is_causal,
                                  sm_scale=ctx.sm_scale)
            return dq, dk, dv, None, None

    return FlashAttention


def __getattr__(name):
    if name == "FlashAttention":
        fn = _autograd_function()
        globals()["FlashAttention"] = fn
        return fn
    raise AttributeError(name)


def device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status word:
    0 if no kernel recorded a failure, else a negative status (e.g. -9 for an expired wait)."""
    import torch

    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        return int(_lib.load().attn_debug_status(_stream_handle(dev)))
