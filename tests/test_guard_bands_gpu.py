"""Guard bands: no entry point writes outside the memory it was given.

Every output (and every caller-provided workspace) is carved out of a larger byte buffer filled
with the pattern 0xA5; after the call, the bytes before and after it, and the padding columns of
strided outputs, must still hold the pattern, while the outputs themselves match the oracle.
This stands in for a memory checker on outputs (ragged N, where the stores must clip at N; head
dimensions below the padded width, where the columns past D must not be written; split
workspaces sized exactly to the entry point's own figure).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu

PAD = 4096  # guard bytes on each side (keeps every carved-out pointer 16-byte aligned)
PATTERN = 0xA5


class Guarded:
    """`nbytes` usable bytes inside a buffer whose PAD bytes on either side hold PATTERN."""

    def __init__(self, nbytes):
        self.nbytes = nbytes
        self.buf = torch.full((nbytes + 2 * PAD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.inner = self.buf[PAD:PAD + nbytes]

    def typed(self, dtype, shape):
        return self.inner.view(dtype).view(shape)

    def intact(self):
        return bool((self.buf[:PAD] == PATTERN).all()) and \
            bool((self.buf[PAD + self.nbytes:] == PATTERN).all())


def _outputs(w):
    go = Guarded(w.B * w.Hq * w.N * w.D * 2)
    gl = Guarded(w.B * w.Hq * w.N * 4)
    return go, gl, go.typed(torch.bfloat16, (w.B, w.Hq, w.N, w.D)), \
        gl.typed(torch.float32, (w.B, w.Hq, w.N))


@pytest.mark.parametrize("w", [wl.random_case(1, 4, 2, 300, 256, True, 61),
                               wl.random_case(2, 2, 1, 200, 192, False, 62),
                               wl.random_case(1, 4, 2, 333, 96, True, 63)],
                         ids=["d256-n300", "d192-n200", "d96-n333"])
def test_forward_other_head_dims(w, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    q, k, v = wl.make_qkv(w)
    go, gl, out, lse = _outputs(w)
    attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, sm_scale=w.sm_scale, out=out,
                  lse=lse)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert go.intact() and gl.intact()
    _check(out, lse, *oracle.attn_ref(q, k, v, w.causal, w.sm_scale), w.name)


@pytest.mark.parametrize("w,splits", [(wl.random_case(2, 4, 2, 700, 128, True, 64), 3),
                                      (wl.random_case(1, 2, 1, 1000, 96, False, 65), 4),
                                      (wl.random_case(1, 3, 3, 259, 64, True, 66), 2)],
                         ids=["d128-n700-s3", "d96-n1000-s4", "d64-n259-s2"])
def test_splitkv_outputs_and_workspace(w, splits, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    q, k, v = wl.make_qkv(w)
    go, gl, out, lse = _outputs(w)
    need = attn.splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, splits)
    assert need > 0
    gw = Guarded(need)
    attn.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, sm_scale=w.sm_scale,
                          num_splits=splits, workspace=gw.inner, out=out, lse=lse)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert go.intact() and gl.intact() and gw.intact()
    _check(out, lse, *oracle.attn_ref(q, k, v, w.causal, w.sm_scale), w.name)


@pytest.mark.parametrize("w", [wl.random_case(1, 4, 2, 300, 128, True, 67),
                               wl.random_case(2, 2, 2, 129, 96, False, 68),
                               wl.random_case(1, 2, 1, 200, 256, True, 69)],
                         ids=["d128-n300", "d96-n129", "d256-n200"])
def test_strided_padded_rows_keep_their_padding(w, cuda_lib):
    """Output rows of D + 8 elements: the 8 padding elements of every row stay untouched."""
    import exact_attention_forward_attn_gb300 as attn

    q, k, v = wl.make_qkv(w)
    row = w.D + 8
    g = Guarded(w.B * w.Hq * w.N * row * 2)
    full = g.typed(torch.bfloat16, (w.B, w.Hq, w.N, row))
    out = full[..., :w.D]
    assert not out.is_contiguous()
    gl = Guarded(w.B * w.Hq * w.N * 4)
    lse = gl.typed(torch.float32, (w.B, w.Hq, w.N))
    attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, sm_scale=w.sm_scale, out=out,
                  lse=lse)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert g.intact() and gl.intact()
    pad_bytes = full[..., w.D:].contiguous().view(torch.uint8)
    assert bool((pad_bytes == PATTERN).all()), "padding columns of the output were written"
    _check(out.contiguous(), lse, *oracle.attn_ref(q, k, v, w.causal, w.sm_scale), w.name)


@pytest.mark.parametrize("w", [wl.random_case(1, 4, 2, 300, 128, True, 70),
                               wl.random_case(2, 2, 1, 200, 96, False, 71)],
                         ids=["d128-n300-causal", "d96-n200"])
def test_backward_gradients_and_workspace(w, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn
    from exact_attention_forward_attn_gb300 import _lib

    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
    gen = torch.Generator().manual_seed(72)
    do = torch.randn(q.shape, generator=gen).to(torch.bfloat16)
    gq = Guarded(q.numel() * 2)
    gk = Guarded(k.numel() * 2)
    gv = Guarded(v.numel() * 2)
    need = int(_lib.load().attn_bwd_workspace_bytes(w.B, w.Hq, w.N))
    gw = Guarded(need)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, out, lse, do.cuda(), causal=w.causal,
                               sm_scale=w.sm_scale, dq=gq.typed(torch.bfloat16, q.shape),
                               dk=gk.typed(torch.bfloat16, k.shape),
                               dv=gv.typed(torch.bfloat16, v.shape), workspace=gw.inner)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert gq.intact() and gk.intact() and gv.intact() and gw.intact()
    rq, rk, rv = oracle.attn_bwd_ref(q, k, v, do, w.causal, w.sm_scale)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        gg = g.float().cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(gg - r) / np.linalg.norm(r)
        assert rel <= 1e-2, f"{name}: relative L2 error {rel:.2e}"


@pytest.mark.parametrize("B,T,splits", [(2, 777, 3), (1, 4096, 8)],
                         ids=["ragged-cluster-merge", "t4096-merge-kernel"])
def test_mla_decode_outputs_and_workspace(B, T, splits, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    w = wl.MlaWorkload(f"mla-guard-b{B}-t{T}", B, 128, T, 73)
    q, kv = wl.make_mla(w, device="cuda")
    go = Guarded(B * w.H * attn.MLA_D_C * 2)
    gl = Guarded(B * w.H * 4)
    need = attn.mla_decode_workspace_bytes(B, w.H, T, splits)
    assert (need > 0) == (splits > 4)
    gw = Guarded(max(need, 16))
    out, lse = attn.mla_decode(q, kv, w.sm_scale, num_splits=splits,
                               workspace=gw.inner if need > 0 else None,
                               out=go.typed(torch.bfloat16, (B, w.H, attn.MLA_D_C)),
                               lse=gl.typed(torch.float32, (B, w.H)))
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert go.intact() and gl.intact() and gw.intact()
    ref_o, ref_l = oracle.mla_decode_ref(q.cpu(), kv.cpu(), attn.MLA_D_C, w.sm_scale)
    o = out.float().cpu().numpy()
    assert not (np.abs(o - ref_o) > 2e-2 + 2e-2 * np.abs(ref_o)).any()
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_l).max() <= 1e-3


def test_splitkv_rejects_a_workspace_one_byte_short(cuda_lib):
    """The workspace figure is exact: one byte less is refused before anything is written."""
    from exact_attention_forward_attn_gb300 import _lib

    lib = _lib.load()
    w = wl.random_case(1, 2, 1, 1000, 128, False, 74)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    go, gl, out, lse = _outputs(w)
    need = lib.attn_fwd_splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, 4)
    gw = Guarded(need)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.D, 0,
                              ctypes.c_float(w.sm_scale), 4, gw.inner.data_ptr(), need - 1, stream)
    assert st == -13  # ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert go.intact() and gl.intact() and gw.intact()
    assert bool((go.inner == PATTERN).all()) and bool((gw.inner == PATTERN).all())
