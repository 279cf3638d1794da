"""The index-checking debug build (libgb300attn_debug.so, compiled with ATTN_DEBUG).

Its kernels check, before every store whose address they compute, that the indices behind it are
in range, and record a failed check in the device status word (attn_debug_status returns
ATTN_ERR_RANGE) instead of storing; nothing traps.  With compute-sanitizer unavailable it stands
in for a memory checker.  Here every entry point runs once under it (one-CTA and CTA-pair
forward, ragged N, strided, split-KV with its merge, wide heads, backward, MLA decode with the
cluster merge and with the merge kernel); each must report no failed check and match the oracle.
(The whole suite can also run on this build: ATTN_DEBUG_LIB=1 pytest -m gpu.)
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import build, _lib
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg(cuda_lib):
    return _lib.load(build.build(debug=True))


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _fwd_args(w, q, k, v, out, lse):
    return (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), w.B, w.Hq,
            w.Hkv, w.N, w.D, int(w.causal), ctypes.c_float(w.sm_scale))


def _outputs(w):
    return (torch.empty(w.B, w.Hq, w.N, w.D, dtype=torch.bfloat16, device="cuda"),
            torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda"))


CASES = [wl.random_case(2, 4, 2, 300, 128, True, 81), wl.random_case(1, 6, 3, 383, 64, False, 82),
         wl.random_case(1, 4, 1, 200, 256, True, 83), wl.random_case(1, 2, 2, 129, 96, True, 84),
         wl.GQA4_CAUSAL]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_under_index_checks(w, dbg):
    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = _outputs(w)
    assert dbg.attn_fwd(*_fwd_args(w, qd, kd, vd, out, lse), _stream()) == 0
    assert dbg.attn_debug_status(_stream()) == 0
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out, lse, o_ref, l_ref, w.name)
    if 64 < w.D <= 128:  # the CTA-pair kernel too
        out2, lse2 = _outputs(w)
        assert dbg.attn_fwd_test_kernel(*_fwd_args(w, qd, kd, vd, out2, lse2), 2, -1,
                                        _stream()) == 0
        assert dbg.attn_debug_status(_stream()) == 0
        _check(out2, lse2, o_ref, l_ref, f"pair {w.name}")
    if w.D <= 128:  # split-KV partials and the merge kernel
        out3, lse3 = _outputs(w)
        need = dbg.attn_fwd_splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, 3)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        assert dbg.attn_fwd_splitkv(*_fwd_args(w, qd, kd, vd, out3, lse3), 3, ws.data_ptr(),
                                    need, _stream()) == 0
        assert dbg.attn_debug_status(_stream()) == 0
        _check(out3, lse3, o_ref, l_ref, f"split {w.name}")


def test_strided_and_backward_under_index_checks(dbg):
    w = wl.random_case(2, 4, 2, 257, 128, True, 85)
    q, k, v = wl.make_qkv(w)
    # [B, N, H, D] memory seen as [B, H, N, D]
    qs, ks, vs = (t.cuda().transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v))
    out = torch.empty(w.B, w.N, w.Hq, w.D, dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    strides = [(ctypes.c_longlong * 3)(t.stride(0), t.stride(1), t.stride(2))
               for t in (qs, ks, vs, out)]
    assert dbg.attn_fwd_strided(*_fwd_args(w, qs, ks, vs, out, lse),
                                *[ctypes.cast(a, ctypes.c_void_p) for a in strides],
                                _stream()) == 0
    assert dbg.attn_debug_status(_stream()) == 0
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out.contiguous(), lse, o_ref, l_ref, "strided")
    # backward on the contiguous layout
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o2, l2 = _outputs(w)
    assert dbg.attn_fwd(*_fwd_args(w, qd, kd, vd, o2, l2), _stream()) == 0
    gen = torch.Generator().manual_seed(86)
    do = torch.randn(q.shape, generator=gen).to(torch.bfloat16)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    need = int(dbg.attn_bwd_workspace_bytes(w.B, w.Hq, w.N))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert dbg.attn_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o2.data_ptr(), l2.data_ptr(),
                        do.cuda().data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B,
                        w.Hq, w.Hkv, w.N, w.D, 1, ctypes.c_float(w.sm_scale), ws.data_ptr(), need,
                        _stream()) == 0
    assert dbg.attn_debug_status(_stream()) == 0
    rq, rk, rv = oracle.attn_bwd_ref(q, k, v, do, True, w.sm_scale)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        gg = g.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(gg - r) / np.linalg.norm(r) <= 1e-2, name


@pytest.mark.parametrize("T,splits", [(777, 3), (4096, 8)], ids=["cluster-merge", "merge-kernel"])
def test_mla_decode_under_index_checks(T, splits, dbg):
    w = wl.MlaWorkload(f"mla-dbg-t{T}", 2, 128, T, 87)
    q, kv = wl.make_mla(w, device="cuda")
    out = torch.empty(w.B, w.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.B, w.H, dtype=torch.float32, device="cuda")
    need = dbg.attn_mla_decode_workspace_bytes(w.B, w.H, w.T, splits)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    assert dbg.attn_mla_decode(q.data_ptr(), kv.data_ptr(), out.data_ptr(), lse.data_ptr(), w.B,
                               w.H, w.T, 512, 64, ctypes.c_float(w.sm_scale), splits,
                               ws.data_ptr(), need, _stream()) == 0
    assert dbg.attn_debug_status(_stream()) == 0
    ref_o, ref_l = oracle.mla_decode_ref(q.cpu(), kv.cpu(), 512, w.sm_scale)
    o = out.float().cpu().numpy()
    assert not (np.abs(o - ref_o) > 2e-2 + 2e-2 * np.abs(ref_o)).any()
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_l).max() <= 1e-3
