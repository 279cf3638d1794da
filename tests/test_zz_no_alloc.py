"""The allocation-free split-KV entry point (attn_fwd_splitkv_noalloc), through the C ABI.

It exists for callers that may not allocate device memory when they call the library (a plug-in
whose host application owns the device-memory budget, a serving loop that forbids allocation
after start-up): the split partials live in a fixed buffer compiled into the library instead of
a caller workspace.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL = 2e-2
O_RTOL = 2e-2
LSE_ATOL = 1e-3


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _inputs(w):
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    out = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    return q, k, v, out, lse


def _close(o_new, l_new, o_ref, l_ref):
    o_new, o_ref = o_new.float().cpu().numpy(), o_ref.float().cpu().numpy()
    bad = np.abs(o_new - o_ref) > O_ATOL + O_RTOL * np.abs(o_ref)
    assert not bad.any(), f"{int(bad.sum())} O elements differ beyond tolerance"
    assert (l_new - l_ref).abs().max().item() <= LSE_ATOL


def _noalloc(lib, w, splits, q, k, v, out, lse):
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                        lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.D, int(w.causal),
                                        ctypes.c_float(w.sm_scale), splits, _stream())


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(cuda_lib):
    lib = cuda_lib
    cases = [(wl.FEWHEADS, 4), (wl.random_case(2, 4, 2, 700, 128, True, 21), 3)]
    for w, splits in cases:  # two calls in a row, different problems, the same shared buffer
        q, k, v, out_ref, lse_ref = _inputs(w)
        need = lib.attn_fwd_splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, splits)
        assert 0 < need <= lib.attn_fwd_splitkv_noalloc_max_bytes()
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        st = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out_ref.data_ptr(),
                                  lse_ref.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.D, int(w.causal),
                                  ctypes.c_float(w.sm_scale), splits, ws.data_ptr(), need,
                                  _stream())
        assert st == 0
        out = torch.full_like(out_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _noalloc(lib, w, splits, q, k, v, out, lse) == 0
        torch.cuda.synchronize()
        assert lib.attn_debug_status(_stream()) == 0
        _close(out, lse, out_ref, lse_ref)


def test_noalloc_matches_the_oracle(cuda_lib):
    """Not only the workspace entry point: the fp64 oracle, on a causal ragged case."""
    lib = cuda_lib
    w = wl.random_case(1, 4, 2, 1100, 128, True, 22)
    q, k, v, out, lse = _inputs(w)
    assert _noalloc(lib, w, 4, q, k, v, out, lse) == 0
    torch.cuda.synchronize()
    assert lib.attn_debug_status(_stream()) == 0
    o_ref, l_ref = oracle.attn_ref(q.cpu(), k.cpu(), v.cpu(), w.causal, w.sm_scale)
    o = out.float().cpu().numpy().astype(np.float64)
    assert not (np.abs(o - o_ref) > O_ATOL + O_RTOL * np.abs(o_ref)).any()
    assert np.abs(lse.cpu().numpy().astype(np.float64) - l_ref).max() <= LSE_ATOL


def test_noalloc_allocates_nothing(cuda_lib):
    """Free device memory (driver view) and torch's allocator are unchanged across calls."""
    lib = cuda_lib
    w = wl.FEWHEADS
    q, k, v, out, lse = _inputs(w)
    assert _noalloc(lib, w, 4, q, k, v, out, lse) == 0  # first call: the buffer's address lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch0 = torch.cuda.memory_allocated()
    for splits in (4, 2, 0):
        assert _noalloc(lib, w, splits, q, k, v, out, lse) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_allocated() == torch0
    assert lib.attn_debug_status(_stream()) == 0


def test_noalloc_rejects_problems_beyond_its_buffer(cuda_lib):
    lib = cuda_lib
    B, Hq, Hkv, N, D, splits = 1, 64, 8, 4096, 128, 4
    assert lib.attn_fwd_splitkv_workspace_bytes(B, Hq, N, D, splits) > \
        lib.attn_fwd_splitkv_noalloc_max_bytes()
    gap = 1 << 30  # distinct, aligned addresses; rejected before any of them is touched
    st = lib.attn_fwd_splitkv_noalloc(gap, 2 * gap, 3 * gap, 4 * gap, 5 * gap, B, Hq, Hkv, N, D,
                                      1, ctypes.c_float(D ** -0.5), splits, _stream())
    assert st == -14  # ATTN_ERR_SCRATCH


def test_noalloc_default_split_count_fits_its_buffer(cuda_lib):
    """num_splits = 0: the default is the best split count whose partials fit the buffer, so it
    never runs out of it, also where attn_fwd_splitkv's own default would need more."""
    lib = cuda_lib
    cap = lib.attn_fwd_splitkv_noalloc_max_bytes()
    over = [(B, Hq, N, D) for B in (1, 2) for Hq in (1, 2, 4) for N in (32768, 65536)
            for D in (64, 128) if lib.attn_fwd_splitkv_workspace_bytes(B, Hq, N, D, 0) > cap]
    cases = [wl.random_case(1, 4, 1, 8192, 128, True, 23), wl.random_case(1, 8, 2, 8192, 64, True, 24)]
    if over:  # a shape whose unlimited default exceeds the buffer, when the sweep finds one
        B, Hq, N, D = over[0]
        cases.append(wl.random_case(B, Hq, 1, N, D, False, 25))
    for w in cases:
        q, k, v, out, lse = _inputs(w)
        assert _noalloc(lib, w, 0, q, k, v, out, lse) == 0
        torch.cuda.synchronize()
        assert lib.attn_debug_status(_stream()) == 0
        ref = torch.empty_like(out)
        ref_l = torch.empty_like(lse)
        assert lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ref.data_ptr(),
                            ref_l.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.D, int(w.causal),
                            ctypes.c_float(w.sm_scale), _stream()) == 0
        torch.cuda.synchronize()
        _close(out, lse, ref, ref_l)
