"""Failure detection on the GPU without a fault: a test hook withholds one K/V tile, the kernel's
bounded waits expire (about one second), and the host reads ATTN_ERR_TIMEOUT from the device
status word; the CUDA context stays usable for the next, correct call."""
import ctypes
import time

import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives(cuda_lib):
    lib = cuda_lib
    w = wl.TINY_NONCAUSAL  # 2 CTAs, one K/V tile: item 1 is V tile 0
    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.zeros_like(qd)
    lse = torch.zeros(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_debug_status(stream) == 0  # clear any earlier state
    t0 = time.time()
    st = lib.attn_fwd_test_stall(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                                 lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.D, 0,
                                 ctypes.c_float(w.sm_scale), 1, stream)
    assert st == 0
    assert lib.attn_debug_status(stream) == -9  # ATTN_ERR_TIMEOUT, read by the host
    elapsed = time.time() - t0
    assert 0.5 < elapsed < 30.0, elapsed
    assert lib.attn_debug_status(stream) == 0  # the word was cleared
    # the context is still usable: an ordinary call succeeds and is correct
    import exact_attention_forward_attn_gb300 as attn

    o2, l2 = attn.attn_fwd(qd, kd, vd, causal=False, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    o_ref, l_ref = oracle.attn_ref(q, k, v, False, w.sm_scale)
    _check(o2, l2, o_ref, l_ref, "after an expired wait")


def test_stall_item_past_the_end_stalls_nothing(cuda_lib):
    lib = cuda_lib
    w = wl.TINY_CAUSAL
    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty_like(qd)
    lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.attn_fwd_test_stall(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                                 lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.D, 1,
                                 ctypes.c_float(w.sm_scale), 1000, stream)
    assert st == 0
    assert lib.attn_debug_status(stream) == 0
    o_ref, l_ref = oracle.attn_ref(q, k, v, True, w.sm_scale)
    _check(out, lse, o_ref, l_ref, "stall item beyond the ring")


def test_mla_expired_wait_skips_the_cluster_merge(cuda_lib):
    """MLA decode with two splits merged inside a cluster: the CTAs of split 1 are starved of one
    cache tile and time out.  Their clusters must then skip the merge (out and lse keep their
    zeros), the expiry must reach the host, and 70 further launches must all merge correctly."""
    import exact_attention_forward_attn_gb300 as attn
    from test_mla_gpu import _check as mla_check

    lib = cuda_lib
    w = wl.MlaWorkload("mla-stall", 1, 16, 256, 98)  # 4 token tiles: split 1 holds tiles 2-3
    q, kv = wl.make_mla(w, device="cuda")
    splits = 2
    need = attn.mla_decode_workspace_bytes(w.B, w.H, w.T, splits)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.zeros(w.B, w.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(w.B, w.H, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_debug_status(stream) == 0
    st = lib.attn_mla_decode_test_stall(q.data_ptr(), kv.data_ptr(), out.data_ptr(),
                                        lse.data_ptr(), w.B, w.H, w.T, 512, 64,
                                        ctypes.c_float(w.sm_scale), splits, ws.data_ptr(), need,
                                        3, stream)
    assert st == 0
    assert lib.attn_debug_status(stream) == -9  # ATTN_ERR_TIMEOUT
    assert lib.attn_debug_status(stream) == 0
    assert torch.all(out == 0) and torch.all(lse == 0)
    runs = [attn.mla_decode(q, kv, w.sm_scale, num_splits=splits) for _ in range(70)]
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    for o, l in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
    mla_check(runs[-1][0], runs[-1][1], q, kv, w.sm_scale)
