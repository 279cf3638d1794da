"""Key-axis splits merged inside thread-block clusters, on the GPU.

attn_fwd itself splits the key axis of problems whose query tiles leave most SMs idle (few heads,
long sequences): the splits of each pair of Q tiles run as one cluster and merge their partial
results through distributed shared memory, with no workspace (the split-T merge of "Attention
Kernel 实现与正确性验证", section 2.4).  attn_fwd_splitkv takes the same path when all of its
clusters fit on the device at once, and otherwise its workspace and merge kernel.  Every result
is compared with the fp64 oracle.
"""
import ctypes
import time

import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_guard_bands_gpu import PATTERN, Guarded
from test_parity_gpu import _check

pytestmark = pytest.mark.gpu

# few query tiles, many key tiles: attn_fwd splits these on a GB300 (152 SMs)
AUTO = [wl.FEWHEADS,
        wl.random_case(1, 1, 1, 8192, 64, False, 81),
        wl.random_case(1, 2, 1, 3000, 128, True, 82),
        wl.random_case(2, 1, 1, 2500, 96, False, 83)]


def _sampled(w, q, k, v, out, lse, per_head=32):
    rows = wl.sample_rows(w, min(per_head, w.N))
    rows[..., 0] = 0
    rows[..., -1] = w.N - 1
    rows = rows.sort(dim=-1).values
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale, rows=rows.numpy())
    idx = rows.long()
    o_c, l_c = out.cpu(), lse.cpu()
    o_s = torch.stack([o_c[b, h][idx[b, h]] for b in range(w.B) for h in range(w.Hq)])
    l_s = torch.stack([l_c[b, h][idx[b, h]] for b in range(w.B) for h in range(w.Hq)])
    _check(o_s.reshape(o_ref.shape), l_s.reshape(l_ref.shape), o_ref, l_ref, w.name)


@pytest.mark.parametrize("w", AUTO, ids=[w.name for w in AUTO])
def test_attn_fwd_splits_low_occupancy_problems(w, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    n = attn.fwd_num_splits(w.B, w.Hq, w.N, w.D, w.causal)
    assert n >= 2, n
    q, k, v = wl.make_qkv(w)
    out, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(out, lse, *oracle.attn_ref(q, k, v, w.causal, w.sm_scale), f"{w.name} auto-split {n}")


def test_attn_fwd_split_is_the_cluster_path_of_splitkv(cuda_lib):
    """attn_fwd's split and attn_fwd_splitkv with the same count run the same launch: the same
    bits, and the split-KV workspace is left untouched (its bytes keep their guard pattern)."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.FEWHEADS
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    n = attn.fwd_num_splits(w.B, w.Hq, w.N, w.D, w.causal)
    assert n > 1
    o1, l1 = attn.attn_fwd(q, k, v, causal=w.causal, sm_scale=w.sm_scale)
    gw = Guarded(attn.splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, n))
    o2, l2 = attn.attn_fwd_splitkv(q, k, v, causal=w.causal, sm_scale=w.sm_scale, num_splits=n,
                                   workspace=gw.inner)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert gw.intact() and bool((gw.inner == PATTERN).all())
    # one split is the single pass: close to the split result, not necessarily the same bits
    o3, l3 = attn.attn_fwd_splitkv(q, k, v, causal=w.causal, sm_scale=w.sm_scale, num_splits=1)
    torch.cuda.synchronize()
    assert (o3.float() - o1.float()).abs().max().item() < 2e-2
    assert (l3 - l1).abs().max().item() < 1e-4


def test_strided_views_split_too(cuda_lib):
    """[B, N, H, D] memory seen as [B, H, N, D] (attn_fwd_strided) on a problem attn_fwd splits."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(1, 2, 1, 4096, 128, True, 84)
    q, k, v = wl.make_qkv(w)
    assert attn.fwd_num_splits(w.B, w.Hq, w.N, w.D, w.causal) > 1
    qs, ks, vs = (t.transpose(1, 2).contiguous().cuda().transpose(1, 2) for t in (q, k, v))
    out = torch.empty(w.B, w.N, w.Hq, w.D, dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    assert not qs.is_contiguous() and not out.is_contiguous()
    o, lse = attn.attn_fwd(qs, ks, vs, causal=w.causal, sm_scale=w.sm_scale, out=out)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(o.contiguous(), lse, *oracle.attn_ref(q, k, v, w.causal, w.sm_scale), w.name)


def test_long_causal_split_sampled_rows(cuda_lib):
    """One head of 16384 causal rows: attn_fwd's cluster split, 32 sampled rows per head."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(1, 1, 1, 16384, 128, True, 85)
    assert attn.fwd_num_splits(w.B, w.Hq, w.N, w.D, w.causal) > 1
    q, k, v = wl.make_qkv(w)
    out, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _sampled(w, q, k, v, out, lse)


@pytest.mark.parametrize("shape", [(1, 4, 1, 8192, 128), (1, 1, 1, 32768, 128), (1, 2, 1, 12000, 64)],
                         ids=["hq4-n8192", "hq1-n32768", "hq2-n12000-d64"])
def test_attn_fwd_workspace_split_on_causal_few_heads(shape, cuda_lib):
    """Causal few-head problems whose pairs are more clusters than fit at once: attn_fwd splits
    them through its own scratch slots (persistent split kernel + merge kernel)."""
    import exact_attention_forward_attn_gb300 as attn

    B, Hq, Hkv, N, D = shape
    w = wl.random_case(B, Hq, Hkv, N, D, True, 92)
    assert attn.fwd_num_splits(B, Hq, N, D, True) >= 2
    q, k, v = wl.make_qkv(w)
    out, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _sampled(w, q, k, v, out, lse)


def test_attn_fwd_scratch_slots_under_concurrent_streams(cuda_lib):
    """Six streams run attn_fwd's workspace split at once, three rounds: the scratch slots are
    leased one launch at a time, so every result equals the same call made alone."""
    import exact_attention_forward_attn_gb300 as attn

    ws_ = [wl.random_case(1, 4, 1, 8192, 128, True, 93 + i) for i in range(6)]
    ins = [tuple(t.cuda() for t in wl.make_qkv(w)) for w in ws_]
    refs = []
    for w, (q, k, v) in zip(ws_, ins):
        refs.append(attn.attn_fwd(q, k, v, causal=True, sm_scale=w.sm_scale))
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in ws_]
    outs = [(torch.empty_like(q), torch.empty(1, w.Hq, w.N, device="cuda"))
            for w, (q, _, _) in zip(ws_, ins)]
    for _ in range(3):
        for o, l in outs:
            o.zero_()
            l.zero_()
        torch.cuda.synchronize()
        for st, w, (q, k, v), (o, l) in zip(streams, ws_, ins, outs):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                attn.attn_fwd(q, k, v, causal=True, sm_scale=w.sm_scale, out=o, lse=l)
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        for (o, l), (ro, rl) in zip(outs, refs):
            assert torch.equal(o, ro) and torch.equal(l, rl)


def test_attn_fwd_under_capture_does_not_use_the_scratch(cuda_lib):
    """While its stream is captured, attn_fwd takes only cluster splits: for four causal heads of
    8192 rows (too many pairs for one wave of clusters) that is the single pass, bit for bit."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(1, 4, 1, 8192, 128, True, 99)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    assert attn.fwd_num_splits(w.B, w.Hq, w.N, w.D, True) >= 2  # outside a capture
    o1, l1 = attn.attn_fwd_splitkv(q, k, v, causal=True, sm_scale=w.sm_scale, num_splits=1)
    out = torch.zeros_like(q)
    lse = torch.zeros(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        attn.attn_fwd(q, k, v, causal=True, sm_scale=w.sm_scale, out=out, lse=lse)
    g.replay()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert torch.equal(out, o1) and torch.equal(lse, l1)


def test_splitkv_default_on_causal_few_heads_uses_the_workspace(cuda_lib):
    """Four causal heads of 8192 rows: the model splits in two; 128 pairs of Q tiles are more
    clusters than fit at once, so the persistent split kernel and the merge kernel run (the
    workspace is written)."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(1, 4, 1, 8192, 128, True, 86)
    n = attn.splitkv_num_splits(w.B, w.Hq, w.N, w.D, True)
    assert n >= 2, n
    q, k, v = wl.make_qkv(w)
    gw = Guarded(attn.splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, 0))
    out, lse = attn.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=True,
                                     sm_scale=w.sm_scale, num_splits=0, workspace=gw.inner)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert gw.intact() and not bool((gw.inner == PATTERN).all())
    _sampled(w, q, k, v, out, lse)


@pytest.mark.parametrize("w,splits", [(wl.random_case(1, 2, 1, 1000, 128, False, 87), 2),
                                      (wl.random_case(1, 3, 1, 1300, 64, True, 88), 3),
                                      (wl.random_case(1, 2, 2, 2000, 128, True, 89), 4),
                                      (wl.random_case(1, 2, 2, 700, 80, False, 90), 4)],
                         ids=["d128-s2", "d64-causal-s3", "d128-causal-s4", "d80-s4"])
def test_splitkv_cluster_path_matches_oracle_and_leaves_workspace(w, splits, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    q, k, v = wl.make_qkv(w)
    gw = Guarded(attn.splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, splits))
    out, lse = attn.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=w.causal,
                                     sm_scale=w.sm_scale, num_splits=splits, workspace=gw.inner)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert bool((gw.buf == PATTERN).all()), "the cluster path wrote into the workspace"
    _check(out, lse, *oracle.attn_ref(q, k, v, w.causal, w.sm_scale), f"{w.name} s={splits}")


def test_cluster_split_reports_an_expired_wait_and_merges_nothing(cuda_lib):
    """The kernel hook's cluster split with a withheld K/V ring entry: every CTA's wait expires,
    no cluster merges, the host reads ATTN_ERR_TIMEOUT, and the context stays usable."""
    lib = cuda_lib
    w = wl.random_case(1, 2, 1, 1024, 128, False, 91)
    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.zeros_like(qd)
    lse = torch.zeros(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_debug_status(stream) == 0
    args = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), lse.data_ptr(), w.B,
            w.Hq, w.Hkv, w.N, w.D, 0, ctypes.c_float(w.sm_scale), 3)
    t0 = time.time()
    assert lib.attn_fwd_test_kernel(*args, 1, stream) == 0  # entry 1: V tile 0 of every CTA
    assert lib.attn_debug_status(stream) == -9
    assert 0.5 < time.time() - t0 < 30.0
    assert bool((out == 0).all()) and bool((lse == 0).all())  # nothing merged or stored
    assert lib.attn_fwd_test_kernel(*args, -1, stream) == 0
    assert lib.attn_debug_status(stream) == 0
    _check(out, lse, *oracle.attn_ref(q, k, v, False, w.sm_scale), "cluster split after expiry")


def test_cluster_split_in_a_cuda_graph(cuda_lib):
    """attn_fwd's cluster split captured into a CUDA graph (no claim counter is involved) and
    replayed on another stream gives the eager launch's bits."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.FEWHEADS
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    assert attn.fwd_num_splits(w.B, w.Hq, w.N, w.D, w.causal) > 1
    o_ref, l_ref = attn.attn_fwd(q, k, v, causal=w.causal, sm_scale=w.sm_scale)
    out = torch.zeros_like(q)
    lse = torch.zeros(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm up on the capturing stream
        attn.attn_fwd(q, k, v, causal=w.causal, sm_scale=w.sm_scale, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        attn.attn_fwd(q, k, v, causal=w.causal, sm_scale=w.sm_scale, out=out, lse=lse)
    for _ in range(2):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)


def test_scratch_and_counters_from_several_host_threads(cuda_lib):
    """Four host threads, each with its own stream, call attn_fwd at the same time on problems
    that take the scratch path, the cluster path and the single pass; the slot leases and claim
    counters keep every result equal to the same call made alone."""
    import threading

    import exact_attention_forward_attn_gb300 as attn

    shapes = [wl.random_case(1, 4, 1, 8192, 128, True, 110),   # workspace split, own scratch
              wl.FEWHEADS,                                      # cluster split
              wl.random_case(1, 32, 8, 2048, 128, True, 111),  # single pass (persistent)
              wl.random_case(1, 1, 1, 16384, 64, True, 112)]   # workspace split, D = 64
    ins = [tuple(t.cuda() for t in wl.make_qkv(w)) for w in shapes]
    refs = []
    for w, (q, k, v) in zip(shapes, ins):
        refs.append(attn.attn_fwd(q, k, v, causal=w.causal, sm_scale=w.sm_scale))
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            w, (q, k, v) = shapes[i], ins[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(8):
                    o, l = attn.attn_fwd(q, k, v, causal=w.causal, sm_scale=w.sm_scale)
                    st.synchronize()
                    if not (torch.equal(o, refs[i][0]) and torch.equal(l, refs[i][1])):
                        errors.append(f"{w.name}: result differs")
        except Exception as e:  # reported below, on the main thread
            errors.append(f"{shapes[i].name}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(shapes))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert attn.device_status() == 0


@pytest.mark.parametrize("shape", [(1, 1, 1, 6000, 8, False), (1, 1, 1, 6000, 40, True),
                                   (1, 2, 1, 3000, 16, False), (2, 1, 1, 5000, 72, True)],
                         ids=["d8", "d40-causal", "d16", "d72-causal-b2"])
def test_attn_fwd_split_narrow_heads(shape, cuda_lib):
    """Head dimensions below the padded width (the merge writes only the first D columns) on
    problems attn_fwd splits, against the oracle on sampled rows."""
    import exact_attention_forward_attn_gb300 as attn

    B, Hq, Hkv, N, D, causal = shape
    w = wl.random_case(B, Hq, Hkv, N, D, causal, 120 + D)
    assert attn.fwd_num_splits(B, Hq, N, D, causal) >= 2
    q, k, v = wl.make_qkv(w)
    out, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _sampled(w, q, k, v, out, lse)


@pytest.mark.parametrize("shape", [(1, 4, 1, 8192, 128), (1, 4, 2, 8192, 96)],
                         ids=["d128", "d96-padded-rows"])
def test_strided_workspace_split(shape, cuda_lib):
    """[B, N, H, D] views through attn_fwd_strided on a causal few-head problem that splits
    through attn_fwd's scratch: the merge kernel writes O through the caller's strides (rows of
    D + 8 elements here, whose 8 padding elements keep their guard pattern)."""
    import exact_attention_forward_attn_gb300 as attn

    B, Hq, Hkv, N, D = shape
    w = wl.random_case(B, Hq, Hkv, N, D, True, 130 + D)
    assert attn.fwd_num_splits(B, Hq, N, D, True) >= 2
    q, k, v = wl.make_qkv(w)
    qs, ks, vs = (t.transpose(1, 2).contiguous().cuda().transpose(1, 2) for t in (q, k, v))
    g = Guarded(B * N * Hq * (D + 8) * 2)
    full = g.typed(torch.bfloat16, (B, N, Hq, D + 8))
    out = full[..., :D].transpose(1, 2)  # [B, H, N, D] view with row stride Hq * (D + 8)
    o, lse = attn.attn_fwd(qs, ks, vs, causal=True, sm_scale=w.sm_scale, out=out)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert g.intact()
    assert bool((full[..., D:].contiguous().view(torch.uint8) == PATTERN).all())
    _sampled(w, q, k, v, o.contiguous(), lse)
