"""The persistent forward's work claiming, exercised through the C ABI.

The two-tile forward runs one CTA per SM; each CTA takes one work item (a pair of Q tiles of one
head) and then claims more from a per-launch counter, one of 64 the host hands out round robin;
the launch's last claim sets its counter back to zero, and a launch that reuses a counter waits
for the counter's previous launch.  Launches captured into a CUDA graph take no counter and use
the kernel's static schedule.  These tests check what that must not change: every item is
computed exactly once whatever the launch order, the number of launches (more than the 64
counters), the grid size (more items than SMs, or fewer), concurrent launches on many streams,
or graph replays.  Each item's arithmetic does not depend on which CTA runs it, so repeated
launches must give bit-identical outputs; one launch per shape is also checked against the oracle.
"""
import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu

# More items than SMs (several claims per CTA), fewer (one static item per CTA), and a split run.
SHAPES = [
    wl.GQA4_CAUSAL,                                            # 256 items
    wl.TINY_CAUSAL,                                            # 2 items
    wl.Workload("pers-mqa-n2000", 1, 40, 1, 2000, 128, True, 41),  # 320 items, ragged N
    wl.Workload("pers-d64-n3000", 2, 8, 4, 3000, 64, False, 42),   # 192 items, D = 64
    # 15 Q tiles per head: every head's last item has one Q tile, so items with and without
    # the ping-pong partner alternate in every CTA's sequence
    wl.Workload("pers-odd-n1900", 1, 24, 6, 1900, 128, True, 43),  # 192 items
]


def _inputs(w, dev):
    q, k, v = wl.make_qkv(w)
    return (q, k, v), tuple(t.to(dev) for t in (q, k, v))


def test_many_launches_alternating_shapes_are_bit_identical(cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    data = [_inputs(w, dev) for w in SHAPES]
    first = []
    for w, (host, (qd, kd, vd)) in zip(SHAPES, data):
        out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
        torch.cuda.synchronize()
        o_ref, l_ref = oracle.attn_ref(*host, w.causal, w.sm_scale)
        _check(out, lse, o_ref, l_ref, w.name)
        first.append((out.clone(), lse.clone()))
    # 3 x 5 x 13 = 195 launches: every counter slot is reused, by shapes of different grids
    for rnd in range(13):
        for i, (w, (host, (qd, kd, vd))) in enumerate(zip(SHAPES, data)):
            out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
            out2, lse2 = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
            out3, lse3 = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
            torch.cuda.synchronize()
            for o, l in ((out, lse), (out2, lse2), (out3, lse3)):
                assert torch.equal(o, first[i][0]), f"{w.name}: O differs in round {rnd}"
                assert torch.equal(l, first[i][1]), f"{w.name}: LSE differs in round {rnd}"
    assert attn.device_status(dev) == 0


def test_concurrent_launches_on_two_streams(cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    wa, wb = SHAPES[0], SHAPES[2]
    (_, (qa, ka, va)), (_, (qb, kb, vb)) = _inputs(wa, dev), _inputs(wb, dev)
    ref_a = attn.attn_fwd(qa, ka, va, causal=wa.causal, sm_scale=wa.sm_scale)
    ref_b = attn.attn_fwd(qb, kb, vb, causal=wb.causal, sm_scale=wb.sm_scale)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    outs = []
    for _ in range(20):
        with torch.cuda.stream(sa):
            oa = attn.attn_fwd(qa, ka, va, causal=wa.causal, sm_scale=wa.sm_scale)
        with torch.cuda.stream(sb):
            ob = attn.attn_fwd(qb, kb, vb, causal=wb.causal, sm_scale=wb.sm_scale)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    for oa, ob in outs:
        assert torch.equal(oa[0], ref_a[0]) and torch.equal(oa[1], ref_a[1])
        assert torch.equal(ob[0], ref_b[0]) and torch.equal(ob[1], ref_b[1])
    assert attn.device_status(dev) == 0


def test_eighty_concurrent_launches_on_eighty_streams(cuda_lib):
    """More overlapping launches than there are claim counters: the 65th launch reuses the
    first one's counter and must wait for it, not share it.  Every launch is enqueued (two
    shapes, alternating) before anything is synchronised; all 80 results must be the serial
    launches' bits."""
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    shapes = [wl.Workload("conc-a-n2048", 1, 16, 4, 2048, 128, True, 51),   # 128 items
              wl.Workload("conc-b-n3000", 1, 24, 8, 3000, 128, False, 52)]  # 288 items
    data = [_inputs(w, dev)[1] for w in shapes]
    ref = []
    for w, (qd, kd, vd) in zip(shapes, data):
        ref.append(attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(dev) for _ in range(80)]
    outs = []
    for i, st in enumerate(streams):
        w, (qd, kd, vd) = shapes[i % 2], data[i % 2]
        with torch.cuda.stream(st):
            outs.append(attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale))
    torch.cuda.synchronize()
    for i, (o, l) in enumerate(outs):
        assert torch.equal(o, ref[i % 2][0]) and torch.equal(l, ref[i % 2][1]), f"launch {i}"
    assert attn.device_status(dev) == 0


@pytest.mark.parametrize("w", [wl.FEWHEADS, wl.Workload("pers-split-causal-n1900", 1, 4, 2, 1900,
                                                          128, True, 44)],
                         ids=["fewheads-n4096", "causal-n1900"])
def test_split_launches_reuse_counters(w, cuda_lib):
    """Split-KV launches claim (item, split) pairs through the same counters; under the causal
    mask some items have only their second Q tile, or no tile, in a split."""
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    host, (qd, kd, vd) = _inputs(w, dev)
    o_ref, l_ref = oracle.attn_ref(*host, w.causal, w.sm_scale)
    base = {}
    for n_splits in (2, 3, 4, 7) * 20:
        out, lse = attn.attn_fwd_splitkv(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale,
                                         num_splits=n_splits)
        torch.cuda.synchronize()
        if n_splits not in base:
            _check(out, lse, o_ref, l_ref, f"{w.name} splits={n_splits}")
            base[n_splits] = (out.clone(), lse.clone())
        else:
            assert torch.equal(out, base[n_splits][0]) and torch.equal(lse, base[n_splits][1])
    assert attn.device_status(dev) == 0


def test_cuda_graph_replays(cuda_lib):
    """Launches captured in a CUDA graph run the static schedule (no claim counter), so every
    replay computes every item once."""
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    wa, wb = SHAPES[0], SHAPES[4]
    (_, (qa, ka, va)), (_, (qb, kb, vb)) = _inputs(wa, dev), _inputs(wb, dev)
    ref_a = attn.attn_fwd(qa, ka, va, causal=wa.causal, sm_scale=wa.sm_scale)
    ref_b = attn.attn_fwd(qb, kb, vb, causal=wb.causal, sm_scale=wb.sm_scale)
    torch.cuda.synchronize()
    oa, la = torch.empty_like(ref_a[0]), torch.empty_like(ref_a[1])
    ob, lb = torch.empty_like(ref_b[0]), torch.empty_like(ref_b[1])
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):  # warm up on the capture stream
        attn.attn_fwd(qa, ka, va, causal=wa.causal, sm_scale=wa.sm_scale, out=oa, lse=la)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(2):
            attn.attn_fwd(qa, ka, va, causal=wa.causal, sm_scale=wa.sm_scale, out=oa, lse=la)
            attn.attn_fwd(qb, kb, vb, causal=wb.causal, sm_scale=wb.sm_scale, out=ob, lse=lb)
    for _ in range(20):
        oa.zero_()
        ob.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(oa, ref_a[0]) and torch.equal(la, ref_a[1])
        assert torch.equal(ob, ref_b[0]) and torch.equal(lb, ref_b[1])
    assert attn.device_status(dev) == 0


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_one_tile_items_match_pairs(causal, cuda_lib):
    """A launch with few Q-tile pairs runs one Q tile per work item; the same heads inside a
    larger batch run as pairs.  Each tile's arithmetic is the same either way, so the first
    batch's outputs must be bit-identical."""
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    small = wl.Workload("one-tile-n640", 1, 8, 2, 640, 128, causal, 45)  # 24 pairs < SMs / 2
    big = wl.Workload("pairs-n640", 8, 8, 2, 640, 128, causal, 46)       # 192 pairs
    q1, k1, v1 = wl.make_qkv(small)
    qb, kb, vb = wl.make_qkv(big)
    qb[0], kb[0], vb[0] = q1[0], k1[0], v1[0]
    o1, l1 = attn.attn_fwd(q1.to(dev), k1.to(dev), v1.to(dev), causal=causal)
    ob, lb = attn.attn_fwd(qb.to(dev), kb.to(dev), vb.to(dev), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1[0], ob[0]) and torch.equal(l1[0], lb[0])
    o_ref, l_ref = oracle.attn_ref(q1, k1, v1, causal, small.sm_scale)
    _check(o1, l1, o_ref, l_ref, small.name)
    assert attn.device_status(dev) == 0


def test_graphs_of_the_same_launches_replay_concurrently(cuda_lib):
    """Two graphs captured from the same launches, replayed at the same time on two streams
    (and beside an eager launch of the same shape): captured launches hold no shared state."""
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    w = SHAPES[2]
    _, (qd, kd, vd) = _inputs(w, dev)
    ref = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    bufs = [(torch.empty_like(ref[0]), torch.empty_like(ref[1])) for _ in range(2)]
    graphs = []
    for o, l in bufs:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=o, lse=l)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(3):
                attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=o, lse=l)
        graphs.append(g)
    s0, s1, s2 = (torch.cuda.Stream(dev) for _ in range(3))
    for _ in range(10):
        for (o, l) in bufs:
            o.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(s0):
            graphs[0].replay()
        with torch.cuda.stream(s1):
            graphs[1].replay()
        with torch.cuda.stream(s2):
            eager = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
        torch.cuda.synchronize()
        for o, l in (*bufs, eager):
            assert torch.equal(o, ref[0]) and torch.equal(l, ref[1])
    assert attn.device_status(dev) == 0


def test_dependent_launch_chains_in_a_cuda_graph(cuda_lib):
    """The split-KV forward (partials kernel + merge kernel), the backward (Delta, dK/dV, dQ) and
    the MLA decode with the merge kernel launch their second kernels as programmatic dependants;
    captured into a CUDA graph and replayed, they give the eager launches' bits."""
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    w = wl.Workload("graph-chain", 1, 4, 2, 1500, 128, True, 47)
    _, (qd, kd, vd) = _inputs(w, dev)
    gen = torch.Generator().manual_seed(48)
    do = torch.randn(qd.shape, generator=gen).to(torch.bfloat16).to(dev)
    wm = wl.MlaWorkload("graph-mla", 1, 128, 2048, 49)
    qm, kvm = wl.make_mla(wm, device=dev)
    ws = torch.empty(attn.splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, 3), dtype=torch.uint8,
                     device=dev)
    wsm = torch.empty(max(16, attn.mla_decode_workspace_bytes(wm.B, wm.H, wm.T, 8)),
                      dtype=torch.uint8, device=dev)

    def run():
        o, l = attn.attn_fwd_splitkv(qd, kd, vd, causal=True, num_splits=3, workspace=ws)
        o2, l2 = attn.attn_fwd(qd, kd, vd, causal=True)
        g = attn.attn_bwd(qd, kd, vd, o2, l2, do, causal=True)
        m = attn.mla_decode(qm, kvm, wm.sm_scale, num_splits=8, workspace=wsm)
        return (o, l, *g, *m)

    ref = [t.clone() for t in run()]
    torch.cuda.synchronize()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = run()
    for _ in range(5):
        for t in outs:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(outs, ref):
            assert torch.equal(a, b)
    assert attn.device_status(dev) == 0
