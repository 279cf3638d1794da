"""The CTA-pair forward (two SMs share each M = 256 tcgen05 MMA), through the C ABI.

attn_fwd runs the one-CTA kernel (measured faster); attn_fwd_test_kernel runs either kernel on
any shape (1: one CTA, 2: CTA pair).  The pair kernel is checked here against the oracle on
ragged and edge shapes: N not a multiple of 128 or 512 (M-tiles whose second CTA holds only rows
past N, quads with one M-tile), causal and not, GQA / MQA / MHA, padded head dimensions, several
batches; and its bounded waits against a withheld K/V half.
Tolerance as everywhere: |dO| <= 2e-2 + 2e-2 |O_ref| per element, |dLSE| <= 1e-3.
"""
import ctypes

import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu


def _run(lib, w, q, k, v, kernel, stall_item=-1):
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.Hq, w.N), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.attn_fwd_test_kernel(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.D, int(w.causal),
                                  ctypes.c_float(w.sm_scale), kernel, stall_item, stream)
    assert st == 0, st
    torch.cuda.synchronize()
    if stall_item < 0:
        assert lib.attn_debug_status(stream) == 0
    return out, lse


SHAPES = [
    # (B, Hq, Hkv, N, D, causal)
    (1, 2, 1, 1, 128, True), (1, 2, 1, 1, 128, False), (1, 2, 2, 100, 128, True),
    (1, 2, 1, 128, 128, True), (1, 2, 1, 129, 128, True), (1, 4, 2, 200, 128, False),
    (1, 4, 1, 255, 128, True), (2, 4, 2, 256, 128, True), (1, 3, 3, 300, 128, False),
    (1, 4, 2, 383, 128, True), (1, 2, 1, 384, 128, True), (1, 4, 4, 511, 128, True),
    (1, 4, 2, 512, 128, True), (1, 4, 2, 512, 128, False), (1, 2, 1, 513, 128, True),
    (2, 6, 2, 640, 128, True), (1, 8, 1, 700, 128, False), (1, 4, 2, 1000, 128, True),
    (1, 16, 4, 1100, 128, True), (3, 4, 2, 1500, 128, False),
    # padded head dimensions (zero-filled to 128 by the TMA)
    (1, 4, 2, 300, 96, True), (1, 2, 1, 700, 72, False), (2, 4, 4, 600, 120, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{b}h{h}k{kv}n{n}d{d}{'c' if c else ''}"
                                               for b, h, kv, n, d, c in SHAPES])
def test_pair_kernel_matches_oracle(shape, cuda_lib):
    B, Hq, Hkv, N, D, causal = shape
    w = wl.random_case(B, Hq, Hkv, N, D, causal, seed=2000 + N + D)
    q, k, v = wl.make_qkv(w)
    out, lse = _run(cuda_lib, w, q.cuda(), k.cuda(), v.cuda(), 2)
    o_ref, l_ref = oracle.attn_ref(q, k, v, causal, w.sm_scale)
    _check(out, lse, o_ref, l_ref, f"pair {w.name}")


@pytest.mark.parametrize("w", [wl.GQA4_CAUSAL, wl.MHA_OUTLIER, wl.MQA],
                         ids=lambda w: w.name)
def test_pair_kernel_on_the_configurations(w, cuda_lib):
    """Configurations attn_fwd runs on the one-CTA kernel, here forced onto pairs; and the two
    kernels against each other."""
    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = _run(cuda_lib, w, qd, kd, vd, 2)
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out, lse, o_ref, l_ref, f"pair {w.name}")
    o1, l1 = _run(cuda_lib, w, qd, kd, vd, 1)
    assert (o1.float() - out.float()).abs().max().item() <= 2e-2
    assert (l1 - lse).abs().max().item() <= 1e-3


def test_pair_kernel_repeated_launches_are_bit_identical(cuda_lib):
    """Quads are claimed from the launch's counter; whichever pair computes a quad, its bits are
    the same."""
    w = wl.random_case(1, 24, 6, 1900, 128, True, 2101)  # 4 quads per head, the last ragged
    qd, kd, vd = (t.cuda() for t in wl.make_qkv(w))
    first = _run(cuda_lib, w, qd, kd, vd, 2)
    for _ in range(30):
        again = _run(cuda_lib, w, qd, kd, vd, 2)
        assert torch.equal(again[0], first[0]) and torch.equal(again[1], first[1])


def test_attn_fwd_runs_the_one_cta_kernel(cuda_lib):
    """attn_fwd on C3 (B=1, Hq=64, N=4096) equals the forced one-CTA launch bit for bit, and the
    pair kernel within the tolerance."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.GQA8_CAUSAL
    qd, kd, vd = (t.cuda() for t in wl.make_qkv(w))
    out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
    one = _run(cuda_lib, w, qd, kd, vd, 1)
    assert torch.equal(out, one[0]) and torch.equal(lse, one[1])
    pair = _run(cuda_lib, w, qd, kd, vd, 2)
    assert (pair[0].float() - out.float()).abs().max().item() <= 2e-2
    assert (pair[1] - lse).abs().max().item() <= 1e-3


def test_pair_kernel_expired_wait_is_reported(cuda_lib):
    """A withheld K/V half starves every pair: the bounded waits of both CTAs expire, the host
    reads ATTN_ERR_TIMEOUT, and the next pair launch on the same context is correct."""
    lib = cuda_lib
    w = wl.Workload("pair-stall", 2, 64, 8, 1024, 128, False, 2102)
    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_debug_status(stream) == 0
    _run(lib, w, qd, kd, vd, 2, stall_item=1)
    assert lib.attn_debug_status(stream) == -9
    assert lib.attn_debug_status(stream) == 0
    o2, l2 = _run(lib, w, qd, kd, vd, 2)
    rows = wl.sample_rows(w, 16)
    o_ref, l_ref = oracle.attn_ref(q, k, v, False, w.sm_scale, rows=rows.numpy())
    idx = rows.long()
    o_s = torch.stack([o2[b, h].cpu()[idx[b, h]] for b in range(w.B) for h in range(w.Hq)])
    l_s = torch.stack([l2[b, h].cpu()[idx[b, h]] for b in range(w.B) for h in range(w.Hq)])
    _check(o_s.reshape(o_ref.shape), l_s.reshape(l_ref.shape), o_ref, l_ref, "after the stall")


def test_pair_kernel_long_ragged_sequence(cuda_lib):
    """N = 70000 (137 quads per head, the last one ragged): 32 seeded rows per head."""
    w = wl.random_case(1, 4, 1, 70000, 128, True, 2103)
    q, k, v = wl.make_qkv(w)
    out, lse = _run(cuda_lib, w, q.cuda(), k.cuda(), v.cuda(), 2)
    rows = wl.sample_rows(w, 32)
    rows[..., -1] = w.N - 1
    rows = rows.sort(dim=-1).values
    o_ref, l_ref = oracle.attn_ref(q, k, v, True, w.sm_scale, rows=rows.numpy())
    idx = rows.long()
    o_c, l_c = out.cpu(), lse.cpu()
    o_s = torch.stack([o_c[0, h][idx[0, h]] for h in range(w.Hq)])
    l_s = torch.stack([l_c[0, h][idx[0, h]] for h in range(w.Hq)])
    _check(o_s.reshape(o_ref.shape), l_s.reshape(l_ref.shape), o_ref, l_ref, w.name)
