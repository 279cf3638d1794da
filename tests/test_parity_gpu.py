"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle, element by element.

Tolerance (the pages' bf16 check, read as torch.assert_close semantics, plus the LSE bound):
    |O_gpu - O_ref| <= 2e-2 + 2e-2 * |O_ref|   for every element,
    |LSE_gpu - LSE_ref| <= 1e-3                 for every row.
The five configurations are compared in full (C3, B=1 Hq=64 N=4096, is 0.27 TFLOP of fp64 work:
seconds on the host cores); only the long-context sweep (N >= 8192) and the wide-head workload are
compared on 64 seeded query rows per head.
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


def _gpu(w, q, k, v, stream=None):
    import exact_attention_forward_attn_gb300 as attn

    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if stream is None:
        out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
    else:
        with torch.cuda.stream(stream):
            out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status(dev) == 0, "device-side wait expired"
    return out, lse


def _check(o_gpu, l_gpu, o_ref, l_ref, label):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    l = l_gpu.float().cpu().numpy().astype(np.float64)
    assert o.shape == o_ref.shape and l.shape == l_ref.shape
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l)), f"{label}: non-finite output"
    err = np.abs(o - o_ref)
    bad = err > O_ATOL + O_RTOL * np.abs(o_ref)
    assert not bad.any(), (f"{label}: {int(bad.sum())}/{bad.size} O elements out of tolerance; "
                           f"max|dO|={err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    lerr = np.abs(l - l_ref)
    assert lerr.max() <= LSE_ATOL, (f"{label}: max|dLSE|={lerr.max():.3e} at "
                                    f"{np.unravel_index(lerr.argmax(), lerr.shape)}")
    return float(err.max()), float(lerr.max())


FULL = [wl.TINY_NONCAUSAL, wl.TINY_CAUSAL, wl.GQA4_CAUSAL, wl.GQA8_CAUSAL, wl.MHA, wl.MHA_OUTLIER,
        wl.MQA]


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_config_full_output(w, cuda_lib):
    q, k, v = wl.make_qkv(w)
    out, lse = _gpu(w, q, k, v)
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out, lse, o_ref, l_ref, w.name)


SAMPLED = [*wl.LONG.values(), wl.WIDE]


@pytest.mark.parametrize("w", SAMPLED, ids=[w.name for w in SAMPLED])
def test_config_sampled_rows(w, cuda_lib):
    """Full-size run (the benchmark's launch); 64 seeded rows per head against the oracle."""
    q, k, v = wl.make_qkv(w)
    out, lse = _gpu(w, q, k, v)
    rows = wl.sample_rows(w, 64)
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale, rows=rows.numpy())
    idx = rows.long()
    o_s = torch.stack([out[b, h].cpu()[idx[b, h]] for b in range(w.B) for h in range(w.Hq)])
    l_s = torch.stack([lse[b, h].cpu()[idx[b, h]] for b in range(w.B) for h in range(w.Hq)])
    _check(o_s.reshape(o_ref.shape), l_s.reshape(l_ref.shape), o_ref, l_ref, w.name)
    # every row (not only the sampled ones) is finite and a convex combination of V
    o_all = out.float()
    assert torch.isfinite(o_all).all() and torch.isfinite(lse).all()
    vmax = v.float().abs().amax().item()
    assert o_all.abs().amax().item() <= vmax * (1 + 1e-2) + 1e-2


RAGGED = [
    # (B, Hq, Hkv, N, D, causal)
    (1, 2, 1, 1, 64, False), (1, 2, 1, 1, 128, True), (2, 4, 2, 2, 128, False),
    (1, 2, 2, 64, 64, True), (1, 3, 3, 127, 128, False), (1, 3, 3, 127, 128, True),
    (2, 4, 2, 129, 64, False), (2, 4, 2, 129, 64, True), (1, 4, 1, 200, 128, False),
    (1, 4, 1, 200, 128, True), (1, 2, 1, 255, 64, True), (1, 2, 2, 256, 128, False),
    (3, 6, 2, 300, 128, True), (1, 8, 2, 383, 64, False), (1, 8, 2, 383, 128, True),
    (2, 2, 1, 384, 128, True), (1, 16, 4, 640, 128, False), (1, 16, 4, 700, 64, True),
    # head dims other than 64/128: computed on 64 or 128 columns zero-filled by the TMA
    (1, 4, 2, 200, 96, True), (1, 2, 1, 130, 32, False), (2, 4, 4, 256, 48, True),
    (1, 8, 2, 300, 80, False), (1, 2, 1, 128, 16, True), (1, 4, 1, 384, 112, True),
    (1, 2, 2, 129, 8, False),
    # wide heads (one Q tile per CTA): D = 256, and 136..248 zero-padded to 256
    (1, 2, 1, 1, 256, True), (1, 4, 2, 128, 256, False), (1, 4, 2, 300, 256, True),
    (2, 4, 1, 383, 256, False), (1, 8, 8, 640, 256, True), (1, 4, 2, 200, 192, True),
    (1, 2, 1, 129, 136, False), (1, 2, 2, 256, 248, True),
]


@pytest.mark.parametrize("shape", RAGGED, ids=[f"b{b}h{h}k{kv}n{n}d{d}{'c' if c else ''}"
                                               for b, h, kv, n, d, c in RAGGED])
def test_ragged_and_edge_shapes(shape, cuda_lib):
    B, Hq, Hkv, N, D, causal = shape
    w = wl.random_case(B, Hq, Hkv, N, D, causal, seed=1000 + N + D)
    q, k, v = wl.make_qkv(w)
    out, lse = _gpu(w, q, k, v)
    o_ref, l_ref = oracle.attn_ref(q, k, v, causal, w.sm_scale)
    _check(out, lse, o_ref, l_ref, w.name)


def test_custom_scale_and_large_scores(cuda_lib):
    """sm_scale other than 1/sqrt(D), with scores large enough to need the max subtraction."""
    w = wl.random_case(1, 4, 2, 256, 128, True, seed=77)
    q, k, v = wl.make_qkv(w)
    q = (q.float() * 4).to(torch.bfloat16)
    for scale in (0.5, 1.0 / 128):
        out, lse = _gpu_scale(q, k, v, True, scale)
        o_ref, l_ref = oracle.attn_ref(q, k, v, True, scale)
        _check(out, lse, o_ref, l_ref, f"scale={scale}")


def _gpu_scale(q, k, v, causal, scale):
    import exact_attention_forward_attn_gb300 as attn

    out, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, sm_scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return out, lse


def test_empty_problems(cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    for shape_q, shape_kv in (((0, 2, 16, 64), (0, 1, 16, 64)), ((1, 2, 0, 64), (1, 1, 0, 64))):
        q = torch.zeros(shape_q, dtype=torch.bfloat16, device="cuda")
        k = torch.zeros(shape_kv, dtype=torch.bfloat16, device="cuda")
        out, lse = attn.attn_fwd(q, k, k, causal=True)
        assert out.shape == q.shape and lse.shape == q.shape[:3]


def test_no_writes_outside_out_and_lse(cuda_lib):
    """Guard bands around out and lse stay untouched (ragged N: TMA stores clip at N)."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(2, 4, 2, 200, 128, False, seed=5)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    n_out, n_lse, pad = q.numel(), w.B * w.Hq * w.N, 4096
    out_buf = torch.full((n_out + 2 * pad,), -777.0, dtype=torch.bfloat16, device="cuda")
    lse_buf = torch.full((n_lse + 2 * pad,), -777.0, dtype=torch.float32, device="cuda")
    out = out_buf[pad:pad + n_out].view(q.shape)
    lse = lse_buf[pad:pad + n_lse].view(w.B, w.Hq, w.N)
    attn.attn_fwd(q, k, v, causal=False, out=out, lse=lse)
    torch.cuda.synchronize()
    for buf, n in ((out_buf, n_out), (lse_buf, n_lse)):
        assert torch.all(buf[:pad] == -777.0) and torch.all(buf[pad + n:] == -777.0)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_deterministic_and_stream_independent(cuda_lib):
    w = wl.GQA4_CAUSAL
    q, k, v = wl.make_qkv(w)
    o1, l1 = _gpu(w, q, k, v)
    o2, l2 = _gpu(w, q, k, v, stream=torch.cuda.Stream())
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_and_mqa_equal_expanded_heads(cuda_lib):
    """The kernel's GQA/MQA head map gives bit-identical results to explicitly repeated heads."""
    for Hq, Hkv in ((8, 2), (6, 1)):
        w = wl.random_case(2, Hq, Hkv, 256, 128, True, seed=Hq * 10 + Hkv)
        q, k, v = wl.make_qkv(w)
        o1, l1 = _gpu(w, q, k, v)
        g = Hq // Hkv
        w2 = w.with_(Hkv=Hq)
        o2, l2 = _gpu(w2, q, k.repeat_interleave(g, 1).contiguous(),
                      v.repeat_interleave(g, 1).contiguous())
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gpu_side_argument_errors(cuda_lib):
    lib = cuda_lib
    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(1, 2, 128, dtype=torch.float32, device="cuda")
    host = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16).pin_memory()
    unreg = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    s = ctypes.c_float(0.125)

    def call(qp, outp):
        return lib.attn_fwd(qp, k.data_ptr(), k.data_ptr(), outp, lse.data_ptr(), 1, 2, 1, 128,
                            64, 0, s, None)

    assert call(host.data_ptr(), out.data_ptr()) == -10      # pinned host memory
    assert call(unreg.data_ptr(), out.data_ptr()) == -10     # pageable host memory
    assert call(q.data_ptr(), q.data_ptr()) == -11           # out aliases q
    assert call(q.data_ptr(), out.data_ptr()) == 0
    torch.cuda.synchronize()


LARGE = [
    # (B, Hq, Hkv, N, D, causal): sequences beyond the configurations (ragged and power of two),
    # and many short heads (items >> SMs)
    (1, 2, 1, 100000, 128, True), (1, 2, 1, 131072, 128, True), (1, 2, 2, 65536, 64, False),
    (1, 1, 1, 1 << 20, 64, True),  # a million keys: 4096 work items of up to 8192 key steps
    (64, 32, 8, 128, 128, True), (16, 48, 16, 300, 128, False),
]


@pytest.mark.parametrize("shape", LARGE, ids=[f"b{b}h{h}k{kv}n{n}d{d}{'c' if c else ''}"
                                              for b, h, kv, n, d, c in LARGE])
def test_large_shapes_sampled_rows(shape, cuda_lib):
    """Long sequences and many heads: 32 seeded rows per head against the oracle (the first and
    last rows included), every row finite and inside the convex hull of V."""
    B, Hq, Hkv, N, D, causal = shape
    w = wl.random_case(B, Hq, Hkv, N, D, causal, seed=3000 + N % 997 + D)
    q, k, v = wl.make_qkv(w)
    out, lse = _gpu(w, q, k, v)
    rows = wl.sample_rows(w, min(32, N))
    rows[..., 0] = 0
    rows[..., -1] = N - 1
    rows = rows.sort(dim=-1).values
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale, rows=rows.numpy())
    idx = rows.long()
    o_c, l_c = out.cpu(), lse.cpu()
    o_s = torch.stack([o_c[b, h][idx[b, h]] for b in range(B) for h in range(Hq)])
    l_s = torch.stack([l_c[b, h][idx[b, h]] for b in range(B) for h in range(Hq)])
    _check(o_s.reshape(o_ref.shape), l_s.reshape(l_ref.shape), o_ref, l_ref, w.name)
    o_all = out.float()
    assert torch.isfinite(o_all).all() and torch.isfinite(lse).all()
    assert o_all.abs().amax().item() <= v.float().abs().amax().item() * (1 + 1e-2) + 1e-2
