"""Host-side checks of the seeded input generators (no GPU)."""
import torch

from exact_attention_forward_attn_gb300 import workloads as wl


def test_generator_is_deterministic_and_bf16():
    w = wl.random_case(1, 4, 2, 96, 64, True, 9)
    a = wl.make_qkv(w)
    b = wl.make_qkv(w)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y) and x.is_contiguous()
    q, k, v = a
    assert q.shape == (1, 4, 96, 64) and k.shape == (1, 2, 96, 64) and v.shape == k.shape
    # Q, K, V are drawn in that order from one generator
    g = torch.Generator().manual_seed(9)
    q2 = torch.randn(1, 4, 96, 64, generator=g).to(torch.bfloat16)
    k2 = torch.randn(1, 2, 96, 64, generator=g).to(torch.bfloat16)
    assert torch.equal(q, q2) and torch.equal(k, k2)


def test_outlier_variant_scales_exactly_one_percent_of_k():
    base = wl.MHA.with_(N=64)
    out = base.with_(outlier_seed=104)
    _, k0, v0 = wl.make_qkv(base)
    _, k1, v1 = wl.make_qkv(out)
    assert torch.equal(v0, v1)
    changed = (k0 != k1)
    n = k0.numel()
    expect = int(round(0.01 * n))
    # entries that were exactly zero stay unchanged; every changed entry is exactly 8x
    assert changed.sum().item() <= expect
    assert torch.equal(k1[changed].float(), 8 * k0[changed].float())
    nonzero_picked = changed.sum().item()
    assert nonzero_picked >= expect - (k0 == 0).sum().item()


def test_sample_rows_distinct_sorted_in_range():
    w = wl.LONG[8192]
    rows = wl.sample_rows(w, 64)
    assert rows.shape == (1, 32, 64) and rows.dtype == torch.int32
    for h in range(32):
        r = rows[0, h]
        assert len(set(r.tolist())) == 64
        assert torch.all(r[1:] > r[:-1]) and r.min() >= 0 and r.max() < w.N
    assert not torch.equal(rows[0, 0], rows[0, 1])
    assert torch.equal(rows, wl.sample_rows(w, 64))


def test_registry_matches_the_five_configurations():
    assert (wl.TINY_NONCAUSAL.B, wl.TINY_NONCAUSAL.Hq, wl.TINY_NONCAUSAL.Hkv,
            wl.TINY_NONCAUSAL.N, wl.TINY_NONCAUSAL.D) == (1, 2, 1, 128, 64)
    assert (wl.GQA4_CAUSAL.B, wl.GQA4_CAUSAL.Hq, wl.GQA4_CAUSAL.Hkv, wl.GQA4_CAUSAL.N) == \
        (2, 32, 8, 1024)
    assert (wl.GQA8_CAUSAL.Hq, wl.GQA8_CAUSAL.Hkv, wl.GQA8_CAUSAL.N) == (64, 8, 4096)
    assert (wl.MHA.Hq, wl.MHA.Hkv, wl.MQA.Hq, wl.MQA.Hkv) == (32, 32, 16, 1)
    assert sorted(wl.LONG) == [8192, 16384, 32768]
    for w in wl.CONFIGS:
        assert abs(w.sm_scale - w.D ** -0.5) < 1e-15
    # FLOP convention: 4*B*Hq*N^2*D, halved when causal
    assert wl.LONG[8192].flops == 4 * 32 * 8192 ** 2 * 128 / 2
    assert wl.MHA.flops == 4 * 32 * 512 ** 2 * 128


def test_mla_workloads_shapes_scale_and_determinism():
    w = wl.MLA_B1[4096]
    assert (w.B, w.H, w.T, w.d_c, w.d_r, w.d_qk) == (1, 128, 4096, 512, 64, 576)
    assert abs(w.sm_scale - 192 ** -0.5) < 1e-15  # d_nope + d_r, not the absorbed width
    q, kv = wl.make_mla(wl.MLA_TINY)
    assert q.shape == (1, 16, 576) and kv.shape == (1, 200, 576)
    assert q.dtype == kv.dtype == torch.bfloat16
    q2, kv2 = wl.make_mla(wl.MLA_TINY)
    assert torch.equal(q, q2) and torch.equal(kv, kv2)
    assert w.flops == 2 * 128 * 4096 * (576 + 512)
    assert w.bytes == 2 * 4096 * 576 + 2 * 128 * 576 + 2 * 128 * 512 + 4 * 128


def test_bench_work_ratio_and_parity_helpers():
    """bench.py's extrapolation ratio counts visible (query, key) pairs exactly, and its parity
    summary applies the tests' tolerance."""
    import numpy as np
    import torch

    import bench

    w = wl.random_case(1, 2, 1, 10, 64, True, 1)
    rows = torch.tensor([[[0, 9], [3, 4]]], dtype=torch.int32)
    assert bench.causal_work(w) == 2 * 55                    # 1 + 2 + ... + 10 keys per head
    assert bench.causal_work(w, rows) == (1 + 10) + (4 + 5)
    wn = w.with_(causal=False)
    assert bench.causal_work(wn) == 2 * 100 and bench.causal_work(wn, rows) == 4 * 10
    ref_o = np.zeros((1, 2, 3, 4))
    ref_l = np.zeros((1, 2, 3))
    good = bench._parity(torch.full((1, 2, 3, 4), 0.015), torch.zeros(1, 2, 3), ref_o, ref_l)
    bad = bench._parity(torch.full((1, 2, 3, 4), 0.03), torch.zeros(1, 2, 3), ref_o, ref_l)
    assert good["within_tolerance"] and not bad["within_tolerance"]
    assert abs(bad["max_abs_dO"] - 0.03) < 1e-6
