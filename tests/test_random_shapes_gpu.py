"""Seeded random shapes against the oracle, through every forward entry point.

Forty problems drawn from one seeded generator: B in 1..3, Hkv in 1..4, Hq = Hkv * (1, 2, 3, 4
or 8), N in 1..2300, D a multiple of 8 in 8..256, causal or not; each runs contiguous through
attn_fwd, as a [B, N, H, D] view through attn_fwd_strided, through attn_fwd_splitkv with 2-5
splits (D <= 128), and on the CTA-pair kernel (64 < D <= 128).  Every element of every result
is compared with the fp64 oracle at the tests' tolerance (|dO| <= 2e-2 + 2e-2 |O_ref|,
|dLSE| <= 1e-3).  Twenty more (one or two heads over 2000-16000 keys, D a multiple of 8 up to
128) exercise the splits that attn_fwd and the split-KV default choose for themselves, on 32
sampled rows per head.
"""
import ctypes
import random

import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu


def _shapes(n=40, seed=20261202):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        hkv = rng.randint(1, 4)
        g = rng.choice([1, 2, 3, 4, 8])
        N = rng.choice([rng.randint(1, 300), rng.randint(300, 1200), rng.randint(1200, 2300)])
        D = 8 * rng.randint(1, 32)
        out.append((rng.randint(1, 3), hkv * g, hkv, N, D, rng.random() < 0.5, 4000 + i))
    return out


SHAPES = _shapes()


@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{b}h{h}k{k}n{n}d{d}{'c' if c else ''}"
                                               for b, h, k, n, d, c, _ in SHAPES])
def test_random_shape_every_entry_point(shape, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    B, Hq, Hkv, N, D, causal, seed = shape
    w = wl.random_case(B, Hq, Hkv, N, D, causal, seed)
    q, k, v = wl.make_qkv(w)
    o_ref, l_ref = oracle.attn_ref(q, k, v, causal, w.sm_scale)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()

    out, lse = attn.attn_fwd(qd, kd, vd, causal=causal, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(out, lse, o_ref, l_ref, f"attn_fwd {w.name}")

    def bnhd(t):
        return t.transpose(1, 2).contiguous().transpose(1, 2)

    out_s = bnhd(torch.empty_like(qd))
    out_s, lse_s = attn.attn_fwd(bnhd(qd), bnhd(kd), bnhd(vd), causal=causal,
                                 sm_scale=w.sm_scale, out=out_s)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(out_s.contiguous(), lse_s, o_ref, l_ref, f"strided {w.name}")

    if D <= 128:
        splits = 2 + seed % 4
        out_k, lse_k = attn.attn_fwd_splitkv(qd, kd, vd, causal=causal, sm_scale=w.sm_scale,
                                             num_splits=splits)
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        _check(out_k, lse_k, o_ref, l_ref, f"splitkv({splits}) {w.name}")

    if 64 < D <= 128:
        out_p = torch.empty_like(qd)
        lse_p = torch.empty(B, Hq, N, dtype=torch.float32, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert cuda_lib.attn_fwd_test_kernel(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                             out_p.data_ptr(), lse_p.data_ptr(), B, Hq, Hkv, N,
                                             D, int(causal), ctypes.c_float(w.sm_scale), 2, -1,
                                             stream) == 0
        torch.cuda.synchronize()
        assert cuda_lib.attn_debug_status(stream) == 0
        _check(out_p, lse_p, o_ref, l_ref, f"pair {w.name}")


def _split_shapes(n=20, seed=20261203):
    """Few heads over long key axes, where attn_fwd splits the key axis itself."""
    rng = random.Random(seed)
    out = []
    for i in range(n):
        hkv = rng.randint(1, 2)
        hq = hkv * rng.choice([1, 2])
        N = rng.randint(2000, 16000)
        D = 8 * rng.randint(1, 16)
        out.append((rng.randint(1, 2), hq, hkv, N, D, rng.random() < 0.5, 5000 + i))
    return out


SPLIT_SHAPES = _split_shapes()


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=[f"b{b}h{h}k{k}n{n}d{d}{'c' if c else ''}"
                                                     for b, h, k, n, d, c, _ in SPLIT_SHAPES])
def test_random_split_shapes_sampled_rows(shape, cuda_lib):
    """attn_fwd's own split (in clusters or through its scratch, as its cost model picks) and the
    split-KV default, against the oracle on 32 seeded rows per head (the first and last included)."""
    import exact_attention_forward_attn_gb300 as attn

    B, Hq, Hkv, N, D, causal, seed = shape
    w = wl.random_case(B, Hq, Hkv, N, D, causal, seed)
    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rows = wl.sample_rows(w, 32)
    rows[..., 0] = 0
    rows[..., -1] = N - 1
    rows = rows.sort(dim=-1).values
    o_ref, l_ref = oracle.attn_ref(q, k, v, causal, w.sm_scale, rows=rows.numpy())
    idx = rows.long()
    for name, (out, lse) in (
            ("attn_fwd", attn.attn_fwd(qd, kd, vd, causal=causal, sm_scale=w.sm_scale)),
            ("splitkv", attn.attn_fwd_splitkv(qd, kd, vd, causal=causal, sm_scale=w.sm_scale))):
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        o_c, l_c = out.cpu(), lse.cpu()
        o_s = torch.stack([o_c[b, h][idx[b, h]] for b in range(B) for h in range(Hq)])
        l_s = torch.stack([l_c[b, h][idx[b, h]] for b in range(B) for h in range(Hq)])
        splits = attn.fwd_num_splits(B, Hq, N, D, causal)
        _check(o_s.reshape(o_ref.shape), l_s.reshape(l_ref.shape), o_ref, l_ref,
               f"{name} (attn_fwd splits {splits}) {w.name}")
