"""Parity of the absorbed-MLA decode kernel (attn_mla_decode) with the fp64 oracle.

Element by element on seeded inputs: the DeepSeek-V3 widths (d_c = 512, d_r = 64, 128 heads),
one decode query per head, with ragged token counts (tail tiles), head counts below and above one
128-head tile, one token, and the token axis run whole or split (2-4 splits merged inside a thread-block
cluster, more by the merge kernel).
Tolerance as for the forward: |dO| <= 2e-2 + 2e-2 |O| elementwise, |dLSE| <= 1e-3.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_forward_attn_gb300 as attn
import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-2, 2e-2, 1e-3


def _check(out, lse, q, kv, scale, batches=None):
    qc, kvc = q.cpu(), kv.cpu()
    if batches is not None:
        qc, kvc = qc[batches], kvc[batches]
        out, lse = out[batches], lse[batches]
    ref_o, ref_l = oracle.mla_decode_ref(qc, kvc, 512, scale)
    got_o = out.float().cpu().numpy()
    got_l = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_l))
    err = np.abs(got_o - ref_o) - (O_ATOL + O_RTOL * np.abs(ref_o))
    assert err.max() <= 0, f"O: worst excess {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert np.abs(got_l - ref_l).max() <= LSE_ATOL, f"LSE err {np.abs(got_l - ref_l).max():.3e}"


def _run(w, splits):
    q, kv = wl.make_mla(w, device="cuda")
    out, lse = attn.mla_decode(q, kv, w.sm_scale, num_splits=splits)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return q, kv, out, lse


@pytest.mark.parametrize("w", [wl.MLA_TINY, wl.MLA_RAGGED, wl.MLA_B1[4096]],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_parity_full(w, splits):
    q, kv, out, lse = _run(w, splits)
    _check(out, lse, q, kv, w.sm_scale)


def test_parity_long_context_default_splits():
    w = wl.MLA_B1[16384]
    q, kv, out, lse = _run(w, 0)
    assert attn.mla_decode_num_splits(w.B, w.H, w.T) > 1
    _check(out, lse, q, kv, w.sm_scale)


def test_parity_batch32_sampled_batches():
    w = wl.MLA_B32
    q, kv, out, lse = _run(w, 0)
    _check(out, lse, q, kv, w.sm_scale, batches=[0, 13, 31])


@pytest.mark.parametrize("B,H,T,splits", [
    (1, 200, 130, 1),   # two head tiles, the second 72 heads
    (3, 1, 65, 2),      # one head, a one-token tail tile
    (2, 64, 1, 1),      # one cached token
    (1, 256, 640, 5),   # two full head tiles, splits of two tiles
])
def test_parity_shapes(B, H, T, splits):
    w = wl.MlaWorkload(f"mla-case-{B}-{H}-{T}", B, H, T, 90 + T)
    q, kv, out, lse = _run(w, splits)
    _check(out, lse, q, kv, w.sm_scale)


def test_single_token_returns_its_row():
    w = wl.MlaWorkload("mla-one", 2, 32, 1, 95)
    q, kv, out, lse = _run(w, 1)
    want = kv[:, 0, :512].unsqueeze(1).expand(-1, 32, -1)
    assert torch.equal(out, want)  # p = 1 exactly, then the bf16 row back


def test_deterministic_and_split_independent():
    w = wl.MLA_RAGGED
    q, kv, o1, l1 = _run(w, 3)
    o2, l2 = attn.mla_decode(q, kv, w.sm_scale, num_splits=3)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = attn.mla_decode(q, kv, w.sm_scale, num_splits=1)
    torch.cuda.synchronize()
    assert (o1.float() - o3.float()).abs().max().item() <= 2e-2
    assert (l1 - l3).abs().max().item() <= 1e-4


def test_device_errors_are_reported(cuda_lib):
    lib = cuda_lib
    q = torch.zeros(1, 4, 576, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, 8, 576, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, 4, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 4, dtype=torch.float32, device="cuda")
    host = (ctypes.c_uint16 * 16)()
    st = lib.attn_mla_decode(ctypes.addressof(host), kv.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), 1, 4, 8, 512, 64, ctypes.c_float(0.1), 1, None, 0,
                             None)
    assert st == -10  # host memory for q


def test_cluster_merge_repeated_launches():
    """With 2-4 splits the split CTAs of a group form a thread-block cluster and merge through
    distributed shared memory: one head, a partial second head tile and 3 or 4 splits (rows
    shared unevenly among the cluster's CTAs); 30 more launches of each must give the bits of
    the first."""
    cases = [(wl.MLA_RAGGED, 2), (wl.MlaWorkload("mla-fuse-h1", 3, 1, 65, 96), 2),
             (wl.MlaWorkload("mla-fuse-h200", 2, 200, 700, 97), 4),
             (wl.MlaWorkload("mla-fuse-h72", 1, 72, 1000, 99), 3)]
    data, first = [], []
    for w, splits in cases:
        q, kv, out, lse = _run(w, splits)
        _check(out, lse, q, kv, w.sm_scale)
        data.append((q, kv))
        first.append((out.clone(), lse.clone()))
    for _ in range(30):
        outs = [attn.mla_decode(q, kv, w.sm_scale, num_splits=splits)
                for (w, splits), (q, kv) in zip(cases, data)]
        torch.cuda.synchronize()
        for (o, l), (o0, l0) in zip(outs, first):
            assert torch.equal(o, o0) and torch.equal(l, l0)
    assert attn.device_status() == 0
