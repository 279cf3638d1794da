"""GPU parity of the split-KV forward (key-axis splits + fused safe-softmax merge) against the
fp64 oracle, with the same element-wise tolerance as the single-pass forward."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu


def _run_split(w, q, k, v, splits, workspace=None):
    import exact_attention_forward_attn_gb300 as attn

    out, lse = attn.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=w.causal,
                                     sm_scale=w.sm_scale, num_splits=splits,
                                     workspace=workspace)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return out, lse


CASES = [(wl.MHA, 2), (wl.MHA, 4), (wl.MHA_OUTLIER, 3), (wl.MQA, 4), (wl.TINY_NONCAUSAL, 2),
         (wl.TINY_CAUSAL, 2), (wl.GQA4_CAUSAL, 4), (wl.GQA4_CAUSAL, 8),
         (wl.random_case(2, 4, 2, 700, 128, True, 11), 3),
         (wl.random_case(1, 6, 3, 383, 64, False, 12), 2),
         (wl.random_case(1, 4, 1, 1000, 128, True, 13), 16),
         (wl.random_case(3, 2, 2, 129, 64, True, 14), 2),
         (wl.random_case(1, 4, 2, 1000, 96, True, 15), 4),
         (wl.random_case(2, 2, 1, 600, 40, False, 16), 3)]


@pytest.mark.parametrize("w,splits", CASES, ids=[f"{w.name}-s{s}" for w, s in CASES])
def test_splitkv_matches_oracle(w, splits, cuda_lib):
    q, k, v = wl.make_qkv(w)
    out, lse = _run_split(w, q, k, v, splits)
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out, lse, o_ref, l_ref, f"{w.name} splits={splits}")


def test_splitkv_close_to_single_pass_and_ignores_stale_workspace(cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    w = wl.MHA
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    o1, l1 = attn.attn_fwd(q, k, v, causal=False, sm_scale=w.sm_scale)
    need = attn.splitkv_workspace_bytes(w.B, w.Hq, w.N, w.D, 4)
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device="cuda")
    o2, l2 = attn.attn_fwd_splitkv(q, k, v, causal=False, sm_scale=w.sm_scale, num_splits=4,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert torch.isfinite(o2.float()).all() and torch.isfinite(l2).all()
    assert (o1.float() - o2.float()).abs().max().item() < 2e-2
    assert (l1 - l2).abs().max().item() < 1e-4


def test_splitkv_heuristic_splits_low_occupancy_shapes(cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    # 32 query tiles of 32 key tiles each on a GPU with >100 SMs: the cost model splits; 4 key
    # tiles per query tile (N=512) or enough query tiles (the long workload): it does not
    assert attn.splitkv_num_splits(1, 2, 4096, 128) > 1
    assert attn.splitkv_num_splits(1, 32, 512, 128) == 1
    assert attn.splitkv_num_splits(1, 16, 512, 128) == 1
    assert attn.splitkv_num_splits(1, 32, 32768, 128, True) == 1
    w = wl.FEWHEADS
    q, k, v = wl.make_qkv(w)
    out, lse = _run_split(w, q, k, v, 0)  # 0: the library's choice
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out, lse, o_ref, l_ref, "fewheads heuristic")
