"""Pins for the oracle's backward (dQ, dK, dV of softmax attention, recomputed from the
definition): a textbook library routine on tiny inputs (torch float64 autograd), closed forms and
invariants of the softmax Jacobian, and a brute-force GQA expansion."""
import math

import numpy as np
import pytest
import torch

import oracle

TOL = 1e-11


def _randn(g, *shape):
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b) / (1.0 + np.abs(b))) if a.size else 0.0
    assert err <= tol, f"max scaled error {err:.3e} > {tol:.1e}"


@pytest.mark.parametrize("shape", [(1, 2, 1, 9, 8), (2, 4, 2, 23, 16), (1, 3, 3, 40, 32)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_float64_autograd(shape, causal):
    B, Hq, Hkv, N, D = shape
    g = torch.Generator().manual_seed(60 + N)
    q, k, v, do = (_randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D),
                   _randn(g, B, Hq, N, D))
    scale = 1 / math.sqrt(D)
    dq, dk, dv = oracle.attn_bwd_ref(q, k, v, do, causal, scale)
    qd = q.double().requires_grad_()
    kd = k.double().requires_grad_()
    vd = v.double().requires_grad_()
    grp = Hq // Hkv
    s = scale * (qd @ kd.repeat_interleave(grp, 1).transpose(-1, -2))
    if causal:
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    o = torch.softmax(s, dim=-1) @ vd.repeat_interleave(grp, 1)
    o.backward(do.double())
    _close(dq, qd.grad.numpy())
    _close(dk, kd.grad.numpy())
    _close(dv, vd.grad.numpy())


@pytest.mark.parametrize("causal", [False, True])
def test_single_key(causal):
    """N = 1: p = 1 for the only key, so ds = 0: dQ = dK = 0 and dV = the sum of dO over the
    query heads of the KV head."""
    g = torch.Generator().manual_seed(61)
    B, Hq, Hkv, D = 2, 4, 2, 16
    q, k, v, do = (_randn(g, B, Hq, 1, D), _randn(g, B, Hkv, 1, D), _randn(g, B, Hkv, 1, D),
                   _randn(g, B, Hq, 1, D))
    dq, dk, dv = oracle.attn_bwd_ref(q, k, v, do, causal, 0.25)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    dod = do.double().numpy()
    for hk in range(Hkv):
        _close(dv[:, hk], dod[:, 2 * hk] + dod[:, 2 * hk + 1])


def test_identical_keys_give_zero_dq():
    """Identical keys: dQ_i = scale * sum_j ds_ij k = scale * k * sum_j ds_ij = 0, because every
    row of ds sums to zero (softmax Jacobian)."""
    g = torch.Generator().manual_seed(62)
    B, Hq, Hkv, N, D = 1, 2, 1, 30, 16
    q, v, do = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hq, N, D)
    k = _randn(g, B, Hkv, 1, D).expand(B, Hkv, N, D).contiguous()
    for causal in (False, True):
        dq, _, _ = oracle.attn_bwd_ref(q, k, v, do, causal, 0.3)
        assert np.max(np.abs(dq)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_column_sums(causal):
    """sum_j dK_j = scale * sum_i q_i sum_j ds_ij = 0, and sum_j dV_j = sum over the group's
    query heads and rows of dO (each probability row sums to 1)."""
    g = torch.Generator().manual_seed(63)
    B, Hq, Hkv, N, D = 2, 4, 2, 37, 32
    q, k, v, do = (_randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D),
                   _randn(g, B, Hq, N, D))
    _, dk, dv = oracle.attn_bwd_ref(q, k, v, do, causal, 1 / math.sqrt(D))
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-10
    dod = do.double().numpy()
    for hk in range(Hkv):
        want = dod[:, 2 * hk].sum(axis=1) + dod[:, 2 * hk + 1].sum(axis=1)
        _close(dv[:, hk].sum(axis=1), want, 1e-10)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_heads(causal):
    g = torch.Generator().manual_seed(64)
    B, Hq, Hkv, N, D = 1, 6, 2, 21, 16
    q, k, v, do = (_randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D),
                   _randn(g, B, Hq, N, D))
    grp = Hq // Hkv
    dq, dk, dv = oracle.attn_bwd_ref(q, k, v, do, causal, 0.25)
    dq2, dk2, dv2 = oracle.attn_bwd_ref(q, k.repeat_interleave(grp, 1).contiguous(),
                                        v.repeat_interleave(grp, 1).contiguous(), do, causal, 0.25)
    assert np.array_equal(dq, dq2)
    for hk in range(Hkv):
        sk = np.zeros_like(dk[:, hk])
        sv = np.zeros_like(dv[:, hk])
        for r in range(grp):  # the oracle adds the query heads in this order
            sk = sk + dk2[:, hk * grp + r]
            sv = sv + dv2[:, hk * grp + r]
        assert np.array_equal(dk[:, hk], sk) and np.array_equal(dv[:, hk], sv)


def test_threading_does_not_change_gradients():
    g = torch.Generator().manual_seed(65)
    q, k, v, do = (_randn(g, 1, 4, 25, 16), _randn(g, 1, 2, 25, 16), _randn(g, 1, 2, 25, 16),
                   _randn(g, 1, 4, 25, 16))
    a = oracle.attn_bwd_ref(q, k, v, do, True, 0.25, n_threads=1)
    b = oracle.attn_bwd_ref(q, k, v, do, True, 0.25, n_threads=3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
