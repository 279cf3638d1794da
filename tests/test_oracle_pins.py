"""Pins for the fp64 CPU oracle: checks against what the pages and the mathematics fix.

None of these compares the oracle with itself.  Each pins it to something independent:
closed forms (tests/golden and the identical-key / causal-row-0 / N=1 cases), invariants
(probability rows sum to 1, shift invariance in K, affinity in V), a second evaluation order that
the pages prescribe (the blockwise online-softmax recurrence), a brute-force GQA expansion, and a
textbook library routine on tiny inputs (torch float64 softmax / logsumexp).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
TOL = 1e-12


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


def _randn(g, *shape):
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b) / (1.0 + np.abs(b))) if a.size else 0.0
    assert err <= tol, f"max scaled error {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------------------------
# Golden closed-form cases ("Attention Kernel 实现与正确性验证" sections 1.1-1.2; "Triton-CUDA
# Attention" online softmax + variants; "Flash Attention 与 Kernel 优化" LSE = m + log l).
# --------------------------------------------------------------------------------------------
with open(os.path.join(HERE, "golden", "closed_form_cases.json")) as fh:
    GOLDEN = json.load(fh)["cases"]


def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp, "log": math.log}))


def _eval_tree(x):
    if isinstance(x, list):
        return [_eval_tree(e) for e in x]
    return _eval(x)


@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
def test_golden_closed_form(case):
    q, k, v = _bf16(case["q"]), _bf16(case["k"]), _bf16(case["v"])
    # inputs of the fixtures are exact in bf16
    assert torch.equal(q.float(), torch.tensor(case["q"], dtype=torch.float32))
    assert torch.equal(k.float(), torch.tensor(case["k"], dtype=torch.float32))
    assert q.shape == (case["B"], case["Hq"], case["N"], case["D"])
    assert k.shape == (case["B"], case["Hkv"], case["N"], case["D"])
    out, lse = oracle.attn_ref(q, k, v, case["causal"], case["sm_scale"], n_threads=1)
    _close(out, _eval_tree(case["O"]))
    _close(lse, _eval_tree(case["LSE"]))


# --------------------------------------------------------------------------------------------
# Closed forms on random inputs
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_visible_values(causal):
    """All keys of a head equal => uniform softmax over J(i): O_i = mean V[J(i)],
    LSE_i = sm_scale * q_i.k + ln |J(i)| (|J(i)| = i+1 under the top-left causal mask)."""
    g = torch.Generator().manual_seed(21)
    B, Hq, Hkv, N, D = 2, 4, 2, 37, 16
    q = _randn(g, B, Hq, N, D)
    k = _randn(g, B, Hkv, 1, D).expand(B, Hkv, N, D).contiguous()
    v = _randn(g, B, Hkv, N, D)
    scale = 0.3
    out, lse = oracle.attn_ref(q, k, v, causal, scale)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    for b in range(B):
        for h in range(Hq):
            hk = h * Hkv // Hq
            for i in range(N):
                n = i + 1 if causal else N
                _close(out[b, h, i], vd[b, hk, :n].mean(axis=0))
                _close(lse[b, h, i], scale * float(qd[b, h, i] @ kd[b, hk, 0]) + math.log(n))


def test_causal_row0_is_first_value():
    """Under the causal mask row 0 sees key 0 only: O_0 = V[0], LSE_0 = sm_scale * q_0.k_0."""
    g = torch.Generator().manual_seed(22)
    B, Hq, Hkv, N, D = 2, 6, 3, 50, 64
    q, k, v = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D)
    out, lse = oracle.attn_ref(q, k, v, True, 0.125)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    for b in range(B):
        for h in range(Hq):
            hk = h * Hkv // Hq
            assert np.array_equal(out[b, h, 0], vd[b, hk, 0])
            _close(lse[b, h, 0], 0.125 * float(qd[b, h, 0] @ kd[b, hk, 0]))


@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_value(causal):
    """N = 1: the only key gets probability 1 in either mode."""
    g = torch.Generator().manual_seed(23)
    q, k, v = _randn(g, 3, 4, 1, 128), _randn(g, 3, 2, 1, 128), _randn(g, 3, 2, 1, 128)
    out, lse = oracle.attn_ref(q, k, v, causal, 1 / math.sqrt(128))
    vd = _f64(v)
    for h in range(4):
        assert np.array_equal(out[:, h, 0], vd[:, h * 2 // 4, 0])


def test_empty_batch_and_sequence():
    z = torch.zeros(0, 2, 5, 8, dtype=torch.bfloat16)
    out, lse = oracle.attn_ref(z, z[:, :1], z[:, :1], False, 1.0)
    assert out.shape == (0, 2, 5, 8) and lse.shape == (0, 2, 5)
    z = torch.zeros(1, 2, 0, 8, dtype=torch.bfloat16)
    out, lse = oracle.attn_ref(z, z, z, True, 1.0)
    assert out.shape == (1, 2, 0, 8) and lse.shape == (1, 2, 0)


# --------------------------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows(causal):
    """Each probability row sums to 1, is zero on masked keys and positive on visible ones,
    equals exp(s_ij - LSE_i), and O = P V."""
    g = torch.Generator().manual_seed(24)
    B, Hq, Hkv, N, D = 1, 4, 1, 19, 32
    q, k, v = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D)
    scale = 1 / math.sqrt(D)
    out, lse, p = oracle.attn_probs(q, k, v, causal, scale)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    _close(p.sum(axis=-1), np.ones((B, Hq, N)))
    for h in range(Hq):
        s = scale * (qd[0, h] @ kd[0, 0].T)
        vis = np.tril(np.ones((N, N), bool)) if causal else np.ones((N, N), bool)
        assert np.all(p[0, h][~vis] == 0.0) and np.all(p[0, h][vis] > 0.0)
        _close(p[0, h][vis], np.exp(s - lse[0, h][:, None])[vis])
        _close(out[0, h], p[0, h] @ vd[0, 0])


def test_shift_invariance_in_keys():
    """K' = K + 1 u^T (the same u added to every key) leaves O unchanged and adds
    sm_scale * q_i.u to LSE_i.  Integer inputs keep K' exact in bf16."""
    g = torch.Generator().manual_seed(25)
    B, Hq, Hkv, N, D = 1, 2, 1, 23, 8
    q = torch.randint(-3, 4, (B, Hq, N, D), generator=g).to(torch.bfloat16)
    k = torch.randint(-3, 4, (B, Hkv, N, D), generator=g).to(torch.bfloat16)
    v = _randn(g, B, Hkv, N, D)
    u = torch.randint(-2, 3, (D,), generator=g).to(torch.bfloat16)
    k2 = (k.float() + u.float()).to(torch.bfloat16)
    assert torch.equal(k2.float(), k.float() + u.float())
    for causal in (False, True):
        o1, l1 = oracle.attn_ref(q, k, v, causal, 0.25)
        o2, l2 = oracle.attn_ref(q, k2, v, causal, 0.25)
        _close(o2, o1, 1e-11)
        _close(l2, l1 + 0.25 * (_f64(q) @ _f64(u)), 1e-11)


def test_affine_in_values():
    """V' = a V + b gives O' = a O + b (probability rows sum to 1)."""
    g = torch.Generator().manual_seed(26)
    B, Hq, Hkv, N, D = 2, 2, 2, 17, 16
    q, k = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D)
    v = torch.randint(-4, 5, (B, Hkv, N, D), generator=g).to(torch.bfloat16)
    v2 = (2.0 * v.float() + 1.0).to(torch.bfloat16)
    assert torch.equal(v2.float(), 2.0 * v.float() + 1.0)
    for causal in (False, True):
        o1, l1 = oracle.attn_ref(q, k, v, causal, 0.2)
        o2, l2 = oracle.attn_ref(q, k, v2, causal, 0.2)
        _close(o2, 2.0 * o1 + 1.0, 1e-11)
        assert np.array_equal(l1, l2)


# --------------------------------------------------------------------------------------------
# The blockwise online-softmax recurrence equals the dense definition
# ("Attention Kernel 实现与正确性验证" section 1.1: block-wise evaluation is equivalent to the
#  full-sequence softmax; section 1.2 and "Triton-CUDA Attention", online softmax: running max
#  m_i, running sum l_i rescaled by alpha = exp(m_old - m_new), accumulator rescaled by alpha,
#  final division by l_i; "Flash Attention 与 Kernel 优化": LSE = m_i + log l_i).
# --------------------------------------------------------------------------------------------
def _online_softmax_rows(qd, kd, vd, scale, causal, block):
    """fp64 restatement of the pages' blockwise recurrence for one head (no tiling of Q)."""
    N, D = qd.shape
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    acc = np.zeros((N, D))
    for start in range(0, N, block):
        stop = min(start + block, N)
        s = scale * (qd @ kd[start:stop].T)
        if causal:
            rows = np.arange(N)[:, None]
            cols = np.arange(start, stop)[None, :]
            s = np.where(rows >= cols, s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        alpha = np.exp(m - m_new)
        p = np.exp(s - m_new[:, None])
        l = l * alpha + p.sum(axis=1)
        acc = acc * alpha[:, None] + p @ vd[start:stop]
        m = m_new
    return acc / l[:, None], m + np.log(l)


@pytest.mark.parametrize("block", [1, 7, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_recurrence_equals_dense(block, causal):
    g = torch.Generator().manual_seed(27)
    B, Hq, Hkv, N, D = 1, 4, 2, 150, 32
    q, k, v = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D)
    scale = 1 / math.sqrt(D)
    out, lse = oracle.attn_ref(q, k, v, causal, scale)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    for h in range(Hq):
        hk = h * Hkv // Hq
        o_ref, l_ref = _online_softmax_rows(qd[0, h], kd[0, hk], vd[0, hk], scale, causal, block)
        _close(out[0, h], o_ref)
        _close(lse[0, h], l_ref)


# --------------------------------------------------------------------------------------------
# GQA brute force ("Triton-CUDA Attention", GQA variant: integer division, never a modulus)
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_heads(causal):
    g = torch.Generator().manual_seed(28)
    B, Hq, Hkv, N, D = 2, 8, 2, 33, 16
    q, k, v = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D)
    grp = Hq // Hkv
    k_rep = k.repeat_interleave(grp, dim=1).contiguous()
    v_rep = v.repeat_interleave(grp, dim=1).contiguous()
    o_gqa, l_gqa = oracle.attn_ref(q, k, v, causal, 0.25)
    o_mha, l_mha = oracle.attn_ref(q, k_rep, v_rep, causal, 0.25)
    assert np.array_equal(o_gqa, o_mha) and np.array_equal(l_gqa, l_mha)
    # the interleaved (modulus) map would differ: this is the mistake the pages warn about
    k_mod = k.repeat(1, grp, 1, 1).contiguous()
    v_mod = v.repeat(1, grp, 1, 1).contiguous()
    o_bad, _ = oracle.attn_ref(q, k_mod, v_mod, causal, 0.25)
    assert not np.allclose(o_bad, o_gqa)


def test_mqa_is_gqa_with_one_kv_head():
    g = torch.Generator().manual_seed(29)
    B, Hq, N, D = 1, 5, 20, 16
    q, k, v = _randn(g, B, Hq, N, D), _randn(g, B, 1, N, D), _randn(g, B, 1, N, D)
    o1, l1 = oracle.attn_ref(q, k, v, False, 0.25)
    o2, l2 = oracle.attn_ref(q, k.expand(B, Hq, N, D).contiguous(),
                             v.expand(B, Hq, N, D).contiguous(), False, 0.25)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# --------------------------------------------------------------------------------------------
# A textbook library routine on tiny inputs: torch float64 softmax and logsumexp
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(1, 2, 1, 9, 8), (2, 4, 2, 31, 64), (1, 3, 3, 64, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_float64_softmax(shape, causal):
    B, Hq, Hkv, N, D = shape
    g = torch.Generator().manual_seed(30 + N)
    q, k, v = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D)
    scale = 1 / math.sqrt(D)
    out, lse = oracle.attn_ref(q, k, v, causal, scale)
    grp = Hq // Hkv
    qd = q.double()
    kd = k.double().repeat_interleave(grp, dim=1)
    vd = v.double().repeat_interleave(grp, dim=1)
    s = scale * (qd @ kd.transpose(-1, -2))
    if causal:
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    _close(out, (torch.softmax(s, dim=-1) @ vd).numpy())
    _close(lse, torch.logsumexp(s, dim=-1).numpy())


def test_row_subset_matches_full():
    g = torch.Generator().manual_seed(31)
    B, Hq, Hkv, N, D = 2, 4, 2, 70, 32
    q, k, v = _randn(g, B, Hq, N, D), _randn(g, B, Hkv, N, D), _randn(g, B, Hkv, N, D)
    rows = torch.randint(0, N, (B, Hq, 9), generator=g).numpy().astype(np.int32)
    for causal in (False, True):
        o_full, l_full = oracle.attn_ref(q, k, v, causal, 0.2)
        o_sub, l_sub = oracle.attn_ref(q, k, v, causal, 0.2, rows=rows)
        for b in range(B):
            for h in range(Hq):
                assert np.array_equal(o_sub[b, h], o_full[b, h, rows[b, h]])
                assert np.array_equal(l_sub[b, h], l_full[b, h, rows[b, h]])


def test_threading_does_not_change_results():
    g = torch.Generator().manual_seed(32)
    q, k, v = _randn(g, 1, 4, 40, 16), _randn(g, 1, 2, 40, 16), _randn(g, 1, 2, 40, 16)
    o1, l1 = oracle.attn_ref(q, k, v, True, 0.25, n_threads=1)
    o7, l7 = oracle.attn_ref(q, k, v, True, 0.25, n_threads=7)
    assert np.array_equal(o1, o7) and np.array_equal(l1, l7)


def test_rejects_bad_arguments():
    z = torch.zeros(1, 3, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.attn_ref(z, z[:, :2], z[:, :2], False, 1.0)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attn_ref(z, z, z, False, 1.0, rows=np.full((1, 3, 1), 4, np.int32))  # row >= N
