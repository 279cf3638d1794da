"""Pins for the absorbed-MLA decode oracle (``oracle.mla_decode_ref``), independent of it.

The strongest pin is the page's own claim ("Attention Kernel 实现与正确性验证", walkerchi.com,
section 2.2): absorbing W_uk into the query and applying W_uv after the attention gives the same
result as reconstructing full K and V from c_kv and running standard attention.  The un-absorbed
side is written with torch float64 library routines (einsum, softmax, logsumexp), so a dropped
RoPE term, a wrong scale or a transposed operand in the oracle fails it.  Closed forms and an
invariance cover the degenerate cases.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _naive(c_kv, k_pe, q_nope, q_pe, w_uk, w_uv):
    """Standard attention on K and V rebuilt from the compressed cache (float64)."""
    H = w_uk.shape[0]
    k_nope = torch.einsum("btc,hdc->bhtd", c_kv, w_uk)
    v = torch.einsum("btc,hvc->bhtv", c_kv, w_uv)
    k = torch.cat([k_nope, k_pe.unsqueeze(1).expand(-1, H, -1, -1)], dim=-1)
    q = torch.cat([q_nope, q_pe], dim=-1)  # [B, H, d]
    s = torch.einsum("bhd,bhtd->bht", q, k) / math.sqrt(q.shape[-1])
    return torch.einsum("bht,bhtv->bhv", torch.softmax(s, dim=-1), v), torch.logsumexp(s, dim=-1)


def _absorbed(c_kv, k_pe, q_nope, q_pe, w_uk, w_uv, n_threads=0):
    q_abs = torch.einsum("bhd,hdc->bhc", q_nope, w_uk)
    q = torch.cat([q_abs, q_pe], dim=-1)
    kv = torch.cat([c_kv, k_pe], dim=-1)
    scale = 1.0 / math.sqrt(q_nope.shape[-1] + q_pe.shape[-1])
    out_c, lse = oracle.mla_decode_ref(q, kv, c_kv.shape[-1], scale, n_threads=n_threads)
    return torch.einsum("bhc,hvc->bhv", torch.from_numpy(out_c), w_uv).numpy(), lse


@pytest.mark.parametrize("dims", [
    # (B, H, T, d_c, d_r, d_nope, d_v)
    (2, 4, 23, 32, 8, 16, 16),
    (1, 8, 9, 512, 64, 128, 128),   # the page's DeepSeek-V3 widths, few heads and tokens
    (3, 2, 1, 16, 4, 8, 12),
])
def test_absorbed_equals_naive_reconstruction(dims):
    B, H, T, d_c, d_r, d_nope, d_v = dims
    g = torch.Generator().manual_seed(70 + T)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)  # noqa: E731
    c_kv, k_pe = r(B, T, d_c), r(B, T, d_r)
    q_nope, q_pe = r(B, H, d_nope), r(B, H, d_r)
    w_uk, w_uv = r(H, d_nope, d_c) / math.sqrt(d_c), r(H, d_v, d_c) / math.sqrt(d_c)
    want_o, want_l = _naive(c_kv, k_pe, q_nope, q_pe, w_uk, w_uv)
    got_o, got_l = _absorbed(c_kv, k_pe, q_nope, q_pe, w_uk, w_uv)
    np.testing.assert_allclose(got_o, want_o.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(got_l, want_l.numpy(), rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_row():
    g = torch.Generator().manual_seed(71)
    q = torch.randn(2, 3, 40, generator=g, dtype=torch.float64)
    kv = torch.randn(2, 1, 40, generator=g, dtype=torch.float64)
    out, lse = oracle.mla_decode_ref(q, kv, 32, 0.2)
    for b in range(2):
        np.testing.assert_array_equal(out[b], np.broadcast_to(kv[b, 0, :32].numpy(), (3, 32)))
        np.testing.assert_allclose(lse[b], 0.2 * (q[b] @ kv[b, 0]).numpy(), rtol=0, atol=1e-13)


def test_identical_tokens_give_uniform_weights():
    g = torch.Generator().manual_seed(72)
    T = 37
    q = torch.randn(1, 4, 24, generator=g, dtype=torch.float64)
    row = torch.randn(24, generator=g, dtype=torch.float64)
    kv = row.expand(1, T, 24).contiguous()
    out, lse = oracle.mla_decode_ref(q, kv, 16, 0.3)
    np.testing.assert_allclose(out[0], np.broadcast_to(row[:16].numpy(), (4, 16)), atol=1e-14)
    np.testing.assert_allclose(lse[0], 0.3 * (q[0] @ row).numpy() + math.log(T), atol=1e-12)


def test_shift_of_the_rope_part_only_moves_lse():
    """Adding u to every token's k_pe adds sm_scale * q_pe.u to all scores of a head: the
    weights and out_c stay, LSE moves by that constant.  A shift of c_kv would move out_c too, so
    this separates the two parts of each cached row."""
    g = torch.Generator().manual_seed(73)
    d_c, d_r, scale = 20, 6, 0.25
    q = torch.randn(2, 3, d_c + d_r, generator=g, dtype=torch.float64)
    kv = torch.randn(2, 15, d_c + d_r, generator=g, dtype=torch.float64)
    u = torch.randn(d_r, generator=g, dtype=torch.float64)
    kv2 = kv.clone()
    kv2[:, :, d_c:] += u
    o1, l1 = oracle.mla_decode_ref(q, kv, d_c, scale)
    o2, l2 = oracle.mla_decode_ref(q, kv2, d_c, scale)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, scale * (q[:, :, d_c:] @ u).numpy(), atol=1e-12)


def test_bf16_inputs_are_widened_exactly_and_threads_do_not_matter():
    g = torch.Generator().manual_seed(74)
    q = torch.randn(2, 5, 72, generator=g).to(torch.bfloat16)
    kv = torch.randn(2, 33, 72, generator=g).to(torch.bfloat16)
    a = oracle.mla_decode_ref(q, kv, 64, 0.125, n_threads=1)
    b = oracle.mla_decode_ref(q.double(), kv.double(), 64, 0.125, n_threads=3)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_rejects_bad_arguments():
    q = np.zeros((1, 2, 8))
    with pytest.raises(ValueError):
        oracle.mla_decode_ref(q, np.zeros((1, 0, 8)), 4, 1.0)  # no cached token
    with pytest.raises(ValueError):
        oracle.mla_decode_ref(q, np.zeros((1, 3, 9)), 4, 1.0)  # widths differ
