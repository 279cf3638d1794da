"""GPU parity of the backward (attn_bwd, by recompute) against the fp64 oracle's gradients.

Tolerance: the pages state none for the backward.  The GPU path rounds P and dS to bf16 before
the MMAs (as the pages' forward rounds P before P.V), forms dO.O from the bf16 O, and stores bf16
gradients; each of these is a relative rounding of 2^-9, and dS = P (dP - dO.O) can cancel.  The
bound used, per gradient tensor G with reference R, is
    |G - R| <= 2e-2 * max|R| + 2e-2 * |R|      element-wise,
i.e. the forward's bf16 tolerance with the absolute part scaled to the tensor's magnitude.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _grad_check(name, g, ref):
    g = g.float().cpu().numpy().astype(np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 1.0
    err = np.abs(g - ref)
    bad = err > 2e-2 * scale + 2e-2 * np.abs(ref)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    assert not bad.any(), (f"{name}: {int(bad.sum())}/{bad.size} out of tolerance; "
                           f"max err {err.max():.3e} (max|ref| {scale:.3e})")
    return float(err.max() / max(scale, 1e-30))


def _dout(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(w.B, w.Hq, w.N, w.D, generator=g).to(torch.bfloat16)


CASES = [
    wl.TINY_NONCAUSAL, wl.TINY_CAUSAL,
    wl.random_case(2, 4, 2, 300, 128, True, 41),
    wl.random_case(1, 4, 4, 256, 64, False, 42),
    wl.random_case(1, 6, 2, 129, 96, True, 43),
    wl.random_case(2, 4, 1, 200, 128, False, 44),
    wl.random_case(1, 8, 2, 640, 128, True, 45),
    # GQA-8 over 8 key tiles: 64 steps per dK/dV CTA, so every operand ring wraps many times
    wl.random_case(1, 8, 1, 1024, 128, True, 47),
    wl.random_case(1, 4, 1, 1000, 64, False, 48),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_backward_matches_oracle(w, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    q, k, v = wl.make_qkv(w)
    do = _dout(w, 900 + w.N)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, out, lse, dod, causal=w.causal, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rq, rk, rv = oracle.attn_bwd_ref(q, k, v, do, w.causal, w.sm_scale)
    e = [_grad_check(n, g, r) for n, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv))]
    print(f"{w.name}: relative max errors dq {e[0]:.2e} dk {e[1]:.2e} dv {e[2]:.2e}")


def test_autograd_function(cuda_lib):
    """FlashAttention.apply(q, k, v, is_causal) runs our forward and backward under autograd."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(1, 4, 2, 256, 128, True, 46)
    q, k, v = wl.make_qkv(w)
    do = _dout(w, 946)
    qd = q.cuda().requires_grad_()
    kd = k.cuda().requires_grad_()
    vd = v.cuda().requires_grad_()
    out = attn.FlashAttention.apply(qd, kd, vd, True)
    out.backward(do.cuda())
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attn_bwd_ref(q, k, v, do, True, w.sm_scale)
    _grad_check("dq", qd.grad, rq)
    _grad_check("dk", kd.grad, rk)
    _grad_check("dv", vd.grad, rv)
