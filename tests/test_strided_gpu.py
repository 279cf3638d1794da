"""GPU parity for strided (non-contiguous) inputs and outputs through attn_fwd_strided: the
[B, N, H, D] layout that projections produce, padded rows and a sliced batch, against the oracle
on contiguous copies."""
import pytest
import torch

import oracle
from exact_attention_forward_attn_gb300 import workloads as wl

from test_parity_gpu import _check

pytestmark = pytest.mark.gpu


def _bnhd(t):
    """The same values stored as [B, N, H, D] and viewed as [B, H, N, D] (non-contiguous)."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _padded(t, pad=8):
    """Rows padded to D + pad elements: a [B, H, N, D] view with row stride D + pad."""
    B, H, N, D = t.shape
    buf = torch.zeros(B, H, N, D + pad, dtype=t.dtype, device=t.device)
    buf[..., :D] = t
    return buf[..., :D]


CASES = [
    ("bnhd", wl.random_case(2, 8, 2, 300, 128, True, 31)),
    ("bnhd", wl.random_case(1, 4, 4, 256, 64, False, 32)),
    ("padded", wl.random_case(1, 4, 1, 200, 128, False, 33)),
    ("mixed", wl.random_case(2, 6, 3, 129, 128, True, 34)),
    ("bnhd", wl.random_case(1, 4, 2, 250, 96, True, 36)),
    ("bnhd", wl.random_case(1, 4, 2, 300, 256, True, 37)),
    ("padded", wl.random_case(1, 2, 1, 200, 192, False, 38)),
]


@pytest.mark.parametrize("layout,w", CASES, ids=[f"{a}-{w.name}" for a, w in CASES])
def test_strided_layouts_match_oracle(layout, w, cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    q, k, v = wl.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if layout == "bnhd":
        qd, kd, vd = _bnhd(qd), _bnhd(kd), _bnhd(vd)
        out = _bnhd(torch.empty_like(q, device="cuda"))
    elif layout == "padded":
        qd, kd, vd = _padded(qd), _padded(kd, 16), _padded(vd, 24)
        out = _padded(torch.empty_like(q, device="cuda"), 8)
    else:  # q in [B, N, H, D], k padded, v contiguous, out from a larger batch (sliced)
        qd, kd = _bnhd(qd), _padded(kd)
        big = torch.empty(w.B + 1, w.Hq, w.N, w.D, dtype=torch.bfloat16, device="cuda")
        out = big[1:]
    assert not qd.is_contiguous()
    out, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=out)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out.contiguous(), lse, o_ref, l_ref, f"{layout} {w.name}")


def test_unaligned_stride_is_rejected(cuda_lib):
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(1, 2, 1, 128, 64, False, 35)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    with pytest.raises(attn.AttnError, match="ATTN_ERR_STRIDE"):
        attn.attn_fwd(_padded(q, 4), k, v)  # row stride 68 elements = 136 bytes


def test_offsets_beyond_2_31_elements(cuda_lib):
    """Batch strides of 2^31 + 1024 elements: the second batch of q, k, v and out lies more than
    2^31 elements (4 GiB) past its tensor's base, so every address the TMA maps and the epilogue
    form needs 64-bit arithmetic.  The gap between out's two batches must stay untouched."""
    import exact_attention_forward_attn_gb300 as attn

    w = wl.random_case(2, 4, 2, 300, 128, True, 39)
    q, k, v = wl.make_qkv(w)
    S = (1 << 31) + 1024
    per_b = [t[0].numel() for t in (q, k, v)]
    offs = [0, per_b[0], per_b[0] + per_b[1]]
    # q, k and v share one buffer (inputs may overlap each other); out has its own
    inp = torch.empty(S + sum(per_b), dtype=torch.bfloat16, device="cuda")
    views = []
    for t, off in zip((q, k, v), offs):
        view = inp.as_strided(t.shape, (S, t.shape[2] * t.shape[3], t.shape[3], 1), off)
        view.copy_(t)
        views.append(view)
    obuf = torch.empty(S + per_b[0], dtype=torch.bfloat16, device="cuda")
    sentinel = -7.5
    band = 1 << 20
    obuf[per_b[0]:per_b[0] + band].fill_(sentinel)  # just after batch 0
    obuf[S - band:S].fill_(sentinel)                # just before batch 1
    out = obuf.as_strided(q.shape, (S, q.shape[2] * q.shape[3], q.shape[3], 1), 0)
    out, lse = attn.attn_fwd(*views, causal=w.causal, sm_scale=w.sm_scale, out=out)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert (obuf[per_b[0]:per_b[0] + band] == sentinel).all()
    assert (obuf[S - band:S] == sentinel).all()
    o_ref, l_ref = oracle.attn_ref(q, k, v, w.causal, w.sm_scale)
    _check(out.contiguous(), lse, o_ref, l_ref, f"64-bit offsets {w.name}")
    del views, out, inp, obuf
    torch.cuda.empty_cache()
