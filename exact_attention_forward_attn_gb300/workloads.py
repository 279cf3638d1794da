"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws inputs.  Both the CUDA path and the CPU
oracle receive exactly the bf16 tensors made here.

Recipe (one CPU ``torch.Generator`` per workload, seeded as listed):
  draw ``randn`` float32 in the order Q [B,Hq,N,D], K [B,Hkv,N,D], V [B,Hkv,N,D] from the one
  generator, then round each to bf16 (round-to-nearest-even).  ``sm_scale = 1/sqrt(D)``.

The shapes are the test shapes of "Attention Kernel 实现与正确性验证" (walkerchi.com), section 1.3
(GQA-4, GQA-8, MHA, MQA), a tiny GQA-2 case, an outlier variant of the MHA case that stresses the
running-maximum rescale, and the long-context sweep of section 1.4 (N = 8K..32K) with 8 KV heads.
The pages measure no public dataset; these iid N(0,1) inputs stand in for activations.

Absorbed MLA decode (``MlaWorkload``, the second workload): the DeepSeek-V3 widths of section 2.3
of the same page (d_c = 512 compressed, d_r = 64 RoPE, d_nope = 128, so sm_scale = 1/sqrt(192)),
128 heads, one decode query per head, T cached tokens.  Recipe: one generator per workload, draw
``randn`` float32 q [B, H, d_c + d_r] then kv [B, T, d_c + d_r], round each to bf16.  q stands for
q_nope W_uk concatenated with q_pe, kv for c_kv concatenated with k_pe.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    D: int
    causal: bool
    seed: int
    outlier_seed: int | None = None  # if set: 1% of K entries (seeded positions) scaled by 8
    outlier_frac: float = 0.01
    tags: tuple = field(default_factory=tuple)

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*Hq*N^2*D, halved under the causal mask."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.D
        return f / 2.0 if self.causal else f

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once, O written once (bf16), LSE written (fp32)."""
        return 2 * (2 * self.B * self.Hq * self.N * self.D + 2 * self.B * self.Hkv * self.N * self.D) \
            + 4 * self.B * self.Hq * self.N

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five configurations (C1..C5) plus the outlier variant of C4a.
TINY_NONCAUSAL = Workload("tiny-gqa2", 1, 2, 1, 128, 64, False, 0)
TINY_CAUSAL = Workload("tiny-gqa2-causal", 1, 2, 1, 128, 64, True, 0)
GQA4_CAUSAL = Workload("gqa4-causal-n1024", 2, 32, 8, 1024, 128, True, 1)
GQA8_CAUSAL = Workload("gqa8-causal-n4096", 1, 64, 8, 4096, 128, True, 2)
MHA = Workload("mha-n512", 1, 32, 32, 512, 128, False, 3)
MHA_OUTLIER = Workload("mha-n512-outlier", 1, 32, 32, 512, 128, False, 3, outlier_seed=104)
MQA = Workload("mqa-n512", 1, 16, 1, 512, 128, False, 4)
# Few query heads over a longer sequence: 32 query tiles in all, far fewer than the SMs, so the
# key axis is split (split-KV forward).  Not one of the five configurations; a context workload.
FEWHEADS = Workload("fewheads-n4096", 1, 2, 1, 4096, 128, False, 8)
# Few causal heads over a long sequence: 128 pairs of Q tiles, the split-KV default splits the key
# axis in two (more clusters than fit at once: the workspace path).  A context workload.
FEWHEADS_CAUSAL = Workload("fewheads-causal-n8192", 1, 4, 1, 8192, 128, True, 9)
LONG = {n: Workload(f"long-gqa8-causal-n{n}", 1, 32, 8, n, 128, True, s)
        for n, s in ((8192, 5), (16384, 6), (32768, 7))}

# Wide heads (D = 256, one Q tile per CTA): the robustness row's widest head dimension over a long
# causal sequence.  Not one of the five configurations.
WIDE = Workload("wide-d256-causal-n8192", 1, 16, 4, 8192, 256, True, 9)

CONFIGS = [TINY_NONCAUSAL, TINY_CAUSAL, GQA4_CAUSAL, GQA8_CAUSAL, MHA, MHA_OUTLIER, MQA,
           *LONG.values(), FEWHEADS, FEWHEADS_CAUSAL, WIDE]
BY_NAME = {w.name: w for w in CONFIGS}


@dataclass(frozen=True)
class MlaWorkload:
    name: str
    B: int
    H: int
    T: int
    seed: int
    d_c: int = 512
    d_r: int = 64
    d_nope: int = 128

    @property
    def d_qk(self) -> int:
        return self.d_c + self.d_r

    @property
    def sm_scale(self) -> float:
        """The un-absorbed head width sets the scale: 1/sqrt(d_nope + d_r)."""
        return 1.0 / math.sqrt(self.d_nope + self.d_r)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs of the compressed-space core: scores (2*d_qk) and output (2*d_c) per
        head and token."""
        return 2.0 * self.B * self.H * self.T * (self.d_qk + self.d_c)

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes: the cache and the queries read once (bf16), out_c written
        (bf16), LSE written (fp32)."""
        return 2 * self.B * self.T * self.d_qk + 2 * self.B * self.H * self.d_qk \
            + 2 * self.B * self.H * self.d_c + 4 * self.B * self.H


MLA_TINY = MlaWorkload("mla-tiny", 1, 16, 200, 30)
MLA_RAGGED = MlaWorkload("mla-ragged", 2, 128, 777, 31)
MLA_B1 = {t: MlaWorkload(f"mla-b1-t{t}", 1, 128, t, s) for t, s in ((4096, 32), (16384, 33))}
MLA_B32 = MlaWorkload("mla-b32-t4096", 32, 128, 4096, 34)
MLA_CONFIGS = [MLA_TINY, MLA_RAGGED, *MLA_B1.values(), MLA_B32]


def make_mla(w: MlaWorkload, device="cpu"):
    """bf16 q [B, H, d_c + d_r] and kv [B, T, d_c + d_r] for MLA workload ``w``."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn(w.B, w.H, w.d_qk, generator=g, dtype=torch.float32).to(torch.bfloat16)
    kv = torch.randn(w.B, w.T, w.d_qk, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if device != "cpu":
        q, kv = q.to(device), kv.to(device)
    return q, kv


def make_qkv(w: Workload, device="cpu"):
    """bf16 Q, K, V for workload ``w`` (drawn on the CPU, then moved to ``device``)."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn(w.B, w.Hq, w.N, w.D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(w.B, w.Hkv, w.N, w.D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(w.B, w.Hkv, w.N, w.D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if w.outlier_seed is not None:
        k = _scale_outliers(k, w.outlier_seed, w.outlier_frac)
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def _scale_outliers(k: torch.Tensor, seed: int, frac: float) -> torch.Tensor:
    """Multiply round(frac*numel) distinct, seeded flat positions of K by 8 (exact in bf16)."""
    g = torch.Generator().manual_seed(seed)
    n = k.numel()
    count = int(round(frac * n))
    idx = torch.randperm(n, generator=g)[:count]
    flat = k.reshape(-1).clone()
    flat[idx] = flat[idx] * 8
    return flat.reshape(k.shape)


def sample_rows(w: Workload, per_head: int = 64) -> torch.Tensor:
    """Seeded query rows compared against the oracle at full size: int32 [B, Hq, per_head].

    For head hq the rows are ``randperm(N, seed=5000 + N + hq)[:per_head]`` (the same rows for
    every batch index), sorted ascending.
    """
    per_head = min(per_head, w.N)
    rows = torch.empty(w.B, w.Hq, per_head, dtype=torch.int32)
    for h in range(w.Hq):
        g = torch.Generator().manual_seed(5000 + w.N + h)
        r = torch.randperm(w.N, generator=g)[:per_head].sort().values.to(torch.int32)
        rows[:, h, :] = r
    return rows


def random_case(B, Hq, Hkv, N, D, causal, seed) -> Workload:
    """An ad-hoc seeded workload (used for ragged/edge-case parity tests)."""
    return Workload(f"case-b{B}-hq{Hq}-hkv{Hkv}-n{N}-d{D}-{'c' if causal else 'nc'}-s{seed}",
                    B, Hq, Hkv, N, D, causal, seed)
