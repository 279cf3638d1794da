// attn_fwd_d256_kernel.cuh - the exact-attention forward for head dimensions 136..256 (sm_103a).
//
// Same computation as attn_fwd_kernel ("Attention Kernel 实现与正确性验证", walkerchi.com,
// section 1.2: scores, online softmax, P.V, O/l and LSE; GQA head map, top-left causal mask), for
// the wide heads the robustness row asks for ("Triton-CUDA Attention", skillmd.com, pads D to a
// power of two; D is zero-padded to 256 here by the TMA).  At D = 256 one Q tile's fp32 output
// already takes 256 TMEM columns, so a CTA holds one 128-row Q tile instead of two:
//   TMEM (512 columns): S[2] (128 each, double-buffered: S(j+2) forms as soon as the softmax
//   has read S(j)) | O (256).
//   Shared memory: Q (4 panels, 64 KiB, loaded once, reused to stage O), a 4-slot ring of 16 KiB
//   K panels (128 keys x 64 columns; S accumulates over the four panels of a key tile, issued
//   panel by panel, each slot refilled as soon as its MMAs have read it), P (bf16, two 128B-
//   swizzled 128 x 64 panels, the K-major A operand of P.V), V (4 panels, 64 KiB, the MN-major
//   B operand of one N=256 MMA per 16 keys).
// Warps: 0-3 softmax (one row per thread), 4 issues S, 5 issues P.V, 6 loads (lane p < 4: Q
// panel p and K panel p of every key tile, in K slot p; lane 4+p: V panel p).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"
#include "ptx.cuh"

namespace gb300attn {

constexpr int kW256Threads = 224;
constexpr int kW256MmaS = 4, kW256MmaPV = 5, kW256Load = 6;

struct Fwd256Smem {
    static constexpr int kPanel = 128 * 128;  // 128 rows x 64 bf16
    static constexpr int kKSlots = 4;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + 4 * kPanel;
    static constexpr int kP = kK + kKSlots * kPanel;
    static constexpr int kV = kP + 2 * kPanel;
    static constexpr int kBars = kV + 4 * kPanel;
    static constexpr int kBarQ = 0;
    static constexpr int kBarKFull = 1;                    // [kKSlots]
    static constexpr int kBarKEmpty = kBarKFull + kKSlots;  // [kKSlots]
    static constexpr int kBarVFull = kBarKEmpty + kKSlots;
    static constexpr int kBarVEmpty = kBarVFull + 1;
    static constexpr int kBarSFull = kBarVEmpty + 1;  // [2]
    static constexpr int kBarPFull = kBarSFull + 2;   // [2] (count 128)
    static constexpr int kBarPvDone = kBarPFull + 2;  // [2]
    static constexpr int kBarSFree = kBarPvDone + 2;  // [2] the softmax has read S (count 128)
    static constexpr int kNumBars = kBarSFree + 2;
    static constexpr int kTmemSlot = kBars + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 232448, "D=256 forward shared memory exceeds the per-block limit");
};

__global__ void __launch_bounds__(kW256Threads, 1)
    attn_fwd_d256_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ CUtensorMap tmap_o, const AttnParams p,
                         unsigned int* status_word) {
    using L = Fwd256Smem;
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0);   // Q (K-major) x K (K-major)
    constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 1);  // P (TMEM) x V (MN-major)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    auto bar = [=](int i) -> uint32_t { return sbase + L::kBars + 8u * i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // work: blocks of kv_block (batch, KV head) pairs whose K/V fit in L2 together; within a
    // block, Q tiles heaviest (latest) first, then the KV heads, then the query heads of each
    const int item = static_cast<int>(blockIdx.x);
    const int per_kv = p.n_tiles * p.group;
    const int blk = item / (p.kv_block * per_kv);
    const int in_blk = item % (p.kv_block * per_kv);
    const int kvs = min(p.kv_block, p.B * p.Hkv - blk * p.kv_block);
    const int bh_kv = blk * p.kv_block + (in_blk % (kvs * p.group)) / p.group;
    const int m_tile = p.n_tiles - 1 - in_blk / (kvs * p.group);
    const int b = bh_kv / p.Hkv, hkv = bh_kv % p.Hkv;
    const int hq = hkv * p.group + in_blk % p.group;
    const int n_kv = p.causal ? m_tile + 1 : p.n_tiles;  // key tiles 0 .. n_kv-1

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kBarQ), 4);  // one arrive (+ tx) per Q panel
        for (int s = 0; s < L::kKSlots; ++s) {
            mbar_init(bar(L::kBarKFull + s), 1);
            mbar_init(bar(L::kBarKEmpty + s), 1);
        }
        mbar_init(bar(L::kBarVFull), 4);  // one arrive (+ tx) per V panel
        mbar_init(bar(L::kBarVEmpty), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(L::kBarSFull + i), 1);
            mbar_init(bar(L::kBarPFull + i), 128);
            mbar_init(bar(L::kBarPvDone + i), 1);
            mbar_init(bar(L::kBarSFree + i), 128);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kW256MmaS) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto t_s = [=](int j) { return tmem + (j & 1) * 128; };
    const uint32_t t_o = tmem + 256;

    if (warp == kW256Load) {
        // One thread's bulk tensor copies are processed one after another (~29 bytes per cycle
        // per SM from one issuing thread), so every 16 KiB panel stream has its own lane.
        static_assert(L::kKSlots == 4, "K panel p of every key tile goes to slot p");
        static_assert(L::kBarVFull < 32, "load barriers must fit the ArmedPhases mask");
        ArmedPhases armed;  // this lane's loads (by barrier index), drained after an abort
        if (lane < 4) {  // Q panel `lane` once, then K panel `lane` of every key tile
            const int pn = lane;
            if (pn == 0) {
                tma_prefetch_desc(&tmap_q);
                tma_prefetch_desc(&tmap_k);
            }
            mbar_arrive_expect_tx(bar(L::kBarQ), L::kPanel);
            armed.arm(L::kBarQ, 0u);
            tma_load_4d(sbase + L::kQ + pn * L::kPanel, &tmap_q, bar(L::kBarQ), pn * 64,
                        m_tile * 128, hq, b);
            for (int j = 0; j < n_kv; ++j) {
                if (!mbar_wait_bounded<true>(bar(L::kBarKEmpty + pn), (j & 1) ^ 1u, abort_flag,
                                             status_word))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarKFull + pn), L::kPanel);
                armed.arm(L::kBarKFull + pn, static_cast<uint32_t>(j));
                tma_load_4d(sbase + L::kK + pn * L::kPanel, &tmap_k, bar(L::kBarKFull + pn),
                            pn * 64, j * 128, hkv, b);
            }
        } else if (lane < 8) {  // V panel lane-4 of every key tile, once P.V(j-1) has read V
            const int pn = lane - 4;
            if (pn == 0) tma_prefetch_desc(&tmap_v);
            for (int j = 0; j < n_kv; ++j) {
                if (!mbar_wait_bounded<true>(bar(L::kBarVEmpty), (j & 1) ^ 1u, abort_flag,
                                             status_word))
                    break;
                mbar_arrive_expect_tx(bar(L::kBarVFull), L::kPanel);
                armed.arm(L::kBarVFull, static_cast<uint32_t>(j));
                tma_load_4d(sbase + L::kV + pn * L::kPanel, &tmap_v, bar(L::kBarVFull), pn * 64,
                            j * 128, hkv, b);
            }
        }
        if (*abort_flag) armed.drain(bar(0), globaltimer_ns() + kDrainLimitNs);
        __syncwarp();
    } else if (warp == kW256MmaS) {
        // S(j) = Q K_j^T into buffer j&1, once the softmax has read S(j-2).  (The issuers' and
        // the softmax warps' waits suspend instead of polling, leaving the issue slots of their
        // SM sub-partitions to the softmax warps: measured 2 % faster.)
        bool ok = mbar_wait_warp<true>(bar(L::kBarQ), 0, abort_flag, status_word);
        for (int j = 0; ok && j < n_kv; ++j) {
            if (j >= 2) {
                ok = mbar_wait_warp<true>(bar(L::kBarSFree + (j & 1)), ((j - 2) >> 1) & 1,
                                          abort_flag, status_word);
                if (!ok) break;
                tc_fence_after();
            }
            // panel by panel: each panel's MMAs start as soon as it lands, and its slot is
            // released as soon as they have read it
            for (int pn = 0; ok && pn < 4; ++pn) {
                const int k = 4 * j + pn;
                ok = mbar_wait_warp<true>(bar(L::kBarKFull + k % L::kKSlots),
                                          (k / L::kKSlots) & 1, abort_flag, status_word);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kp = sbase + L::kK + (k % L::kKSlots) * L::kPanel;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss_warp(t_s(j),
                                     smem_desc_sw128(sbase + L::kQ + pn * L::kPanel + kk * 32, 16, 1024),
                                     smem_desc_sw128(kp + kk * 32, 16, 1024), kIdescS,
                                     (pn > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(bar(L::kBarKEmpty + k % L::kKSlots));
            }
            if (!ok) break;
            mma_commit_warp(bar(L::kBarSFull + (j & 1)));
        }
        __syncwarp();
    } else if (warp == kW256MmaPV) {
        // O += P(j) V_j: A = P from shared memory, B = the four V panels (N = 256)
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            ok = mbar_wait_warp<true>(bar(L::kBarVFull), j & 1, abort_flag, status_word);
            if (ok) ok = mbar_wait_warp<true>(bar(L::kBarPFull + (j & 1)), (j >> 1) & 1,
                                              abort_flag, status_word);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ss_warp(t_o,
                                 smem_desc_sw128(sbase + L::kP + (kk >> 2) * L::kPanel + (kk & 3) * 32,
                                                 16, 1024),
                                 smem_desc_sw128(sbase + L::kV + kk * 2048, L::kPanel, 1024),
                                 kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit_warp(bar(L::kBarPvDone + (j & 1)));
            mma_commit_warp(bar(L::kBarVEmpty));
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps 0-3: row `row` of the Q tile --------------------------
        const int row = warp * 32 + lane;
        const int row_g = m_tile * 128 + row;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float c = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            ok = mbar_wait_warp<true>(bar(L::kBarSFull + (j & 1)), (j >> 1) & 1, abort_flag,
                                      status_word);
            if (!ok) break;
            tc_fence_after();
            float s[128];
            {
                uint32_t r[128];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    tmem_ld32(lane_base + t_s(j) + cc * 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&r[cc * 32]));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(L::kBarSFree + (j & 1)));  // S(j+2) may now be formed over it
#pragma unroll
                for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(r[i]);
            }
            // masks: the causal diagonal tile, or the ragged last key tile
            const bool diag = p.causal && j == m_tile;
            const bool tail = !p.causal && j == p.n_tiles - 1 && (p.N % 128) != 0;
            if (diag || tail) {
                const int lim = diag ? row + 1 : p.N - j * 128;  // first masked key
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= lim) s[i] = -INFINITY;
            }
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
            for (int i = 16; i < 128; i += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[i + k], s[i + 8 + k]);
            const float row_max =
                fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            const float m_cand = row_max * c;
            const float m_new = (m_cand > m + kRescaleThreshold) ? m_cand : m;
            const float alpha = ex2_approx(m - m_new);  // 1 if unchanged, 0 on the first tile
            const bool rescale = j > 0 && __any_sync(0xffffffffu, m_new != m);
            m = m_new;
            const float neg_m = -m;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                float x0, x1;
                ffma2(x0, x1, s[2 * i], s[2 * i + 1], c, c, neg_m, neg_m);
                const float p0 = ex2_approx(x0);
                const float p1 = ex2_approx(x1);
                const int a = (i & 1) * 2;
                fadd2(acc[a], acc[a + 1], acc[a], acc[a + 1], p0, p1);
                pk[i] = pack_bf16x2(p0, p1);
            }
            // P.V(j-1) must have read the previous P (and landed, for the O correction)
            if (j > 0) {
                ok = mbar_wait_warp<true>(bar(L::kBarPvDone + ((j - 1) & 1)),
                                          ((j - 1) >> 1) & 1, abort_flag, status_word);
                if (!ok) break;
                tc_fence_after();
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // keys 64h .. 64h+63 -> panel h, 128B swizzle
                const uint32_t prow = sbase + L::kP + h * L::kPanel + row * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_shared_v4(prow + ((ch ^ (row & 7)) << 4), pk[32 * h + 4 * ch],
                                 pk[32 * h + 4 * ch + 1], pk[32 * h + 4 * ch + 2],
                                 pk[32 * h + 4 * ch + 3]);
            }
            if (rescale) {  // O *= alpha
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + t_o + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tmem_st32(lane_base + t_o + cc * 32, o);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();  // generic-proxy P stores -> the MMA's async reads
            tc_fence_before();
            mbar_arrive(bar(L::kBarPFull + (j & 1)));
            l = l * alpha + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
        }
        // epilogue: O / l -> bf16 -> the Q panels (128B swizzle) -> TMA store; LSE
        if (ok) {
            const int last = n_kv - 1;
            ok = mbar_wait_warp(bar(L::kBarPvDone + (last & 1)), (last >> 1) & 1, abort_flag,
                                status_word);
        }
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.0f / l;
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t o[32];
                tmem_ld32(lane_base + t_o + cc * 32, o);
                tmem_wait_ld();
                const uint32_t prow = sbase + L::kQ + (cc >> 1) * L::kPanel + row * 128;
#pragma unroll
                for (int c16 = 0; c16 < 4; ++c16) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(o[c16 * 8 + 2 * i]) * inv_l,
                                           __uint_as_float(o[c16 * 8 + 2 * i + 1]) * inv_l);
                    const int chunk = (cc & 1) * 4 + c16;
                    st_shared_v4(prow + ((chunk ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
                }
            }
            if (row_g < p.N && ATTN_DCHECK(b < p.B && hq < p.Hq && m_tile < p.n_tiles))
                p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.N + row_g] =
                    (m + __log2f(l)) * 0.69314718055994531f;
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (ok && warp == 0 && lane == 0 && ATTN_DCHECK(b < p.B && hq < p.Hq && m_tile < p.n_tiles)) {
            for (int pn = 0; pn < 4; ++pn)
                tma_store_4d(&tmap_o, sbase + L::kQ + pn * L::kPanel, pn * 64, m_tile * 128, hq, b);
            tma_store_commit_and_wait();
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kW256MmaS) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace gb300attn
