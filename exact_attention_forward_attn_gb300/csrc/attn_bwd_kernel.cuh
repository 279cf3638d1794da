// attn_bwd_kernel.cuh - backward of the exact-attention forward for sm_103a (tcgen05 + TMA).
//
// The gradients are recomputed from the saved log-sum-exp instead of a stored probability matrix
// ("Attention Kernel 实现与正确性验证", walkerchi.com, section 1.1, third idea; "Flash Attention 与
// Kernel 优化", fangpin.github.io, autograd and backward: rebuild s, the causal mask and p, then
// dv, dp, ds, dq, dk).  For query row i of head (b, hq) and visible key j of its KV head:
//   p_ij  = exp(sm_scale q_i.k_j - LSE_i)      dp_ij = dO_i.v_j      Delta_i = dO_i.O_i
//   ds_ij = p_ij (dp_ij - Delta_i)
//   dQ_i  = sm_scale sum_j ds_ij k_j,  dK_j = sm_scale sum_(hq,i) ds_ij q_i,  dV_j = sum_(hq,i) p_ij dO_i
// (Delta_i = sum_j p_ij dp_ij = dO_i . O_i; the kernels use the second form with the stored O.)
//
// Three kernels:
//   attn_bwd_delta_kernel   Delta = rowsum(dO * O), one warp per row.
//   attn_bwd_dkdv_kernel    one CTA per (b, KV head, 128-key tile j): K_j, V_j stay in smem; for
//                           every query head of the group and every query tile i (i >= j under
//                           the causal mask) it forms S^T = K_j Q_i^T and dP^T = V_j dO_i^T,
//                           P^T (bf16, in shared memory) and dS^T (bf16, in TMEM over dP^T),
//                           and accumulates dV += P^T dO_i and dK += dS^T Q_i in TMEM.
//   attn_bwd_dq_kernel      persistent; one work item per (b, query head, 128-row tile i):
//                           S = Q_i K_j^T, dP = dO_i V_j^T, dS (bf16 in TMEM over S),
//                           dQ += dS K_j.
// Zero-filled rows past N contribute nothing: a padded query has dO = 0 and Delta = 0 (so its
// ds and its dV term vanish), a padded key has K = V = 0 (so its dQ term vanishes) and its own
// dK/dV rows are never stored.  Only the causal diagonal tile needs a mask.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"
#include "ptx.cuh"

namespace gb300attn {

struct BwdParams {
    int B, Hq, Hkv, N;
    int group;         // Hq / Hkv
    int causal;
    int n_tiles;       // ceil(N / 128)
    float scale_log2;  // sm_scale * log2(e)
    float sm_scale;
    const float* lse;    // [B, Hq, N] natural-log LSE from the forward
    const float* delta;  // [B, Hq, N] dO . O
    // dQ kernel (persistent): its work items, its claim counter (zero at launch; nullptr: the
    // static schedule), and dQ
    // [B, Hq, N, d_out] bf16, contiguous
    int items;
    unsigned int* sched;
    __nv_bfloat16* dq;
    int d_out;
};

// Warps 0-7 elementwise: warp w serves TMEM lanes 32(w%4) .. 32(w%4)+31 (its quarter) and the
// 64 columns 64(w/4) .. 64(w/4)+63 of the 128-wide S / dP tile, so every lane quarter has two
// warps.  Warps 8 and 10 issue the MMAs of two independent accumulator chains, warp 9 loads.
constexpr int kBwdMmaWarp = 8;
constexpr int kBwdLoadWarp = 9;
constexpr int kBwdMmaWarpB = 10;
constexpr int kBwdThreads = 352;
constexpr int kBwdEwThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Delta_i = dO_i . O_i (fp32 sum of bf16 products); one warp per row, D <= 128 columns.
__global__ void __launch_bounds__(256)
    attn_bwd_delta_kernel(const __nv_bfloat16* __restrict__ out,
                          const __nv_bfloat16* __restrict__ dout, float* __restrict__ delta,
                          long long rows, int D) {
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    griddep_launch_dependents();  // the dK/dV kernel waits for Delta itself
    if (row >= rows) return;
    const __nv_bfloat16* o = out + row * D;
    const __nv_bfloat16* g = dout + row * D;
    float acc = 0.f;
    for (int d = lane; d < D; d += 32) acc += __bfloat162float(o[d]) * __bfloat162float(g[d]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0 && ATTN_DCHECK(row < rows)) delta[row] = acc;
}

// dK/dV layout: K_j, V_j resident; a 3-slot ring of Q_i (read by S^T(i), formed a step ahead,
// and by dK(i), issued last, so the third slot lets Q_(i+2) load while dK(i) is pending); one dO_i
// buffer (read by dP^T(i) and dV(i), both early in the step); P^T (bf16, two 128B-swizzled
// 128 x 64 panels) so that S^T(i+1) can be formed while P^T(i) is still being written and read;
// LSE/Delta vectors in two slots.  This fills the 227 KiB limit, so the layout leaves no slack for
// aligning the base: the kernel checks that the dynamic shared memory starts 1024-aligned and
// reports kDevSmemAlign otherwise.
template <int D>
struct DkdvSmem {
    static constexpr int kPanelBytes = 128 * 64 * 2;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kQSlots = 3;
    static constexpr int kRes0 = 0;                  // K_j
    static constexpr int kRes1 = kTileBytes;         // V_j
    static constexpr int kQ = 2 * kTileBytes;        // Q ring
    static constexpr int kDO = kQ + kQSlots * kTileBytes;
    static constexpr int kPt = kDO + kTileBytes;
    static constexpr int kVec = kPt + 2 * kPanelBytes;  // lse2/delta [slot][2][128]
    static constexpr int kBars = kVec + 2 * 2 * 128 * 4;
    static constexpr int kBarRes = 0;
    static constexpr int kBarQFull = 1;                     // [kQSlots]
    static constexpr int kBarQEmpty = kBarQFull + kQSlots;  // [kQSlots]
    static constexpr int kBarDoFull = kBarQEmpty + kQSlots;
    static constexpr int kBarDoEmpty = kBarDoFull + 1;      // both chains release it
    static constexpr int kBarVecFull = kBarDoEmpty + 1;     // [2] (the producer's 32 lanes)
    static constexpr int kBarVecFree = kBarVecFull + 2;     // [2] (the elementwise threads)
    static constexpr int kBarS = kBarVecFree + 2;
    static constexpr int kBarSFree = kBarS + 1;
    static constexpr int kBarDP = kBarSFree + 1;
    static constexpr int kBarP = kBarDP + 1;
    static constexpr int kBarPFree = kBarP + 1;
    static constexpr int kBarDS = kBarPFree + 1;
    static constexpr int kBarDone = kBarDS + 1;
    static constexpr int kNumBars = kBarDone + 1;
    static constexpr int kTmemSlot = kBars + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes;
    static_assert(kAlloc <= 232448, "dK/dV shared memory exceeds the per-block limit");
};

// A 128 x 128 bf16 operand (dS^T, dS) is packed into TMEM by the two column halves' warps,
// each over the first 32 of its own 64 fp32 columns: K-step kk (16 columns of the operand)
// starts at this column offset.
__device__ __forceinline__ uint32_t packed_col(int kk) {
    return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8);
}

// Stage 32-column chunks [cc_begin, cc_end) of a 128 x D fp32 accumulator row (this thread's TMEM
// lane) as bf16 into a 128B-swizzled panel pair at `stage` (the layout the 4-D TMA store expects).
template <int D>
__device__ __forceinline__ void stage_rows_bf16(uint32_t stage, uint32_t taddr, int row,
                                                float mul, int cc_begin, int cc_end) {
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
        if (cc < cc_begin || cc >= cc_end) continue;
        uint32_t r[32];
        tmem_ld32(taddr + cc * 32, r);
        tmem_wait_ld();
        const int panel = cc >> 1;
#pragma unroll
        for (int c16 = 0; c16 < 4; ++c16) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = pack_bf16x2(__uint_as_float(r[c16 * 8 + 2 * i]) * mul,
                                   __uint_as_float(r[c16 * 8 + 2 * i + 1]) * mul);
            const int chunk = (cc & 1) * 4 + c16;
            st_shared_v4(stage + panel * (128 * 128) + row * 128 + ((chunk ^ (row & 7)) << 4),
                         w[0], w[1], w[2], w[3]);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// dK, dV
// ------------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ CUtensorMap tmap_do,
                         const __grid_constant__ CUtensorMap tmap_dk,
                         const __grid_constant__ CUtensorMap tmap_dv, const BwdParams p,
                         unsigned int* status_word) {
    using L = DkdvSmem<D>;
    constexpr int kPanels = D / 64;
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0);  // K-major x K-major
    constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, 1);  // (TMEM or K-major) x MN-major
    extern __shared__ __align__(1024) uint8_t dkdv_smem[];
    uint8_t* smem = dkdv_smem;
    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {  // uniform over the CTA: every thread leaves before any barrier
        if (threadIdx.x == 0) atomicOr(status_word, kDevSmemAlign);
        return;
    }
    auto bar = [=](int i) -> uint32_t { return sbase + L::kBars + 8u * i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_launch_dependents();  // the dQ kernel is launched right after this one

    // work: key tile j (smallest, i.e. heaviest under the causal mask, first), then (b, h_kv)
    const int bkv_count = p.B * p.Hkv;
    const int j = static_cast<int>(blockIdx.x / bkv_count);
    const int bh_kv = static_cast<int>(blockIdx.x % bkv_count);
    const int b = bh_kv / p.Hkv, hkv = bh_kv % p.Hkv;
    const int i_first = p.causal ? j : 0;
    const int per_head = p.n_tiles - i_first;     // query tiles per query head
    const int n_it = per_head * p.group;          // iterations: (head in group, query tile)

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kBarRes), 2 * kPanels);  // one arrive (+ tx) per K_j / V_j panel
        for (int s = 0; s < L::kQSlots; ++s) {
            mbar_init(bar(L::kBarQFull + s), kPanels);  // one arrive (+ tx) per panel
            mbar_init(bar(L::kBarQEmpty + s), 1);
        }
        mbar_init(bar(L::kBarDoFull), kPanels);
        mbar_init(bar(L::kBarDoEmpty), 2);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(L::kBarVecFull + s), 32);
            mbar_init(bar(L::kBarVecFree + s), kBwdEwThreads);
        }
        mbar_init(bar(L::kBarS), 1);
        mbar_init(bar(L::kBarSFree), kBwdEwThreads);
        mbar_init(bar(L::kBarDP), 1);
        mbar_init(bar(L::kBarP), kBwdEwThreads);
        mbar_init(bar(L::kBarPFree), 1);
        mbar_init(bar(L::kBarDS), kBwdEwThreads);
        mbar_init(bar(L::kBarDone), 2);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kBwdMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    static_assert(L::kBarDoFull < 32, "load barriers must fit the ArmedPhases mask");
    const uint32_t t_s = tmem, t_dp = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 384;
    auto it_head = [=](int it) { return hkv * p.group + it / per_head; };
    auto it_tile = [=](int it) { return i_first + it % per_head; };

    if (warp == kBwdLoadWarp) {
        // ---------------- producer: lanes 0..kPanels-1 issue the Q panels and lanes kPanels..
        // 2*kPanels-1 the dO panels (one thread's bulk copies run one after another), every lane
        // stages 4+4 vector entries, fetched into registers one iteration ahead ------------------
        ArmedPhases armed;  // this lane's loads (by barrier index), drained after an abort
        if (lane < 2 * kPanels) {  // K_j / V_j panel lane % kPanels
            const int h = lane % kPanels;
            mbar_arrive_expect_tx(bar(L::kBarRes), L::kPanelBytes);
            armed.arm(L::kBarRes, 0u);
            if (lane < kPanels)
                tma_load_4d(sbase + L::kRes0 + h * L::kPanelBytes, &tmap_k, bar(L::kBarRes),
                            h * 64, j * 128, hkv, b);
            else
                tma_load_4d(sbase + L::kRes1 + h * L::kPanelBytes, &tmap_v, bar(L::kBarRes),
                            h * 64, j * 128, hkv, b);
        }
        // -lse2 = -LSE*log2(e) and -Delta of queries lane*4 .. lane*4+3 of the iteration's tile
        // (0 past N: see top), fetched into registers one step ahead; stored negated so the
        // elementwise warps add them with packed f32x2 instructions
        float nl[4], nd[4];
        auto fetch = [&](int it) {
            const size_t rowbase = (static_cast<size_t>(b) * p.Hq + it_head(it)) * p.N;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int q = it_tile(it) * 128 + lane * 4 + e;
                nl[e] = q < p.N ? -p.lse[rowbase + q] * kLog2e : 0.f;
                nd[e] = q < p.N ? -p.delta[rowbase + q] : 0.f;
            }
        };
        bool ok = true;
        auto load_q = [&](int it) {  // Q_it into ring slot it % 3, once dK(it-3) has read it
            const int s = it % L::kQSlots;
            ok = mbar_wait_warp<true>(bar(L::kBarQEmpty + s), ((it / L::kQSlots) & 1) ^ 1u,
                                      abort_flag, status_word);
            if (ok && lane < kPanels) {
                const int h = lane;
                mbar_arrive_expect_tx(bar(L::kBarQFull + s), L::kPanelBytes);
                armed.arm(L::kBarQFull + s, static_cast<uint32_t>(it / L::kQSlots));
                tma_load_4d(sbase + L::kQ + s * L::kTileBytes + h * L::kPanelBytes, &tmap_q,
                            bar(L::kBarQFull + s), h * 64, it_tile(it) * 128, it_head(it), b);
            }
        };
        auto load_vec = [&](int it) {  // vectors of step it, once step it-2 is done with the slot
            const int s = it & 1;
            ok = mbar_wait_warp<true>(bar(L::kBarVecFree + s), ((it >> 1) & 1) ^ 1u, abort_flag,
                                      status_word);
            if (!ok) return;
            float4* vec = reinterpret_cast<float4*>(smem + L::kVec) + s * 64;
            vec[lane] = make_float4(nl[0], nl[1], nl[2], nl[3]);
            vec[32 + lane] = make_float4(nd[0], nd[1], nd[2], nd[3]);
            mbar_arrive(bar(L::kBarVecFull + s));
            if (it + 1 < n_it) fetch(it + 1);
        };
        auto load_do = [&](int it) {  // dO_it, once dP^T(it-1) and dV(it-1) have read the buffer
            ok = mbar_wait_warp<true>(bar(L::kBarDoEmpty), (it & 1) ^ 1u, abort_flag, status_word);
            if (ok && lane >= kPanels && lane < 2 * kPanels) {
                const int h = lane - kPanels;
                mbar_arrive_expect_tx(bar(L::kBarDoFull), L::kPanelBytes);
                armed.arm(L::kBarDoFull, static_cast<uint32_t>(it));
                tma_load_4d(sbase + L::kDO + h * L::kPanelBytes, &tmap_do, bar(L::kBarDoFull),
                            h * 64, it_tile(it) * 128, it_head(it), b);
            }
        };
        griddep_wait();  // Delta comes from the kernel launched right before this one
        if (n_it > 0) {
            fetch(0);
            load_q(0);
        }
        for (int it = 0; ok && it < n_it; ++it) {  // Q runs a step ahead of dO
            if (it + 1 < n_it) load_q(it + 1);
            if (ok) load_vec(it);
            if (ok) load_do(it);
        }
        if (*abort_flag) armed.drain(bar(0), globaltimer_ns() + kDrainLimitNs);
        __syncwarp();
    } else if (warp == kBwdMmaWarp || warp == kBwdMmaWarpB) {
        // ---------------- MMA issuers (warp-uniform, elected lane) -----------------------------
        // A: S^T(it+1) = K_j Q_(it+1)^T as soon as the elementwise warps have read S^T(it), then
        //    dV += P^T(it) dO_it with P^T from shared memory;
        // B: dP^T(it) = V_j dO_it^T, then dK += dS^T(it) Q_it with dS^T over dP^T in TMEM.
        // Each chain reuses its own TMEM region in issue order, so the chains need no common order.
        const bool chain_a = warp == kBwdMmaWarp;
        bool ok = mbar_wait_warp<true>(bar(L::kBarRes), 0, abort_flag, status_word);
        const uint32_t ka = sbase + L::kRes0, va = sbase + L::kRes1, pt = sbase + L::kPt;
        auto stage_q = [&](int it) { return sbase + L::kQ + (it % L::kQSlots) * L::kTileBytes; };
        const uint32_t da = sbase + L::kDO;
        auto wait_full = [&](int it) {  // Q_it landed
            const bool w = mbar_wait_warp<true>(bar(L::kBarQFull + it % L::kQSlots),
                                                (it / L::kQSlots) & 1, abort_flag, status_word);
            tc_fence_after();
            return w;
        };
        auto wait_do = [&](int it) {  // dO_it landed
            const bool w = mbar_wait_warp<true>(bar(L::kBarDoFull), it & 1, abort_flag,
                                                status_word);
            tc_fence_after();
            return w;
        };
        auto s_mma = [&](int it) {  // S^T = K_j Q_it^T
            const uint32_t qa = stage_q(it);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
                mma_bf16_ss_warp(t_s, smem_desc_sw128(ka + off, 16, 1024),
                                 smem_desc_sw128(qa + off, 16, 1024), kIdescS, kk > 0);
            }
            mma_commit_warp(bar(L::kBarS));
        };
        if (chain_a) {
            if (ok && n_it > 0) ok = wait_full(0);
            if (ok && n_it > 0) s_mma(0);
            for (int it = 0; ok && it < n_it; ++it) {
                if (it + 1 < n_it) {
                    ok = wait_full(it + 1);
                    if (ok) ok = mbar_wait_warp(bar(L::kBarSFree), it & 1, abort_flag,
                                                status_word);
                    if (!ok) break;
                    tc_fence_after();
                    s_mma(it + 1);
                }
                ok = mbar_wait_warp(bar(L::kBarP), it & 1, abort_flag, status_word);
                if (ok) ok = wait_do(it);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO_i  (K = 128 queries)
                    mma_bf16_ss_warp(t_dv,
                                     smem_desc_sw128(pt + (kk >> 2) * L::kPanelBytes + (kk & 3) * 32,
                                                     16, 1024),
                                     smem_desc_sw128(da + kk * 2048, L::kPanelBytes, 1024),
                                     kIdescAcc, (it > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(bar(L::kBarPFree));
                mma_commit_warp(bar(L::kBarDoEmpty));
            }
        } else {
            for (int it = 0; ok && it < n_it; ++it) {
                ok = wait_do(it);
                if (!ok) break;
                const uint32_t qa = stage_q(it);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {  // dP^T = V_j dO_i^T
                    const uint32_t off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
                    mma_bf16_ss_warp(t_dp, smem_desc_sw128(va + off, 16, 1024),
                                     smem_desc_sw128(da + off, 16, 1024), kIdescS, kk > 0);
                }
                mma_commit_warp(bar(L::kBarDP));
                mma_commit_warp(bar(L::kBarDoEmpty));
                ok = mbar_wait_warp<true>(bar(L::kBarDS), it & 1, abort_flag, status_word);
                if (ok) ok = wait_full(it);  // Q_it (landed before S^T(it); for visibility)
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dK += dS^T Q_i
                    mma_bf16_ts_warp(t_dk, t_dp + packed_col(kk),
                                     smem_desc_sw128(qa + kk * 2048, L::kPanelBytes, 1024),
                                     kIdescAcc, (it > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(bar(L::kBarQEmpty + it % L::kQSlots));
            }
        }
        if (ok) mma_commit_warp(bar(L::kBarDone));
        __syncwarp();
    } else {
        // ---------------- elementwise warps 0-7: key row `row` of tile j, queries c0 .. c0+63 --
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;  // key within the tile (TMEM lane)
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int c0 = half * 64;
        const float c = p.scale_log2;
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int s = it & 1;
            const float* vec = reinterpret_cast<const float*>(smem + L::kVec) + s * 256 + c0;
            // the step's lse2/Delta vectors, stored by the producer lanes before their arrive
            ok = mbar_wait_warp(bar(L::kBarVecFull + s), (it >> 1) & 1, abort_flag, status_word);
            if (ok) ok = mbar_wait_warp(bar(L::kBarS), it & 1, abort_flag, status_word);
            if (!ok) break;
            tc_fence_after();
            // P^T row: p[q] = exp2(c*s - lse2_q)
            float pr[64];
            {
                uint32_t r[64];
                tmem_ld32(lane_base + t_s + c0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(lane_base + t_s + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(L::kBarSFree));  // S^T(it+1) may now be formed over it
#pragma unroll
                for (int q = 0; q < 64; q += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(vec + q);  // -lse2
                    float x0, x1, x2, x3;
                    ffma2(x0, x1, __uint_as_float(r[q]), __uint_as_float(r[q + 1]), c, c, l4.x, l4.y);
                    ffma2(x2, x3, __uint_as_float(r[q + 2]), __uint_as_float(r[q + 3]), c, c, l4.z,
                          l4.w);
                    pr[q] = ex2_approx(x0);
                    pr[q + 1] = ex2_approx(x1);
                    pr[q + 2] = ex2_approx(x2);
                    pr[q + 3] = ex2_approx(x3);
                }
            }
            if (p.causal && it_tile(it) == j) {  // diagonal tile: query q sees key `row` iff q >= row
#pragma unroll
                for (int q = 0; q < 64; ++q) pr[q] = c0 + q < row ? 0.f : pr[q];
            }
            // P^T row -> bf16 -> panel `half` of the P^T tile (128B swizzle, K-major operand),
            // once dV(it-1) has finished reading the previous P^T
            if (it > 0) {
                ok = mbar_wait_warp(bar(L::kBarPFree), (it - 1) & 1, abort_flag, status_word);
                if (!ok) break;
            }
            {
                const uint32_t prow = sbase + L::kPt + half * L::kPanelBytes + row * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_shared_v4(prow + ((ch ^ (row & 7)) << 4),
                                 pack_bf16x2(pr[8 * ch], pr[8 * ch + 1]),
                                 pack_bf16x2(pr[8 * ch + 2], pr[8 * ch + 3]),
                                 pack_bf16x2(pr[8 * ch + 4], pr[8 * ch + 5]),
                                 pack_bf16x2(pr[8 * ch + 6], pr[8 * ch + 7]));
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(L::kBarP));
            // dS^T row: ds[q] = p[q] (dp[q] - Delta_q); this warp's 64 dP^T columns are read in one
            // go, and the 32 packed results go over the first 32 of them.
            ok = mbar_wait_warp(bar(L::kBarDP), it & 1, abort_flag, status_word);
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t r[64];
                tmem_ld32(lane_base + t_dp + c0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(lane_base + t_dp + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_wait_ld();
                uint32_t pk[32];
#pragma unroll
                for (int q = 0; q < 64; q += 4) {
                    const float4 d4 = *reinterpret_cast<const float4*>(vec + 128 + q);  // -Delta
                    float t0, t1, t2, t3, d0, d1, d2, d3;
                    fadd2(t0, t1, __uint_as_float(r[q]), __uint_as_float(r[q + 1]), d4.x, d4.y);
                    fadd2(t2, t3, __uint_as_float(r[q + 2]), __uint_as_float(r[q + 3]), d4.z, d4.w);
                    ffma2(d0, d1, pr[q], pr[q + 1], t0, t1, 0.f, 0.f);
                    ffma2(d2, d3, pr[q + 2], pr[q + 3], t2, t3, 0.f, 0.f);
                    pk[q / 2] = pack_bf16x2(d0, d1);
                    pk[q / 2 + 1] = pack_bf16x2(d2, d3);
                }
                tmem_st32(lane_base + t_dp + c0, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(L::kBarDS));
            mbar_arrive(bar(L::kBarVecFree + s));  // this step's vectors are no longer read
        }
        // epilogue: dK = sm_scale * acc (warps 0-3), dV = acc (warps 4-7) -> bf16 -> smem (over
        // K_j, V_j) -> TMA store
        if (ok) ok = mbar_wait_warp(bar(L::kBarDone), 0, abort_flag, status_word);
        if (ok) {
            tc_fence_after();
            if (half == 0)
                stage_rows_bf16<D>(sbase + L::kRes0, lane_base + t_dk, row, p.sm_scale, 0, D / 32);
            else
                stage_rows_bf16<D>(sbase + L::kRes1, lane_base + t_dv, row, 1.0f, 0, D / 32);
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, kBwdEwThreads);
        if (ok && warp == 0 && lane == 0 &&
            ATTN_DCHECK(b < p.B && hkv < p.Hkv && j < p.n_tiles)) {
            for (int h = 0; h < kPanels; ++h) {
                tma_store_4d(&tmap_dk, sbase + L::kRes0 + h * L::kPanelBytes, h * 64, j * 128, hkv, b);
                tma_store_4d(&tmap_dv, sbase + L::kRes1 + h * L::kPanelBytes, h * 64, j * 128, hkv, b);
            }
            tma_store_commit_and_wait();
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// dQ layout: Q_i and dO_i resident, then separate rings for K (3 slots: K_j is read by S(j),
// formed a step ahead, and by dQ(j), issued last) and V (2 slots: read only by dP(j)), so the
// load of K_(j+2) never waits for dQ(j) to finish.
template <int D>
struct DqSmem {
    static constexpr int kPanelBytes = 128 * 64 * 2;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kKSlots = 3, kVSlots = 2;
    static constexpr int kRes0 = 0;                        // Q_i
    static constexpr int kRes1 = kTileBytes;               // dO_i
    static constexpr int kK = 2 * kTileBytes;              // K ring
    static constexpr int kV = kK + kKSlots * kTileBytes;   // V ring
    static constexpr int kBars = kV + kVSlots * kTileBytes;
    static constexpr int kBarQ = 0;                          // Q_i landed (one arrive per panel)
    static constexpr int kBarDo = 1;                         // dO_i landed
    static constexpr int kBarQFree = 2;                      // the item's last S MMA read Q_i
    static constexpr int kBarDoFree = 3;                     // the item's last dP MMA read dO_i
    static constexpr int kBarKFull = 4;                      // [kKSlots]
    static constexpr int kBarKEmpty = kBarKFull + kKSlots;   // [kKSlots]
    static constexpr int kBarVFull = kBarKEmpty + kKSlots;   // [kVSlots]
    static constexpr int kBarVEmpty = kBarVFull + kVSlots;   // [kVSlots]
    static constexpr int kBarS = kBarVEmpty + kVSlots;       // [2]
    static constexpr int kBarDP = kBarS + 2;
    static constexpr int kBarDS = kBarDP + 1;
    static constexpr int kBarDone = kBarDS + 1;              // the item's dQ is complete
    static constexpr int kBarDqFree = kBarDone + 1;          // the epilogue has read dQ
    static constexpr int kBarItemFull = kBarDqFree + 1;      // [2]
    static constexpr int kBarItemEmpty = kBarItemFull + 2;   // [2]
    static constexpr int kNumBars = kBarItemEmpty + 2;
    static constexpr int kItems = kBars + kNumBars * 8;      // int[2]: the item ring
    static constexpr int kTmemSlot = kItems + 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 232448, "dQ shared memory exceeds the per-block limit");
    // readers of an item ring slot besides the claiming lane: the other producer lanes, the two
    // MMA warps and the eight elementwise warps (one arrival per warp)
    static constexpr int kItemReaders = 2 * (D / 64) - 1 + 2 + 8;
};

// Persistent: min(items, SMs) CTAs; a work item is one (128-row query tile i, b, query head),
// latest (heaviest under the causal mask) tiles first.  CTA c takes item c, then claims items
// from the launch's counter (the forward's scheme, one of the same counters, or its static
// schedule in a captured graph).  Across items every
// mbarrier keeps counting phases: Q_i and dO_i reload as soon as the previous item's last S and
// dP MMAs have read them, so the next item's loads and first MMAs overlap the current item's last
// steps and its epilogue, and the first dQ MMA of an item waits until the epilogue has read the
// previous item's dQ out of TMEM.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ CUtensorMap tmap_do, const BwdParams p,
                       unsigned int* status_word) {
    using L = DqSmem<D>;
    constexpr int kPanels = D / 64;
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0);
    constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, 1);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    auto bar = [=](int x) -> uint32_t { return sbase + L::kBars + 8u * x; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    volatile int* item_ring = reinterpret_cast<volatile int*>(smem + L::kItems);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh_count = p.B * p.Hq;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kBarQ), kPanels);
        mbar_init(bar(L::kBarDo), kPanels);
        mbar_init(bar(L::kBarQFree), 1);
        mbar_init(bar(L::kBarDoFree), 1);
        for (int s = 0; s < L::kKSlots; ++s) {
            mbar_init(bar(L::kBarKFull + s), kPanels);
            mbar_init(bar(L::kBarKEmpty + s), 1);
        }
        for (int s = 0; s < L::kVSlots; ++s) {
            mbar_init(bar(L::kBarVFull + s), kPanels);
            mbar_init(bar(L::kBarVEmpty + s), 1);
        }
        mbar_init(bar(L::kBarS), 1);
        mbar_init(bar(L::kBarS + 1), 1);
        mbar_init(bar(L::kBarDP), 1);
        mbar_init(bar(L::kBarDS), kBwdEwThreads);
        mbar_init(bar(L::kBarDone), 1);
        mbar_init(bar(L::kBarDqFree), kBwdEwThreads);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(L::kBarItemFull + s), 1);
            mbar_init(bar(L::kBarItemEmpty + s), L::kItemReaders);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kBwdMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    static_assert(L::kBarVFull + L::kVSlots <= 32, "load barriers must fit the ArmedPhases mask");
    // S is double-buffered (S(g+1) is formed while the elementwise warps work on S(g), g counting
    // the CTA's steps over all its items); dS is written over the S buffer it came from.
    const uint32_t t_s0 = tmem, t_dp = tmem + 128, t_dq = tmem + 256, t_s1 = tmem + 384;
    // item -> query tile and (b, hq)
    auto tile_of = [&](int item) { return p.n_tiles - 1 - item / bh_count; };
    auto steps_of = [&](int i) { return p.causal ? i + 1 : p.n_tiles; };  // key tiles 0 .. n-1

    // Item ring reader (all roles but the claiming lane); warps arrive once.
    auto read_item = [&](int k, bool whole_warp) -> int {
        const int slot = k & 1;
        const uint32_t ph = static_cast<uint32_t>(k >> 1) & 1u;
        bool ok;
        if (whole_warp)
            ok = mbar_wait_warp<true>(bar(L::kBarItemFull + slot), ph, abort_flag, status_word);
        else
            ok = mbar_wait_bounded<true>(bar(L::kBarItemFull + slot), ph, abort_flag, status_word);
        if (!ok) return -1;
        const int item = item_ring[slot];
        if (whole_warp) {
            __syncwarp();
            mbar_arrive_warp(bar(L::kBarItemEmpty + slot));
        } else {
            mbar_arrive(bar(L::kBarItemEmpty + slot));
        }
        return item;
    };

    if (warp == kBwdLoadWarp) {
        // one lane per panel stream (one thread's bulk copies run one after another): lanes
        // 0..kPanels-1 load a Q_i panel, then that panel of every K_j; lanes kPanels..2*kPanels-1
        // a dO_i panel, then that panel of every V_j.  Lane 0 also claims the items.
        if (lane < 2 * kPanels) {
            ArmedPhases armed;  // this lane's loads (by barrier index), drained after an abort
            const bool kside = lane < kPanels;
            const int h = lane % kPanels;
            const int slots = kside ? L::kKSlots : L::kVSlots;
            const int full0 = kside ? L::kBarKFull : L::kBarVFull;
            const int empty0 = kside ? L::kBarKEmpty : L::kBarVEmpty;
            const uint32_t ring_base = sbase + (kside ? L::kK : L::kV);
            const CUtensorMap* map = kside ? &tmap_k : &tmap_v;
            bool claims_done = false;
            int claim_round = 0;
            auto claim = [&]() -> int {
                return claim_next_item(p.sched, p.items, claim_round, claims_done, blockIdx.x,
                                       gridDim.x);
            };
            int g = 0;  // K/V stream position (steps of the earlier items)
            for (int k = 0;; ++k) {
                int item;
                if (lane == 0) {
                    const int slot = k & 1;
                    if (!mbar_wait_bounded<true>(bar(L::kBarItemEmpty + slot),
                                                 (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u,
                                                 abort_flag, status_word))
                        break;
                    item = k == 0 ? static_cast<int>(blockIdx.x) : claim();
                    item_ring[slot] = item;
                    mbar_arrive(bar(L::kBarItemFull + slot));
                } else {
                    item = read_item(k, false);
                }
                if (item < 0) break;
                const int i = tile_of(item), bh = item % bh_count;
                const int b = bh / p.Hq, hq = bh % p.Hq, hkv = hq / p.group;
                const int n_it = steps_of(i);
                // the resident tile, once the previous item's last MMA has read its buffer
                if (k > 0 && !mbar_wait_bounded<true>(bar(kside ? L::kBarQFree : L::kBarDoFree),
                                                      (k - 1) & 1, abort_flag, status_word))
                    break;
                mbar_arrive_expect_tx(bar(kside ? L::kBarQ : L::kBarDo), L::kPanelBytes);
                armed.arm(kside ? L::kBarQ : L::kBarDo, static_cast<uint32_t>(k));
                tma_load_4d(sbase + (kside ? L::kRes0 : L::kRes1) + h * L::kPanelBytes,
                            kside ? &tmap_q : &tmap_do, bar(kside ? L::kBarQ : L::kBarDo), h * 64,
                            i * 128, hq, b);
                bool ok = true;
                for (int it = 0; it < n_it; ++it, ++g) {
                    const int s = g % slots;
                    ok = mbar_wait_bounded<true>(bar(empty0 + s), ((g / slots) & 1) ^ 1u,
                                                 abort_flag, status_word);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(full0 + s), L::kPanelBytes);
                    armed.arm(full0 + s, static_cast<uint32_t>(g / slots));
                    tma_load_4d(ring_base + s * L::kTileBytes + h * L::kPanelBytes, map,
                                bar(full0 + s), h * 64, it * 128, hkv, b);
                }
                if (!ok) break;
            }
            // after an abort, still make this CTA's claims up to the one past the end
            if (lane == 0)
                while (!claims_done) (void)claim();
            if (*abort_flag) armed.drain(bar(0), globaltimer_ns() + kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == kBwdMmaWarp || warp == kBwdMmaWarpB) {
        // A: S(g+1) = Q_i K_(g+1)^T ahead, then dQ += dS(g) K_g once dS(g) is ready;
        // B: dP(g) = dO_i V_g^T, each after the elementwise warps have read the previous one.
        const bool chain_a = warp == kBwdMmaWarp;
        const uint32_t qa = sbase + L::kRes0, da = sbase + L::kRes1;
        auto stage_k = [&](int g) { return sbase + L::kK + (g % L::kKSlots) * L::kTileBytes; };
        auto stage_v = [&](int g) { return sbase + L::kV + (g % L::kVSlots) * L::kTileBytes; };
        auto wait_k = [&](int g) {
            const bool w = mbar_wait_warp<true>(bar(L::kBarKFull + g % L::kKSlots),
                                                (g / L::kKSlots) & 1, abort_flag, status_word);
            tc_fence_after();
            return w;
        };
        auto wait_v = [&](int g) {
            const bool w = mbar_wait_warp<true>(bar(L::kBarVFull + g % L::kVSlots),
                                                (g / L::kVSlots) & 1, abort_flag, status_word);
            tc_fence_after();
            return w;
        };
        auto s_mma = [&](int g) {  // S(g) into buffer g&1
            const uint32_t ka = stage_k(g);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
                mma_bf16_ss_warp((g & 1) ? t_s1 : t_s0, smem_desc_sw128(qa + off, 16, 1024),
                                 smem_desc_sw128(ka + off, 16, 1024), kIdescS, kk > 0);
            }
            mma_commit_warp(bar(L::kBarS + (g & 1)));
        };
        bool ok = true;
        int g0 = 0;  // steps of the earlier items
        for (int k = 0; ok; ++k) {
            const int item = read_item(k, true);
            if (item < 0) break;
            const int n_it = steps_of(tile_of(item));
            if (chain_a) {
                ok = mbar_wait_warp<true>(bar(L::kBarQ), k & 1, abort_flag, status_word);
                if (ok) ok = wait_k(g0);
                if (ok) {
                    s_mma(g0);
                    if (n_it == 1) mma_commit_warp(bar(L::kBarQFree));
                }
                for (int it = 0; ok && it < n_it; ++it) {
                    const int g = g0 + it;
                    if (it + 1 < n_it) {
                        ok = wait_k(g + 1);
                        if (!ok) break;
                        s_mma(g + 1);
                        if (it + 2 == n_it) mma_commit_warp(bar(L::kBarQFree));
                    }
                    ok = mbar_wait_warp(bar(L::kBarDS), g & 1, abort_flag, status_word);
                    // the first dQ MMA overwrites the accumulator: the previous item's epilogue
                    // must have read it
                    if (ok && it == 0 && k > 0)
                        ok = mbar_wait_warp(bar(L::kBarDqFree), (k - 1) & 1, abort_flag,
                                            status_word);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ka = stage_k(g), ts = (g & 1) ? t_s1 : t_s0;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // dQ += dS K_j  (K = 128 keys)
                        mma_bf16_ts_warp(t_dq, ts + packed_col(kk),
                                         smem_desc_sw128(ka + kk * 2048, L::kPanelBytes, 1024),
                                         kIdescAcc, (it > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_warp(bar(L::kBarKEmpty + g % L::kKSlots));
                }
                if (ok) mma_commit_warp(bar(L::kBarDone));
            } else {
                ok = mbar_wait_warp<true>(bar(L::kBarDo), k & 1, abort_flag, status_word);
                for (int it = 0; ok && it < n_it; ++it) {
                    const int g = g0 + it;
                    ok = wait_v(g);
                    if (!ok) break;
                    if (g > 0) {  // dP(g) overwrites dP(g-1): the elementwise warps must have read it
                        ok = mbar_wait_warp<true>(bar(L::kBarDS), (g - 1) & 1, abort_flag,
                                                  status_word);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    const uint32_t va = stage_v(g);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // dP = dO_i V_j^T
                        const uint32_t off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
                        mma_bf16_ss_warp(t_dp, smem_desc_sw128(da + off, 16, 1024),
                                         smem_desc_sw128(va + off, 16, 1024), kIdescS, kk > 0);
                    }
                    mma_commit_warp(bar(L::kBarDP));
                    mma_commit_warp(bar(L::kBarVEmpty + g % L::kVSlots));
                    if (it + 1 == n_it) mma_commit_warp(bar(L::kBarDoFree));
                }
            }
            g0 += n_it;
        }
        __syncwarp();
    } else {
        // elementwise warps 0-7: query row `row` of tile i, keys c0 .. c0+63 of the key tile
        griddep_wait();  // Delta is complete once the kernel launched right before this one is
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int c0 = half * 64;
        const float c = p.scale_log2;
        bool ok = true;
        int g = 0;  // steps of this CTA so far
        for (int k = 0; ok; ++k) {
            const int item = read_item(k, true);
            if (item < 0) break;
            const int i = tile_of(item), bh = item % bh_count;
            const int n_it = steps_of(i);
            const int row_g = i * 128 + row;
            const size_t rix = static_cast<size_t>(bh) * p.N + row_g;
            const float lse2 = row_g < p.N ? p.lse[rix] * kLog2e : 0.f;
            const float dlt = row_g < p.N ? p.delta[rix] : 0.f;
            for (int it = 0; it < n_it; ++it, ++g) {
                const uint32_t ts = (g & 1) ? t_s1 : t_s0;
                ok = mbar_wait_warp(bar(L::kBarS + (g & 1)), (g >> 1) & 1, abort_flag,
                                    status_word);
                if (!ok) break;
                tc_fence_after();
                float pr[64];
                {
                    uint32_t r[64];
                    tmem_ld32(lane_base + ts + c0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                    tmem_ld32(lane_base + ts + c0 + 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 64; x += 2) {
                        float x0, x1;
                        ffma2(x0, x1, __uint_as_float(r[x]), __uint_as_float(r[x + 1]), c, c,
                              -lse2, -lse2);
                        pr[x] = ex2_approx(x0);
                        pr[x + 1] = ex2_approx(x1);
                    }
                }
                if (p.causal && it == i) {  // diagonal tile: key x visible to query `row` iff x <= row
#pragma unroll
                    for (int x = 0; x < 64; ++x) pr[x] = c0 + x > row ? 0.f : pr[x];
                }
                ok = mbar_wait_warp(bar(L::kBarDP), g & 1, abort_flag, status_word);
                if (!ok) break;
                tc_fence_after();
                // dS in 32-column chunks; the packed dS goes over this warp's S columns (all read)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + t_dp + c0 + cc * 32, r);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int kx = cc * 32 + 2 * x;
                        float t0, t1, d0, d1;
                        fadd2(t0, t1, __uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1]),
                              -dlt, -dlt);
                        ffma2(d0, d1, pr[kx], pr[kx + 1], t0, t1, 0.f, 0.f);
                        pk[x] = pack_bf16x2(d0, d1);
                    }
                    tmem_st16(lane_base + ts + c0 + cc * 16, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(L::kBarDS));
            }
            if (!ok) break;
            // ---- epilogue: dQ = sm_scale * acc -> bf16, this warp's columns of its row,
            // straight from registers to global memory (16-byte stores)
            ok = mbar_wait_warp(bar(L::kBarDone), k & 1, abort_flag, status_word);
            if (!ok) break;
            tc_fence_after();
            constexpr int kCols = D / 2;  // columns per warp: half of the row
            __nv_bfloat16* dst = p.dq + rix * p.d_out + half * kCols;
#pragma unroll
            for (int cc = 0; cc < kCols / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(lane_base + t_dq + half * kCols + cc * 32, r);
                tmem_wait_ld();
                if (row_g < p.N && ATTN_DCHECK(rix < static_cast<size_t>(p.B) * p.Hq * p.N)) {
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        if (half * kCols + cc * 32 + c8 * 8 >= p.d_out) break;
                        uint32_t w[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            w[x] = pack_bf16x2(__uint_as_float(r[c8 * 8 + 2 * x]) * p.sm_scale,
                                               __uint_as_float(r[c8 * 8 + 2 * x + 1]) * p.sm_scale);
                        st_global_v4u(dst + cc * 32 + c8 * 8, w[0], w[1], w[2], w[3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(L::kBarDqFree));  // the next item's first dQ MMA may overwrite it
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace gb300attn
