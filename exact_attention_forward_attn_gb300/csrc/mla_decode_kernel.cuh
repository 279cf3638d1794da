// mla_decode_kernel.cuh - absorbed multi-head latent attention (MLA) decode for sm_103a.
//
// "Attention Kernel 实现与正确性验证" (walkerchi.com), section 2.1 (the absorption trick) and 2.2
// (the absorbed reference): with W_uk folded into the query, every head scores the compressed
// cache directly, and the output stays in the compressed space until the caller's W_uv.  Per
// batch b, head h and cached token t (one decode query per head; the cache is shared by all
// heads, like multi-query attention with d_qk = d_c + d_r and d_v = d_c):
//   s_t   = sm_scale * (q_abs[b,h] . c_kv[b,t] + q_pe[b,h] . k_pe[b,t])
//   out_c = sum_t softmax_t(s) c_kv[b,t]        LSE = log sum_t exp(s_t)
// Section 2.4 runs it split over the token axis (split-T) with a safe-softmax merge; so does this.
//
// Widths are fixed at the page's DeepSeek-V3 values: d_c = 512, d_r = 64 (d_qk = 576 = 9 panels
// of 64 columns).  q is [B, H, 576] (q_abs then q_pe), kv is [B, T, 576] (c_kv then k_pe), both
// bf16 and contiguous.
//
// One CTA per (batch, 128-head tile, value half r, token split).  The 128 heads are the MMA's M.
// A 512-wide fp32 output would fill the whole TMEM, so each CTA of a pair owns 256 output columns
// (c_kv panels 4r .. 4r+3, its "value panels") and both form the full scores; the cache tile is
// read by both from L2.  Per 64-token tile the scores take 36 M=128, N=64 MMAs (one issuing
// warp keeps up with the tensor pipe at that size); O += P V is one N=256 MMA per 16 tokens,
// issued by a second warp.
//   TMEM (512 columns): S (64; S(i+1) is issued as soon as the softmax has loaded S(i)) |
//   P (32, bf16) | the five X-side Q panels (5 x 32, bf16, the A operand of their score MMAs) |
//   O (256).
//   Shared memory: the four value-side Q panels (64 KiB); Y = the 4 value panels, double-
//   buffered (2 x 32 KiB, also the B operand of P.V); X = a ring of 12 slots of 8 KiB through
//   which the 5 other cache panels of every tile stream (a slot is refilled as soon as its MMAs
//   have read it, so loads run 2.4 tiles ahead).  The TMEM-bound Q panels are staged through the
//   second Y buffer and the X ring at start.
// Warps: 0-3 softmax (one head row per thread), 4 issues S, 5 issues P.V, 6 loads.
// Token splits: with 2..kMlaMaxClusterSplits splits the split CTAs of one (batch, head tile,
// value half) are a thread-block cluster and combine their partial outputs through distributed
// shared memory at the end (mla_cluster_merge); with more, the partials go to a global workspace
// and mla_merge_kernel combines them.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace gb300attn {

constexpr int kMlaDc = 512;
constexpr int kMlaDr = 64;
constexpr int kMlaDqk = kMlaDc + kMlaDr;
constexpr int kMlaPanels = kMlaDqk / 64;  // 9
constexpr int kMlaBN = 64;                // tokens per tile
constexpr int kMlaHeads = 128;            // heads per CTA (M)
constexpr int kMlaThreads = 224;
constexpr int kMlaMmaA = 4, kMlaMmaB = 5, kMlaLoad = 6;
constexpr float kMlaRescaleThreshold = 8.0f;  // log2 units
constexpr int kMlaMaxClusterSplits = 4;    // up to this many splits merge inside a cluster

struct MlaParams {
    int B, H, T;
    int n_ht;          // ceil(H / 128)
    int n_tiles;       // ceil(T / 64)
    int n_splits;      // token splits
    float scale_log2;  // sm_scale * log2(e)
    __nv_bfloat16* out;  // [B, H, 512]            (n_splits == 1)
    float* lse;          // [B, H]                  (n_splits == 1)
    // 2..kMlaMaxClusterSplits splits: the n_splits CTAs of a (b, ht, r) group form a cluster and
    // merge through distributed shared memory (no workspace); more: the workspace below and
    // mla_merge_kernel.
    int cluster_merge;
    float* ws_o;         // [n_splits, B, H, 512]   (n_splits > kMlaMaxClusterSplits): O_s = acc / l
    float* ws_lse;       // [n_splits, B, H]        (idem): natural-log LSE_s
    int stall_tile;  // test hook: >= 0 withholds the X panels of this token tile (else -1)
};

struct MlaSmem {
    static constexpr int kQPanel = kMlaHeads * 128;  // 16 KiB
    static constexpr int kKvPanel = kMlaBN * 128;    // 8 KiB
    static constexpr int kQ = 0;                     // 4 Q panels: the value panels 4r+y
    static constexpr int kXSlots = 12;
    static constexpr int kYBufs = 2;
    static constexpr int kY = kQ + 4 * kQPanel;                 // kYBufs buffers of 4 panels
    static constexpr int kX = kY + kYBufs * 4 * kKvPanel;       // X ring
    // start-up staging of the 5 TMEM Q panels: the last Y buffer (first used by tile 1) and the
    // X ring, which lie next to each other
    static constexpr int kStage = kY + (kYBufs - 1) * 4 * kKvPanel;
    static constexpr int kBars = kX + kXSlots * kKvPanel;
    // barriers
    static constexpr int kBarQ = 0;         // Q panels landed (tx)
    static constexpr int kBarQt = 1;        // TMEM Q panels written, staging free (count 128)
    static constexpr int kBarXFull = 2;     // [kXSlots]
    static constexpr int kBarXEmpty = kBarXFull + kXSlots;
    static constexpr int kBarYFull = kBarXEmpty + kXSlots;  // [kYBufs]
    static constexpr int kBarYEmpty = kBarYFull + kYBufs;   // [kYBufs]
    static constexpr int kBarSFull = kBarYEmpty + kYBufs;
    static constexpr int kBarSFree = kBarSFull + 1;    // the softmax has read S (count 128)
    static constexpr int kBarPFull = kBarSFree + 1;    // P in TMEM (count 128)
    static constexpr int kBarPvDone = kBarPFull + 1;   // P.V complete
    static constexpr int kNumBars = kBarPvDone + 1;
    static constexpr int kTmemSlot = kBars + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kStage + 5 * kQPanel <= kBars, "staging must fit in the last Y buffer + X ring");
    // cluster merge: each row's LSE_s beside the staged O_s (the X ring is idle by then)
    static constexpr int kLseStage = kX;
    static_assert(kLseStage >= 4 * 32768 && kLseStage + kMlaHeads * 4 <= kBars,
                  "the staged LSE must not overlap the staged O");
    static_assert(kAlloc <= 232448, "MLA shared memory exceeds the per-block limit");
};

// TMEM columns
constexpr uint32_t kMlaTS = 0, kMlaTP = 64, kMlaTQ = 96, kMlaTO = 256;

// Panel (64 columns) of the cache feeding X slot x (x = 0..4) for value half r: the four c_kv
// panels outside the value half, then the k_pe panel.
__device__ __forceinline__ int mla_x_panel(int r, int x) {
    return x == 4 ? 8 : (r == 0 ? 4 + x : x);
}

// The merge of section 2.4's split-T inside a thread-block cluster: the n_splits CTAs of a
// (b, ht, r) group are one cluster, each has staged its O_s = acc / l (fp32; row rr of warp w at
// w * 32 KiB + rr KiB, 16-byte chunk ch at (ch ^ rr) * 16) and its LSE_s (kLseStage[row]) in its
// own shared memory, and CTA s combines rows s*R .. s*R + R - 1 of the 128-row tile (R = 128 /
// n_splits, rounded up) by reading every CTA's staging through distributed shared memory:
// LSE = M + ln sum_s exp(LSE_s - M) and out_c = sum_s exp(LSE_s - LSE) O_s.  A warp takes a row at
// a time, lane i columns 4i..4i+3 and 128+4i..+3.  If a CTA of the cluster gave up (its abort
// flag), nothing is merged; its expiry is in the status word.
__device__ __forceinline__ void mla_cluster_merge(const MlaParams& p, uint32_t sbase, int b,
                                                  int ht, int r, int rank, int warp, int lane) {
    using L = MlaSmem;
    const int ns = p.n_splits;
    uint32_t peer[kMlaMaxClusterSplits];
    bool aborted = false;
#pragma unroll
    for (int s = 0; s < kMlaMaxClusterSplits; ++s) {
        peer[s] = s < ns ? dsmem_addr(sbase, static_cast<uint32_t>(s)) : 0u;
        if (s < ns) aborted |= ld_dsmem_u32(peer[s] + L::kAbort) != 0u;
    }
    if (aborted) return;
    const int per = (kMlaHeads + ns - 1) / ns;
    const int row_end = min((rank + 1) * per, kMlaHeads);
    for (int row = rank * per + warp; row < row_end; row += 4) {
        const int h = ht * kMlaHeads + row;
        if (h >= p.H) break;  // warp-uniform; later rows are past H too
        float ls[kMlaMaxClusterSplits];
        float mx = -INFINITY;
#pragma unroll
        for (int s = 0; s < kMlaMaxClusterSplits; ++s) {
            ls[s] = s < ns ? __uint_as_float(ld_dsmem_u32(peer[s] + L::kLseStage + row * 4))
                           : -INFINITY;
            mx = fmaxf(mx, ls[s]);
        }
        float sum = 0.f;
#pragma unroll
        for (int s = 0; s < kMlaMaxClusterSplits; ++s) {
            ls[s] = s < ns ? __expf(ls[s] - mx) : 0.f;
            sum += ls[s];
        }
        const float inv = 1.0f / sum;
        const int rr = row & 31;
        const uint32_t off = static_cast<uint32_t>((row >> 5) * 32768 + rr * 1024);
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
        for (int s = 0; s < kMlaMaxClusterSplits; ++s) {
            if (s < ns) {
                const float w = ls[s] * inv;
                uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
                ld_dsmem_v4(peer[s] + off + ((lane ^ rr) << 4), x0, x1, x2, x3);
                ld_dsmem_v4(peer[s] + off + (((lane + 32) ^ rr) << 4), y0, y1, y2, y3);
                a0.x += w * __uint_as_float(x0); a0.y += w * __uint_as_float(x1);
                a0.z += w * __uint_as_float(x2); a0.w += w * __uint_as_float(x3);
                a1.x += w * __uint_as_float(y0); a1.y += w * __uint_as_float(y1);
                a1.z += w * __uint_as_float(y2); a1.w += w * __uint_as_float(y3);
            }
        }
        const size_t bh = static_cast<size_t>(b) * p.H + h;
        if (!ATTN_DCHECK(b < p.B && r < 2)) continue;
        __nv_bfloat16* dst = p.out + bh * kMlaDc + r * 256;
        *reinterpret_cast<uint2*>(dst + 4 * lane) =
            make_uint2(pack_bf16x2(a0.x, a0.y), pack_bf16x2(a0.z, a0.w));
        *reinterpret_cast<uint2*>(dst + 128 + 4 * lane) =
            make_uint2(pack_bf16x2(a1.x, a1.y), pack_bf16x2(a1.z, a1.w));
        if (r == 0 && lane == 0) p.lse[bh] = mx + __logf(sum);
    }
}

__global__ void __launch_bounds__(kMlaThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_kv, const MlaParams p,
                      unsigned int* status_word) {
    using L = MlaSmem;
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, kMlaBN, 0);  // Q (K-major) x cache (K-major)
    constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 1);    // P (TMEM) x Y (MN-major)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    auto bar = [=](int i) -> uint32_t { return sbase + L::kBars + 8u * i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_launch_dependents();  // the merge kernel (more than 4 splits) waits for us itself

    // work: blockIdx = ((b * n_ht + ht) * 2 + r) * n_splits + split
    int item = static_cast<int>(blockIdx.x);
    const int split = item % p.n_splits;
    item /= p.n_splits;
    const int r = item & 1;
    item >>= 1;
    const int ht = item % p.n_ht, b = item / p.n_ht;
    const int t_begin = static_cast<int>(static_cast<long long>(p.n_tiles) * split / p.n_splits);
    const int t_end = static_cast<int>(static_cast<long long>(p.n_tiles) * (split + 1) / p.n_splits);
    const int n_t = t_end - t_begin;  // >= 1 (n_splits <= n_tiles)
    auto ybuf = [](int i) { return i % MlaSmem::kYBufs; };
    auto yphase = [](int i) { return static_cast<uint32_t>((i / MlaSmem::kYBufs) & 1); };

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kBarQ), kMlaPanels);  // one arrive (+ tx) per Q panel
        mbar_init(bar(L::kBarQt), 128);
        for (int x = 0; x < L::kXSlots; ++x) {
            mbar_init(bar(L::kBarXFull + x), 1);
            mbar_init(bar(L::kBarXEmpty + x), 1);
        }
        for (int y = 0; y < L::kYBufs; ++y) {
            mbar_init(bar(L::kBarYFull + y), 4);  // one arrive (+ tx) per value panel
            mbar_init(bar(L::kBarYEmpty + y), 1);
        }
        mbar_init(bar(L::kBarSFull), 1);
        mbar_init(bar(L::kBarSFree), 128);
        mbar_init(bar(L::kBarPFull), 128);
        mbar_init(bar(L::kBarPvDone), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kMlaMmaA) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto t_s = [=](int) { return tmem + kMlaTS; };
    const uint32_t t_p = tmem + kMlaTP;
    const uint32_t t_q = tmem + kMlaTQ, t_o = tmem + kMlaTO;

    if (warp == kMlaLoad) {
        // ---------------- producer: one lane per panel.  One thread's bulk tensor copies are
        // processed one after another (~29 bytes per cycle per SM from one issuing thread), so
        // lanes 0-4 stream the five X panels of every tile and lanes 5-8 its four value panels;
        // lanes 0-8 first load one Q panel each ------------------------------------------------
        static_assert(L::kBarYFull + L::kYBufs <= 32, "load barriers must fit the ArmedPhases mask");
        if (lane < kMlaPanels) {
            ArmedPhases armed;  // this lane's loads (by barrier index), drained after an abort
            if (lane == 0) {
                tma_prefetch_desc(&tmap_q);
                tma_prefetch_desc(&tmap_kv);
            }
            __syncwarp(0x1ffu);
            // lanes 0-3: the value-side Q panels -> smem slots 0-3; lanes 4-8: the X-side Q
            // panels -> staging, for TMEM
            mbar_arrive_expect_tx(bar(L::kBarQ), L::kQPanel);
            armed.arm(L::kBarQ, 0u);
            if (lane < 4)
                tma_load_3d(sbase + L::kQ + lane * L::kQPanel, &tmap_q, bar(L::kBarQ),
                            (4 * r + lane) * 64, ht * kMlaHeads, b);
            else
                tma_load_3d(sbase + L::kStage + (lane - 4) * L::kQPanel, &tmap_q, bar(L::kBarQ),
                            mla_x_panel(r, lane - 4) * 64, ht * kMlaHeads, b);
            if (lane < 5) {  // X panel `lane` of every tile, once the start-up staging is done
                const int x = lane;
                bool ok = mbar_wait_bounded<true>(bar(L::kBarQt), 0, abort_flag, status_word);
                for (int i = 0; ok && i < n_t; ++i) {
                    const int k = 5 * i + x, slot = k % L::kXSlots;
                    ok = mbar_wait_bounded<true>(bar(L::kBarXEmpty + slot),
                                                 ((k / L::kXSlots) & 1) ^ 1u, abort_flag,
                                                 status_word);
                    if (!ok) break;
                    if (t_begin + i == p.stall_tile) continue;  // test hook: never deliver it
                    mbar_arrive_expect_tx(bar(L::kBarXFull + slot), L::kKvPanel);
                    armed.arm(L::kBarXFull + slot, static_cast<uint32_t>(k / L::kXSlots));
                    tma_load_3d(sbase + L::kX + slot * L::kKvPanel, &tmap_kv,
                                bar(L::kBarXFull + slot), mla_x_panel(r, x) * 64,
                                (t_begin + i) * kMlaBN, b);
                }
            } else {  // value panel lane-5 of every tile, into Y buffer i % kYBufs
                const int y = lane - 5;
                for (int i = 0; i < n_t; ++i) {
                    const int yb = ybuf(i);
                    // the last buffer holds start-up staging until the Q panels are in TMEM
                    if (i == L::kYBufs - 1 &&
                        !mbar_wait_bounded<true>(bar(L::kBarQt), 0, abort_flag, status_word))
                        break;
                    if (!mbar_wait_bounded<true>(bar(L::kBarYEmpty + yb), yphase(i) ^ 1u,
                                                 abort_flag, status_word))
                        break;
                    mbar_arrive_expect_tx(bar(L::kBarYFull + yb), L::kKvPanel);
                    armed.arm(L::kBarYFull + yb, yphase(i));
                    tma_load_3d(sbase + L::kY + (4 * yb + y) * L::kKvPanel, &tmap_kv,
                                bar(L::kBarYFull + yb), (4 * r + y) * 64, (t_begin + i) * kMlaBN,
                                b);
                }
            }
            if (*abort_flag) armed.drain(bar(0), globaltimer_ns() + kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == kMlaMmaA) {
        // ---------------- S(i) = Q . cache tile i into S[i&1], 36 MMAs (warp-uniform issue) ----
        // (the issuers' and the softmax warps' waits suspend instead of polling, leaving the
        // issue slots of their SM sub-partitions to the softmax warps: measured 2 % faster)
        bool ok = mbar_wait_warp<true>(bar(L::kBarQ), 0, abort_flag, status_word);
        if (ok) ok = mbar_wait_warp<true>(bar(L::kBarQt), 0, abort_flag, status_word);
        tc_fence_after();
        for (int i = 0; ok && i < n_t; ++i) {
            if (i >= 1) {  // the softmax has loaded S(i-1)
                ok = mbar_wait_warp<true>(bar(L::kBarSFree), (i - 1) & 1, abort_flag,
                                          status_word);
                if (!ok) break;
            }
            for (int x = 0; ok && x < 5; ++x) {  // the tile's five X panels have landed
                const int k = 5 * i + x;
                ok = mbar_wait_warp<true>(bar(L::kBarXFull + k % L::kXSlots),
                                          (k / L::kXSlots) & 1, abort_flag, status_word);
            }
            const int yb = ybuf(i);
            if (ok) ok = mbar_wait_warp<true>(bar(L::kBarYFull + yb), yphase(i), abort_flag,
                                              status_word);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int x = 0; x < 5; ++x) {
                const uint32_t kv = sbase + L::kX + ((5 * i + x) % L::kXSlots) * L::kKvPanel;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bdesc = smem_desc_sw128(kv + kk * 32, 16, 1024);
                    const uint32_t acc = (x == 0 && kk == 0) ? 0u : 1u;
                    mma_bf16_ts_warp(t_s(i), t_q + x * 32 + kk * 8, bdesc, kIdescS, acc);
                }
            }
            for (int x = 0; x < 5; ++x) mma_commit_warp(bar(L::kBarXEmpty + (5 * i + x) % L::kXSlots));
#pragma unroll
            for (int y = 0; y < 4; ++y) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss_warp(t_s(i),
                                     smem_desc_sw128(sbase + L::kQ + y * L::kQPanel + kk * 32, 16, 1024),
                                     smem_desc_sw128(sbase + L::kY + (4 * yb + y) * L::kKvPanel + kk * 32,
                                                     16, 1024),
                                     kIdescS, 1u);
            }
            mma_commit_warp(bar(L::kBarSFull));
        }
        __syncwarp();
    } else if (warp == kMlaMmaB) {
        // ---------------- O += P(i) Y_i (four N=256 MMAs), once the softmax has written P(i) ---
        bool ok = true;
        for (int i = 0; ok && i < n_t; ++i) {
            ok = mbar_wait_warp<true>(bar(L::kBarPFull), i & 1, abort_flag, status_word);
            if (!ok) break;
            tc_fence_after();
            const int yb = ybuf(i);
#pragma unroll
            for (int kk = 0; kk < kMlaBN / 16; ++kk)  // O += P Y  (K = 64 tokens, N = 256)
                mma_bf16_ts_warp(t_o, t_p + kk * 8,
                                 smem_desc_sw128(sbase + L::kY + 4 * yb * L::kKvPanel + kk * 2048,
                                                 L::kKvPanel, 1024),
                                 kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
            mma_commit_warp(bar(L::kBarPvDone));
            mma_commit_warp(bar(L::kBarYEmpty + yb));  // S(i) also read Y_i; it completed first
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps 0-3: head row `row` of the tile ------------------------
        const int row = warp * 32 + lane;
        const int h = ht * kMlaHeads + row;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float c = p.scale_log2;
        bool ok = mbar_wait_warp<true>(bar(L::kBarQ), 0, abort_flag, status_word);
        // start-up: the five staged Q panels -> TMEM (bf16 pairs, the MMA's A layout)
        if (ok) {
#pragma unroll 1
            for (int j = 0; j < 5; ++j) {
                const uint32_t src = sbase + L::kStage + j * L::kQPanel + row * 128;
                uint32_t v[32];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    ld_shared_v4(src + ((ch ^ (row & 7)) << 4), v[4 * ch], v[4 * ch + 1],
                                 v[4 * ch + 2], v[4 * ch + 3]);
                tmem_st32(lane_base + t_q + j * 32, v);
            }
            tmem_wait_st();
            tc_fence_before();
        }
        mbar_arrive(bar(L::kBarQt));
        float m = -INFINITY, l = 0.f;
        for (int i = 0; ok && i < n_t; ++i) {
            ok = mbar_wait_warp<true>(bar(L::kBarSFull), i & 1, abort_flag, status_word);
            if (!ok) break;
            tc_fence_after();
            float s[kMlaBN];
            {
                uint32_t ra[kMlaBN];
                tmem_ld32(lane_base + t_s(i), *reinterpret_cast<uint32_t(*)[32]>(&ra[0]));
                tmem_ld32(lane_base + t_s(i) + 32, *reinterpret_cast<uint32_t(*)[32]>(&ra[32]));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(L::kBarSFree));  // S(i+1) may now be formed over it
#pragma unroll
                for (int j = 0; j < kMlaBN; ++j) s[j] = __uint_as_float(ra[j]) * c;
            }
            const int valid = p.T - (t_begin + i) * kMlaBN;  // tokens of this tile inside T
            if (valid < kMlaBN) {
#pragma unroll
                for (int j = 0; j < kMlaBN; ++j)
                    if (j >= valid) s[j] = -INFINITY;
            }
            float mx[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) mx[k] = fmaxf(s[k], s[k + 4]);
#pragma unroll
            for (int j = 8; j < kMlaBN; j += 8)
#pragma unroll
                for (int k = 0; k < 4; ++k) mx[k] = fmax3(mx[k], s[j + k], s[j + 4 + k]);
            const float row_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            const float m_new = (row_max > m + kMlaRescaleThreshold) ? row_max : m;
            const float alpha = ex2_approx(m - m_new);  // 1 if unchanged, 0 on the first tile
            const bool rescale = i > 0 && __any_sync(0xffffffffu, m_new != m);
            m = m_new;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                const float p0 = ex2_approx(s[2 * x] - m);
                const float p1 = ex2_approx(s[2 * x + 1] - m);
                const int a = (x & 1) * 2;
                fadd2(acc[a], acc[a + 1], acc[a], acc[a + 1], p0, p1);
                pk[x] = pack_bf16x2(p0, p1);
            }
            // P(i) overwrites P(i-1) and O may need its correction: both wait for P.V(i-1)
            if (i > 0) {
                ok = mbar_wait_warp<true>(bar(L::kBarPvDone), (i - 1) & 1, abort_flag,
                                          status_word);
                if (!ok) break;
                tc_fence_after();
            }
            tmem_st32(lane_base + t_p, pk);
            if (rescale) {
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
            tc_fence_before();
            mbar_arrive(bar(L::kBarPFull));
            l = l * alpha + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
        }
        // epilogue: O / l of this CTA's 256 columns
        if (ok) ok = mbar_wait_warp(bar(L::kBarPvDone), (n_t - 1) & 1, abort_flag, status_word);
        if (ok) {
            // O / l through shared memory (the Q panels and the X ring are no longer read once the
            // last P.V has landed): each thread stores its row with the 16-byte chunk index XOR-ed
            // by the row, so a warp's 32 rows hit distinct banks; then every store instruction
            // writes 512 contiguous bytes of one row.  Warp w stages its 32 rows at w * 32 KiB.
            tc_fence_after();
            const float inv_l = 1.0f / l;
            const float lse_nat = (m + __log2f(l)) * 0.69314718055994531f;
            const bool split_out = p.n_splits > 1;
            const int chunks = split_out ? 64 : 32;  // 16-byte chunks per row (fp32 or bf16)
            const uint32_t stage = sbase + warp * 32768;
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
                uint32_t o[32];
                tmem_ld32(lane_base + t_o + cc * 32, o);
                tmem_wait_ld();
                if (split_out) {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const int ch = cc * 8 + q4;
                        st_shared_v4(stage + lane * 1024 + ((ch ^ lane) << 4),
                                     __float_as_uint(__uint_as_float(o[4 * q4 + 0]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[4 * q4 + 1]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[4 * q4 + 2]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[4 * q4 + 3]) * inv_l));
                    }
                } else {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int ch = cc * 4 + q4;
                        st_shared_v4(stage + lane * 512 + ((ch ^ lane) << 4),
                                     pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv_l,
                                                 __uint_as_float(o[8 * q4 + 1]) * inv_l),
                                     pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv_l,
                                                 __uint_as_float(o[8 * q4 + 3]) * inv_l),
                                     pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv_l,
                                                 __uint_as_float(o[8 * q4 + 5]) * inv_l),
                                     pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv_l,
                                                 __uint_as_float(o[8 * q4 + 7]) * inv_l));
                    }
                }
            }
            __syncwarp();
            const int row_bytes = chunks * 16;
            const int h0 = ht * kMlaHeads + warp * 32;  // this warp's first head
            // (under the cluster merge the staged rows stay where they are)
            for (int rr = 0; rr < (p.cluster_merge ? 0 : 32); ++rr) {
                if (h0 + rr >= p.H) break;  // warp-uniform
                if (!ATTN_DCHECK(b < p.B && split < p.n_splits && r < 2)) break;
                const size_t bh_r = static_cast<size_t>(b) * p.H + h0 + rr;
                uint8_t* dst = split_out
                    ? reinterpret_cast<uint8_t*>(p.ws_o + (static_cast<size_t>(split) * p.B * p.H + bh_r) * kMlaDc + r * 256)
                    : reinterpret_cast<uint8_t*>(p.out + bh_r * kMlaDc + r * 256);
                for (int ch = lane; ch < chunks; ch += 32) {
                    uint32_t a, b2, c2, d;
                    ld_shared_v4(stage + rr * row_bytes + ((ch ^ rr) << 4), a, b2, c2, d);
                    *reinterpret_cast<uint4*>(dst + ch * 16) = make_uint4(a, b2, c2, d);
                }
            }
            if (p.cluster_merge) {
                reinterpret_cast<float*>(smem + L::kLseStage)[row] = lse_nat;
            } else if (h < p.H && ATTN_DCHECK(b < p.B && split < p.n_splits)) {
                const size_t bh = static_cast<size_t>(b) * p.H + h;
                if (split_out && r == 0)
                    p.ws_lse[static_cast<size_t>(split) * p.B * p.H + bh] = lse_nat;
                else if (!split_out && r == 0)
                    p.lse[bh] = lse_nat;
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMlaMmaA) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (p.cluster_merge) {
        cluster_sync_all();  // every CTA of the cluster has staged its O_s and LSE_s (or gave up)
        if (warp < 4) mla_cluster_merge(p, sbase, b, ht, r, split, warp, lane);
        cluster_sync_all();  // no CTA leaves while another still reads its shared memory
    }
}

// Merge of the token splits: LSE = log sum_s exp(LSE_s), out_c = sum_s exp(LSE_s - LSE) O_s, the
// safe-softmax combination of section 2.4's split-T.  A 512-thread block serves 4 / groups rows;
// within a row, thread (g, i) sums columns 4i .. 4i+3 over the splits s = g (mod groups), so each
// split's row is read as one coalesced 2 KiB sweep, and the groups are added in shared memory.
// groups (1, 2 or 4) grows with the split count to keep enough loads in flight.
constexpr int kMlaMergeThreads = 512;

__host__ __device__ constexpr int mla_merge_groups(int n_splits) {
    return n_splits >= 4 ? 4 : (n_splits >= 2 ? 2 : 1);
}

__global__ void __launch_bounds__(kMlaMergeThreads)
    mla_merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                     __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int BH,
                     int n_splits) {
    constexpr int kCols = kMlaDc / 4;  // float4 columns per row
    __shared__ float w_s[4][64];       // n_splits <= 64
    __shared__ float stats[4][2];
    __shared__ float4 part[3][kCols];
    const int groups = mla_merge_groups(n_splits);
    const int rows_per_block = 4 / groups;
    const int tid = threadIdx.x;
    const int rl = tid / (groups * kCols);  // row within the block
    const int g = (tid / kCols) % groups, col = tid % kCols;
    const int row = static_cast<int>(blockIdx.x) * rows_per_block + rl;
    const bool live = row < BH;
    griddep_wait();  // launched as the decode kernel's dependant: its partials are complete
    if (live && g == 0 && col < 32) {  // one warp per row: weights and statistics
        const int lane = col;
        float mx = -INFINITY;
        for (int s = lane; s < n_splits; s += 32)
            mx = fmaxf(mx, ws_lse[static_cast<size_t>(s) * BH + row]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float sum = 0.f;
        for (int s = lane; s < n_splits; s += 32) {
            const float w = __expf(ws_lse[static_cast<size_t>(s) * BH + row] - mx);
            w_s[rl][s] = w;
            sum += w;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) {
            stats[rl][0] = 1.0f / sum;
            stats[rl][1] = mx + __logf(sum);
        }
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
#pragma unroll 8
        for (int s = g; s < n_splits; s += groups) {
            const float w = w_s[rl][s];
            const float4 v = reinterpret_cast<const float4*>(
                ws_o + (static_cast<size_t>(s) * BH + row) * kMlaDc)[col];
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
    }
    if (g > 0) part[rl * (groups - 1) + g - 1][col] = acc;
    __syncthreads();
    if (live && g == 0) {
        for (int k = 1; k < groups; ++k) {
            const float4 v = part[rl * (groups - 1) + k - 1][col];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float inv = stats[rl][0];
        uint2 w2;
        w2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        w2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        if (ATTN_DCHECK(row < BH && col < kMlaDc / 4))
            *reinterpret_cast<uint2*>(out + static_cast<size_t>(row) * kMlaDc + 4 * col) = w2;
        if (col == 0) lse[row] = stats[rl][1];
    }
}

}  // namespace gb300attn
