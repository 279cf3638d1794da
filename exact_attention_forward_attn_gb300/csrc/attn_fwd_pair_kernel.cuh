// attn_fwd_pair_kernel.cuh - the fused exact-attention forward on CTA pairs (tcgen05 cta_group::2),
// for head dimensions padded to 128.
//
// What it computes is what attn_fwd_kernel computes ("Attention Kernel 实现与正确性验证",
// walkerchi.com, sections 1.1-1.2; "Triton-CUDA Attention", skillmd.com, online-softmax algorithm
// and the Causal/GQA variants; "Flash Attention 与 Kernel 优化", fangpin.github.io, running state
// and saved LSE): per (b, hq) and query row i, O[i,:] = softmax_j(sm_scale q_i.k_j) V over the
// visible keys and LSE[i], with the online-softmax recurrence over 128-key tiles in the exp2
// domain, the lazy maximum (moved only when it grows by more than 8) and the same epilogue.
//
// Why pairs.  In the one-CTA kernel every K/V step moves ~320 KB through each SM's shared memory
// (the K and V tiles written by the TMA, read by the S and P.V MMAs of both Q tiles, plus P's
// shared-memory half), close to what an SM's shared memory delivers.  Here a cluster of two CTAs
// on two SMs shares every MMA: M = 256 query rows, CTA r supplying rows 128r..128r+127 of A (its
// own Q or P) and half of B - for S = Q K^T keys 64r..64r+63 of the key tile, for O += P V
// output columns 64r..64r+63 of V - so each SM loads and reads half of every K and V tile:
// ~224 KB per step.  CTA r's tensor memory holds its own 128 rows of S and O.
// Measured on GB300 it is nevertheless slower than the one-CTA kernel (0.62-0.85x): a pair MMA
// takes ~96 (SS) / ~123 (TS) cycles to issue for 64 cycles of work per SM, so two issuers per
// two SMs halve the issue capacity per SM, and every step's commits and P-ready arrives cross
// between the SMs.  attn_fwd therefore does not use it; attn_fwd_test_kernel runs it.
//
// Work item: a quad of four 128-row Q tiles of one (b, hq).  M-tile t (t = 0, 1) of the item is
// rows 512u + 256t .. + 255; CTA r holds Q tile 4u + 2t + r of it.  Under the causal mask an
// M-tile's key range ends at the diagonal of its second half, so CTA 0's rows see their last key
// tile fully masked (P = 0 there): 1/(2 n) of the MMA work of an M-tile of n key tiles.
//
// Roles (384 threads per CTA, in both CTAs unless marked):
//   warp 10     TMA producer: lane 0 of CTA 0 claims the items and publishes them to both CTAs'
//               item rings; lanes 0-1 stream this CTA's half of K_j (two 64 x 64 boxes), lanes 2-3
//               its half of V_j (two 64 x 64 boxes), into an 8-slot ring of 16 KB halves.  Every
//               load signals CTA 0's full barrier (cta_group::2 TMA), where CTA 0's lanes post the
//               bytes of both halves.
//   warps 8, 9  Q_t loaders (both CTAs, after the previous item's last S MMA of tile t has read the
//               buffer) and, in CTA 0 only, the MMA issuers of M-tile t: S = Q K^T (SS), O += P V
//               (TS for keys 0-63 with P in TMEM, SS for keys 64-127 with P in shared memory);
//               every commit arrives on both CTAs' barriers (multicast).
//   warps 0-7   softmax of this CTA's rows of M-tile 0 / 1 (one thread per row), as in the one-CTA
//               kernel; P-ready arrives, one per warp, on CTA 0's barriers.
//   warp 11     no role.
// Every wait is bounded (1 s): a CTA whose partner stops answering times out and reports it; both
// CTAs meet at a cluster barrier before either frees its tensor memory or exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"
#include "ptx.cuh"

namespace gb300attn {

constexpr int kPairStages = 8;     // K/V ring slots per CTA (one half tile each)
constexpr int kPairLoadLanes = 4;  // producer lanes: K boxes 0, 1; V boxes 0, 1

struct PairSmem {
    static constexpr int kPanelBytes = kBM * 64 * 2;          // 128 rows x 64 bf16, 16 KB
    static constexpr int kBoxBytes = 64 * 64 * 2;             // one TMA box: 64 rows x 64 bf16
    static constexpr int kQTileBytes = 2 * kPanelBytes;       // 128 rows x 128 columns
    static constexpr int kSlotBytes = 2 * kBoxBytes;          // half a K or V tile, 16 KB
    static constexpr int kQ = 0;                              // Q tiles [2]
    static constexpr int kKV = kQ + 2 * kQTileBytes;          // K/V ring
    static constexpr int kP1 = kKV + kPairStages * kSlotBytes;  // P keys 64..127 / O staging [2]
    static constexpr int kP1Bytes = kPanelBytes;
    static constexpr int kBars = kP1 + 2 * kP1Bytes;
    // barrier indices; "leader" barriers are used in CTA 0 only
    static constexpr int kBarQFull = 0;                          // [2] leader: both CTAs' Q_t
    static constexpr int kBarQFree = kBarQFull + 2;              // [2] the item's last S of tile t
    static constexpr int kBarKvFull = kBarQFree + 2;             // [8] leader: both halves landed
    static constexpr int kBarKvEmpty = kBarKvFull + kPairStages;  // [8] both M-tiles' MMAs read it
    static constexpr int kBarSFull = kBarKvEmpty + kPairStages;  // [2]
    static constexpr int kBarPReady = kBarSFull + 2;             // [2 tiles][2 halves] leader
    static constexpr int kBarPVDone = kBarPReady + 4;            // [2]
    static constexpr int kBarODone = kBarPVDone + 2;             // [2]
    static constexpr int kBarTurn = kBarODone + 2;               // [2 groups][2] exp2 turn tokens
    static constexpr int kBarItemFull = kBarTurn + 4;            // [2] item ring slot written
    static constexpr int kBarItemEmpty = kBarItemFull + 2;       // [2] leader: read by all readers
    static constexpr int kBarDrain = kBarItemEmpty + 2;          // [2] leader: issuers' last MMAs
    static constexpr int kNumBars = kBarDrain + 2;
    static constexpr int kItems = kBars + kNumBars * 8;          // int[2]: the item ring
    static constexpr int kTmemSlot = kItems + 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 232448, "pair kernel shared memory exceeds the per-block limit");
    // Readers of an item ring slot besides CTA 0's claiming lane, one arrival each on CTA 0's
    // item-empty barrier: CTA 0's other producer lanes, both CTAs' Q-loader/issuer warps and
    // softmax warps, and all of CTA 1's producer lanes.
    static constexpr int kItemReaders = (kPairLoadLanes - 1) + kPairLoadLanes + 2 * (2 + 8);
};

// Work item of the pair kernel: a quad of Q tiles (p.n_pairs holds the quads per (b, hq)).
// Order as in decode_work: L2-sized blocks of KV heads, heaviest quads first.
__device__ __forceinline__ FwdWork decode_quad_work(const AttnParams& p, int item) {
    FwdWork w;
    w.split = 0;
    const int per_kv = p.n_pairs * p.group;
    const int blk = item / (p.kv_block * per_kv);
    const int in_blk = item % (p.kv_block * per_kv);
    const int kvs = min(p.kv_block, p.B * p.Hkv - blk * p.kv_block);
    const int bh_kv = blk * p.kv_block + (in_blk % (kvs * p.group)) / p.group;
    const int rem = in_blk % p.group;
    const int quad = p.n_pairs - 1 - in_blk / (kvs * p.group);
    w.b = bh_kv / p.Hkv;
    w.hkv = bh_kv % p.Hkv;
    w.hq = w.hkv * p.group + rem;
    w.bh = w.b * p.Hq + w.hq;
    w.tile0 = 4 * quad;  // M-tile t holds Q tiles tile0 + 2t (CTA 0) and tile0 + 2t + 1 (CTA 1)
    w.kv_begin = 0;
    w.last0 = p.causal ? min(p.n_tiles - 1, w.tile0 + 1) : p.n_tiles - 1;
    w.last1 = p.causal ? min(p.n_tiles - 1, w.tile0 + 3) : p.n_tiles - 1;
    w.part0 = true;
    w.part1 = w.tile0 + 2 < p.n_tiles;
    w.kv_end = (w.part1 ? w.last1 : w.last0) + 1;
    return w;
}

// tmap_q: box 64 x 128 rows; tmap_k, tmap_v: box 64 x 64 rows (half tiles).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const AttnParams p,
                         unsigned int* status_word) {
    using L = PairSmem;
    constexpr int D = 128;
    constexpr int kPanels = D / 64;
    constexpr uint32_t kIdescS = idesc_bf16_f32(256, kBN, 0);  // Q (K-major) x K (K-major)
    constexpr uint32_t kIdescPV = idesc_bf16_f32(256, D, 1);   // P x V (MN-major)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    auto bar = [=](int i) -> uint32_t { return sbase + L::kBars + 8u * i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
    volatile int* item_ring = reinterpret_cast<volatile int*>(smem + L::kItems);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    // A barrier of CTA 0 as a shared::cluster address (valid in both CTAs).
    auto lbar = [=](int i) -> uint32_t { return dsmem_addr(bar(i), 0); };

    // ---- setup (once per CTA): barriers, the pair's tensor memory ------------------------------
    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(L::kBarQFull + t), kPanels);  // CTA 0's two Q lanes post both CTAs' bytes
            mbar_init(bar(L::kBarQFree + t), 1);
            mbar_init(bar(L::kBarSFull + t), 1);
            mbar_init(bar(L::kBarPReady + 2 * t + 0), 8);  // one per softmax warp of both CTAs
            mbar_init(bar(L::kBarPReady + 2 * t + 1), 8);
            mbar_init(bar(L::kBarPVDone + t), 1);
            mbar_init(bar(L::kBarODone + t), 1);
            mbar_init(bar(L::kBarTurn + 2 * t + 0), 128);
            mbar_init(bar(L::kBarTurn + 2 * t + 1), 128);
            mbar_init(bar(L::kBarItemFull + t), 1);
            mbar_init(bar(L::kBarItemEmpty + t), L::kItemReaders);
            mbar_init(bar(L::kBarDrain + t), 1);
        }
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(bar(L::kBarKvFull + s), 2);   // CTA 0's two lanes of the entry
            mbar_init(bar(L::kBarKvEmpty + s), 2);  // one release per M-tile issuer
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp0) {  // one warp of each CTA allocates the pair's columns together
        tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == kLoadWarp && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before either touches the other's
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Item ring reader (every role but CTA 0's claiming lane): the k-th item, or -1 at the end.
    auto read_item = [&](int k, bool whole_warp) -> int {
        const int slot = k & 1;
        const uint32_t ph = static_cast<uint32_t>(k >> 1) & 1u;
        bool ok;
        if (whole_warp)
            ok = mbar_wait_cluster_warp(bar(L::kBarItemFull + slot), ph, abort_flag, status_word);
        else
            ok = mbar_wait_cluster_bounded(bar(L::kBarItemFull + slot), ph, abort_flag,
                                           status_word);
        if (!ok) return -1;
        int item = item_ring[slot];
        if (whole_warp) {
            item = __reduce_min_sync(0xffffffffu, item);
            if (lane == 0) mbar_arrive_cluster(lbar(L::kBarItemEmpty + slot));
            __syncwarp();
        } else {
            mbar_arrive_cluster(lbar(L::kBarItemEmpty + slot));
        }
        return item;
    };

    if (warp >= kMmaWarp0) {
    setmaxnreg_dec<kOtherRegs>();
    if (warp == kLoadWarp) {
        // ============== TMA producer: this CTA's halves of K_j and V_j, one lane per box =========
        if (lane < kPairLoadLanes) {
            ArmedPhases kv_armed;  // CTA 0: phases of its full barriers it armed (both halves)
            bool issued = false;   // CTA 1: issued loads (waited out after an abort)
            int ring = 0;
            bool claims_done = false;
            int claim_round = 0;
            const unsigned int pair_id = cluster_id_x(), pairs = cluster_count_x();
            auto claim = [&]() -> int {
                return claim_next_item(p.sched, p.items, claim_round, claims_done, pair_id, pairs);
            };
            const bool claimer = leader && lane == 0;
            for (int k = 0;; ++k) {
                int item;
                if (claimer) {
                    const int slot = k & 1;
                    if (!mbar_wait_cluster_bounded(bar(L::kBarItemEmpty + slot),
                                                   (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u,
                                                   abort_flag, status_word))
                        break;
                    item = k == 0 ? static_cast<int>(pair_id) : claim();
                    item_ring[slot] = item;
                    st_dsmem_u32(dsmem_addr(smem_addr(const_cast<int*>(item_ring) + slot), 1),
                                 static_cast<uint32_t>(item));
                    mbar_arrive(bar(L::kBarItemFull + slot));
                    mbar_arrive_cluster(dsmem_addr(bar(L::kBarItemFull + slot), 1));
                } else {
                    item = read_item(k, false);
                }
                if (item < 0) break;
                const FwdWork w = decode_quad_work(p, item);
                if (lane == 0) (void)ATTN_DCHECK(item < p.items && work_in_range(p, w));
                {
                    const int kv = lane >> 1, h = lane & 1;
                    const CUtensorMap* map = kv ? &tmap_v : &tmap_k;
                    // K: keys j*128 + 64*rank + [0, 64), columns 64h..; V: keys j*128 + 64h +
                    // [0, 64), columns 64*rank.. (this CTA's half of the output columns)
                    const int c0 = kv ? 64 * static_cast<int>(rank) : 64 * h;
                    const int r0 = kv ? 64 * h : 64 * static_cast<int>(rank);
                    bool ok = true;
                    for (int j = w.kv_begin; j < w.kv_end; ++j) {
                        const int idx = ring + 2 * (j - w.kv_begin) + kv;
                        const int slot = idx % kPairStages;
                        const uint32_t ph = (idx / kPairStages) & 1;
                        ok = mbar_wait_bounded(bar(L::kBarKvEmpty + slot), ph ^ 1u, abort_flag,
                                               status_word);
                        if (!ok) break;
                        if (idx == p.stall_item) continue;  // test hook: never deliver this entry
                        if (leader) {
                            mbar_arrive_expect_tx(bar(L::kBarKvFull + slot), 2 * L::kBoxBytes);
                            kv_armed.arm(slot, ph);
                        }
                        issued = true;
                        tma_load_4d_pair(sbase + L::kKV + slot * L::kSlotBytes + h * L::kBoxBytes,
                                         map, lbar(L::kBarKvFull + slot), c0, j * kBN + r0, w.hkv,
                                         w.b);
                    }
                    if (!ok) break;
                }
                ring += 2 * (w.kv_end - w.kv_begin);
            }
            if (claimer)
                while (!claims_done) (void)claim();
            if (*abort_flag) {
                const uint64_t deadline = globaltimer_ns() + kDrainLimitNs;
                if (leader) {
                    kv_armed.drain(bar(L::kBarKvFull), deadline);
                } else if (issued) {  // its loads signal CTA 0's barriers: give them time to land
                    while (globaltimer_ns() < deadline) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
        // ===== Q_t loaders (both CTAs) and, in CTA 0, the MMA issuers of M-tile t ================
        const int t = warp - kMmaWarp0;
        const uint32_t s_tmem = tmem + tmem_s_col(t);
        const uint32_t o_tmem = tmem + tmem_o_col(t);
        const uint32_t qa = sbase + L::kQ + t * L::kQTileBytes;
        auto kv_slot = [](int idx) { return idx % kPairStages; };
        auto kv_phase = [](int idx) { return static_cast<uint32_t>((idx / kPairStages) & 1); };
        auto wait_full = [=](int idx) {
            return mbar_wait_cluster_warp(bar(L::kBarKvFull + kv_slot(idx)), kv_phase(idx),
                                          abort_flag, status_word);
        };
        // S = Q K^T: per CTA, A = its Q_t (128 x 128), B = its 64 keys of K_j (two 64 x 64 boxes)
        auto s_mma = [=](int kslot) {
            const uint32_t ka = sbase + L::kKV + kslot * L::kSlotBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                mma_pair_ss_warp(s_tmem,
                                 smem_desc_sw128(qa + (kk >> 2) * L::kPanelBytes + (kk & 3) * 32,
                                                 16, 1024),
                                 smem_desc_sw128(ka + (kk >> 2) * L::kBoxBytes + (kk & 3) * 32,
                                                 16, 1024),
                                 kIdescS, kk > 0);
            }
        };
        // O += P V in two halves (keys 0-63: P from TMEM over S; keys 64-127: P from smem).  Per
        // CTA, B = its 64 output columns of V_j (128 keys x 64, MN-major).
        const uint32_t p1a = sbase + L::kP1 + t * L::kP1Bytes;
        auto pv_first = [=](int vslot, bool accumulate_first) {
            const uint32_t va = sbase + L::kKV + vslot * L::kSlotBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_pair_ts_warp(o_tmem, s_tmem + kk * 8,
                                 smem_desc_sw128(va + kk * 2048, L::kSlotBytes, 1024), kIdescPV,
                                 (accumulate_first || kk > 0) ? 1u : 0u);
        };
        auto pv_second = [=](int vslot) {
            const uint32_t va = sbase + L::kKV + vslot * L::kSlotBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_pair_ss_warp(o_tmem, smem_desc_sw128(p1a + kk * 32, 16, 1024),
                                 smem_desc_sw128(va + (4 + kk) * 2048, L::kSlotBytes, 1024),
                                 kIdescPV, 1u);
        };

        ArmedPhases q_armed;  // CTA 0: its Q-full phases (both CTAs' bytes)
        bool q_issued = false;
        int ring = 0;
        uint32_t steps = 0;
        uint32_t q_items = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = read_item(k, true);
            if (item < 0) break;
            const FwdWork w = decode_quad_work(p, item);
            const bool part = t == 0 ? w.part0 : w.part1;
            const int last = part ? (t == 0 ? w.last0 : w.last1) : w.kv_begin - 1;
            if (part) {
                // this CTA's Q tile of M-tile t, once the previous item's last S MMA has read it
                if (lane < kPanels) {
                    const bool qok = q_items == 0 ||
                                     mbar_wait_bounded(bar(L::kBarQFree + t), (q_items - 1) & 1u,
                                                       abort_flag, status_word);
                    if (qok) {
                        if (leader) {
                            mbar_arrive_expect_tx(bar(L::kBarQFull + t), 2 * L::kPanelBytes);
                            q_armed.arm(t, q_items);
                        }
                        q_issued = true;
                        tma_load_4d_pair(qa + lane * L::kPanelBytes, &tmap_q,
                                         lbar(L::kBarQFull + t), lane * 64,
                                         (w.tile0 + 2 * t + static_cast<int>(rank)) * kBM, w.hq,
                                         w.b);
                    }
                }
                __syncwarp();
                if (leader) {
                    ok = mbar_wait_cluster_warp(bar(L::kBarQFull + t), q_items & 1u, abort_flag,
                                                status_word);
                    if (ok) ok = wait_full(ring);
                    if (ok) {
                        tc_fence_after();
                        s_mma(kv_slot(ring));
                        mma_commit_pair_warp(bar(L::kBarSFull + t));
                        mma_commit_pair_warp(bar(L::kBarKvEmpty + kv_slot(ring)));
                        if (last == w.kv_begin) mma_commit_pair_warp(bar(L::kBarQFree + t));
                    }
                    for (int j = w.kv_begin; ok && j <= last; ++j) {
                        const int vidx = ring + 2 * (j - w.kv_begin) + 1;  // V_j
                        const int kidx = vidx + 1;                         // K_{j+1}
                        ok = wait_full(vidx);
                        if (ok)
                            ok = mbar_wait_cluster_warp<true>(bar(L::kBarPReady + 2 * t + 0),
                                                              steps & 1u, abort_flag,
                                                              status_word);
                        if (!ok) break;
                        tc_fence_after();
                        pv_first(kv_slot(vidx), j > w.kv_begin);
                        if (j + 1 <= last) {  // S(j+1) overwrites the first half of P(j)
                            ok = wait_full(kidx);
                            if (!ok) break;
                            tc_fence_after();
                            s_mma(kv_slot(kidx));
                            mma_commit_pair_warp(bar(L::kBarSFull + t));
                            mma_commit_pair_warp(bar(L::kBarKvEmpty + kv_slot(kidx)));
                            if (j + 1 == last) mma_commit_pair_warp(bar(L::kBarQFree + t));
                        }
                        ok = mbar_wait_cluster_warp<true>(bar(L::kBarPReady + 2 * t + 1),
                                                          steps & 1u, abort_flag, status_word);
                        if (!ok) break;
                        tc_fence_after();
                        pv_second(kv_slot(vidx));
                        ++steps;
                        mma_commit_pair_warp(bar(L::kBarPVDone + t));
                        if (j == last) mma_commit_pair_warp(bar(L::kBarODone + t));
                        mma_commit_pair_warp(bar(L::kBarKvEmpty + kv_slot(vidx)));
                    }
                }
                ++q_items;
            }
            if (leader) {
                // K/V entries of this item that M-tile t does not use: released once landed
                for (int j = last + 1; ok && j < w.kv_end; ++j) {
                    for (int kv = 0; ok && kv < 2; ++kv) {
                        const int idx = ring + 2 * (j - w.kv_begin) + kv;
                        ok = wait_full(idx);
                        if (ok) mma_commit_pair_warp(bar(L::kBarKvEmpty + kv_slot(idx)));
                    }
                }
            }
            ring += 2 * (w.kv_end - w.kv_begin);
        }
        if (*abort_flag) {
            const uint64_t deadline = globaltimer_ns() + kDrainLimitNs;
            if (leader) {
                // every MMA this warp issued has completed before the pair's memory is released
                mma_commit_pair_warp(bar(L::kBarDrain + t));
                if (lane == 0)
                    while (!mbar_try_wait(bar(L::kBarDrain + t), 0) && globaltimer_ns() < deadline) {
                    }
                q_armed.drain(bar(L::kBarQFull), deadline);
            } else if (q_issued && lane < kPanels) {
                while (globaltimer_ns() < deadline) {
                }
            }
        }
        __syncwarp();
    }
    } else {
        setmaxnreg_inc<kSoftmaxRegs>();
        // ====================== softmax + epilogue (warps 0-7, both CTAs) ======================
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + tmem_s_col(t);
        const uint32_t o_addr = tmem + lane_base + tmem_o_col(t);
        const uint32_t p1 = sbase + L::kP1 + t * L::kP1Bytes;
        const uint32_t pready0 = lbar(L::kBarPReady + 2 * t + 0);
        const uint32_t pready1 = lbar(L::kBarPReady + 2 * t + 1);
        const float c = p.scale_log2;
        constexpr uint32_t kPhStep = 1u, kPhODone = 4u;
        uint32_t ph = 0;
        uint32_t tok = 0;
        bool ok = true;
        for (int k = 0;; ++k) {
            const int item = read_item(k, true);
            if (!named_barrier_and(1 + t, 128, item >= 0)) break;
            int n, first_mask, tok_until, diag;
            {
                const FwdWork w = decode_quad_work(p, item);
                if (!(t == 0 ? w.part0 : w.part1)) continue;
                const bool pingpong = w.part0 && w.part1;
                const int q_tile = w.tile0 + 2 * t + static_cast<int>(rank);
                const int last = t == 0 ? w.last0 : w.last1;
                n = last - w.kv_begin + 1;
                // Masked steps: under the causal mask every step from this CTA's diagonal tile on
                // (CTA 0 has one more step, wholly masked); otherwise a ragged last key tile.
                diag = q_tile - w.kv_begin;
                first_mask = p.causal ? diag : ((p.N % kBN) != 0 ? p.n_tiles - 1 - w.kv_begin : n);
                tok_until = !pingpong ? -1 : (t == 0 ? n - 1 : w.last0 - w.kv_begin);
            }
            float m = -INFINITY;
            float l = 0.f;
            for (int i = 0; i < n; ++i) {
                ok = mbar_wait_warp<true>(bar(L::kBarSFull + t), ph & kPhStep, abort_flag,
                                          status_word);
                if (!ok) break;
                tc_fence_after();
                if (i >= first_mask) {
                    // first masked key of this row in this tile (<= 0: all of them)
                    const int lim = p.causal ? row + 1 - (i - diag) * kBN
                                             : p.N - (p.n_tiles - 1) * kBN;
#pragma unroll
                    for (int cc = 0; cc < kBN / 32; ++cc) {
                        uint32_t r[32];
                        tmem_ld32(s_addr + cc * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 32; ++x)
                            if (cc * 32 + x >= lim) r[x] = __float_as_uint(-INFINITY);
                        tmem_st32(s_addr + cc * 32, r);
                    }
                    tmem_wait_st();
                }
                float s[kBN];
                {
                    uint32_t r[kBN];
#pragma unroll
                    for (int cc = 0; cc < kBN / 32; ++cc)
                        tmem_ld32(s_addr + cc * 32,
                                  *reinterpret_cast<uint32_t(*)[32]>(&r[cc * 32]));
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < kBN; ++x) s[x] = __uint_as_float(r[x]);
                }
                float mx[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx[q] = fmaxf(s[q], s[q + 8]);
#pragma unroll
                for (int x = 16; x < kBN; x += 16)
#pragma unroll
                    for (int q = 0; q < 8; ++q) mx[q] = fmax3(mx[q], s[x + q], s[x + 8 + q]);
                const float row_max =
                    fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                const float m_cand = row_max * c;
                const float m_new = (m_cand > m + kRescaleThreshold) ? m_cand : m;
                const float alpha = ex2_approx(m - m_new);
                const bool rescale = i > 0 && __any_sync(0xffffffffu, m_new != m);
                m = m_new;
                const float neg_m = -m;
                if (i <= tok_until && (t == 1 || tok >= 2)) {
                    const uint32_t x = t == 0 ? tok - 2 : tok;
                    ok = mbar_wait_warp<true>(bar(L::kBarTurn + 2 * t + (x & 1)), (x >> 1) & 1u,
                                              abort_flag, status_word);
                    if (!ok) break;
                }
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                auto exp_half = [&](int h, uint32_t (&pk)[32]) {
#pragma unroll
                    for (int i2 = 0; i2 < 32; ++i2) {
                        const int col = h * 64 + 2 * i2;
                        float x0, x1;
                        ffma2(x0, x1, s[col], s[col + 1], c, c, neg_m, neg_m);
                        const float p0 = ex2_approx(x0);
                        const float p1v = ex2_approx(x1);
                        const int a = (i2 & 1) * 2;
                        fadd2(acc[a], acc[a + 1], acc[a], acc[a + 1], p0, p1v);
                        pk[i2] = pack_bf16x2(p0, p1v);
                    }
                };
                const bool prev_pv = i > 0;
                {
                    uint32_t pk[32];
                    exp_half(0, pk);
                    tmem_st32(s_addr, pk);
                    if (rescale) {
                        ok = mbar_wait_warp(bar(L::kBarPVDone + t), (ph & kPhStep) ^ 1u,
                                            abort_flag, status_word);
                        if (!ok) break;
#pragma unroll
                        for (int cc = 0; cc < D / 32; ++cc) {
                            uint32_t r[32];
                            tmem_ld32(o_addr + cc * 32, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int x = 0; x < 32; ++x)
                                r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
                            tmem_st32(o_addr + cc * 32, r);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(pready0);
                }
                {
                    uint32_t pk[32];
                    exp_half(1, pk);
                    if (prev_pv && !rescale) {
                        ok = mbar_wait_warp(bar(L::kBarPVDone + t), (ph & kPhStep) ^ 1u,
                                            abort_flag, status_word);
                        if (!ok) break;
                    }
                    const uint32_t prow = p1 + row * 128;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4(prow + ((ch ^ (row & 7)) << 4), pk[4 * ch], pk[4 * ch + 1],
                                     pk[4 * ch + 2], pk[4 * ch + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(pready1);
                }
                l = l * alpha + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
                if (i <= tok_until) {
                    mbar_arrive(bar(L::kBarTurn + 2 * (t ^ 1) + (tok & 1)));
                    ++tok;
                }
                ph ^= kPhStep;
            }
            if (ok) ok = mbar_wait_warp(bar(L::kBarODone + t), (ph & kPhODone) ? 1u : 0u,
                                        abort_flag, status_word);
            ph ^= kPhODone;
            if (!named_barrier_and(1 + t, 128, ok)) break;
            tc_fence_after();
            const FwdWork we = decode_quad_work(p, opaque_int(item));
            const int q_row0 = (we.tile0 + 2 * t + static_cast<int>(rank)) * kBM;
            const int row_g = q_row0 + row;
            const float inv_l = 1.0f / l;
            // ---- epilogue: O = acc / l -> bf16 through this tile's P panel, coalesced stores ----
            __nv_bfloat16* obase = p.out + we.b * p.o_sb + we.hq * p.o_sh;
            const int tid = quarter * 32 + lane;
#pragma unroll
            for (int h = 0; h < kPanels; ++h) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + h * 64 + cc * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16) {
                        uint32_t v4[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            v4[x] = pack_bf16x2(__uint_as_float(r[c16 * 8 + 2 * x]) * inv_l,
                                                __uint_as_float(r[c16 * 8 + 2 * x + 1]) * inv_l);
                        const int chunk = cc * 4 + c16;
                        st_shared_v4(p1 + row * 128 + ((chunk ^ (row & 7)) << 4), v4[0], v4[1],
                                     v4[2], v4[3]);
                    }
                }
                named_barrier_sync(1 + t, 128);
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int flat = it * 128 + tid;
                    const int r = flat >> 3, ch = flat & 7;
                    uint32_t v0, v1, v2, v3;
                    ld_shared_v4(p1 + r * 128 + ((ch ^ (r & 7)) << 4), v0, v1, v2, v3);
                    const int col = h * 64 + ch * 8;
                    if (q_row0 + r < p.N && col < p.d_out && ATTN_DCHECK(work_in_range(p, we)))
                        st_global_v4u(obase + static_cast<long long>(q_row0 + r) * p.o_sn + col,
                                      v0, v1, v2, v3);
                }
                named_barrier_sync(1 + t, 128);
            }
            if (row_g < p.N &&
                ATTN_DCHECK(static_cast<size_t>(we.bh) * p.N + row_g <
                            static_cast<size_t>(p.B) * p.Hq * p.N))
                p.lse[static_cast<size_t>(we.bh) * p.N + row_g] = (m + __log2f(l)) * kLn2;
        }
        __syncwarp();
    }

    // ---- teardown: neither CTA frees the pair's tensor memory or leaves while the other may
    // still use its shared memory -------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == kMmaWarp0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace gb300attn
