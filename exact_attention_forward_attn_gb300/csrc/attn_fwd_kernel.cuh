// attn_fwd_kernel.cuh - fused exact-attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes (per batch b, query head hq, query row i):
//   O[i,:] = softmax_j(sm_scale * q_i . k_j)[j in J(i)] . V,   LSE[i] = ln sum_j exp(sm_scale q_i.k_j)
//   with h_kv = hq * Hkv / Hq and J(i) = {0..i} (causal, top-left) or {0..N-1}.
// How ("Attention Kernel 实现与正确性验证", walkerchi.com, sections 1.1-1.2; "Triton-CUDA Attention",
// skillmd.com, online-softmax algorithm and the Causal/GQA variants; "Flash Attention 与 Kernel
// 优化", fangpin.github.io, running state and saved LSE):
//   a Q tile stays on chip while K/V tiles stream past it; per KV tile the running row maximum m,
//   the running denominator l and the fp32 output accumulator are updated with the online-softmax
//   recurrence (exp2 domain: scores are pre-multiplied by sm_scale*log2(e)); after the last tile
//   O = acc / l and LSE = ln2 * (m + log2 l).  The N x N score matrix never leaves the SM.
//
// GB300 mapping (persistent: one CTA per SM, 384 threads, each CTA works through pairs of
// 128-row Q tiles that it claims from a per-launch counter in global memory):
//   warp 10     TMA producer: lane 0 claims the next work item and publishes it through a 2-slot
//               item ring in shared memory; one lane per 64-column panel stream loads K_j, V_j
//               through a 4-slot mbarrier ring, so the next item's K and V load while the
//               current item finishes.
//   warps 8, 9  MMA issuers (one lane each), warp 8 + t for Q tile t: loads Q_t of each item as
//               soon as the previous item's last S MMA has read the buffer; S_t = Q_t K_j^T (SS
//               form, fp32 in TMEM) and O_t += P_t V_j (P from TMEM, V from smem);
//               tcgen05.commit signals completion.  Warp 11 has no role.
//   warps 0-3   softmax for Q tile 0, warps 4-7 for Q tile 1: one thread per query row reads its
//               S row from TMEM, masks (diagonal causal tile / ragged last key tile only), updates
//               m and l, rescales its O row in TMEM when m moved, writes P (bf16): keys 0-63 over
//               S in TMEM, keys 64-127 into a swizzled smem panel; after the last tile it
//               normalises O, stages it through that panel one 64-column panel at a time and
//               writes it with coalesced 16-byte stores, and writes LSE.
//   The two Q tiles ping-pong: while one softmax group works, the tensor core runs the other
//   tile's MMAs.  Across items every barrier keeps counting phases, so item k+1's first S MMAs
//   run while item k's softmax and epilogue finish.
//   The running maximum is only moved when it grows by more than 8 (log2 units): p <= 2^8 stays
//   exact in fp32/bf16 range and the final O = acc / l and LSE = m + log2 l use the same m, so
//   the result is unchanged while most O rescales are skipped.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace gb300attn {

constexpr int kBM = 128;          // query rows per Q tile (MMA M)
constexpr int kBN = 128;          // key rows per KV tile (MMA N of S, K of P.V)
constexpr int kQTiles = 2;        // Q tiles per work item
constexpr int kStages = 4;        // K/V ring slots (K_j and V_j take one slot each)
constexpr int kThreads = 384;     // 12 warps: two softmax warpgroups, one for the other roles
constexpr int kMmaWarp0 = 8;      // issues the MMAs of Q tile 0; warp 9 those of Q tile 1
constexpr int kLoadWarp = 10;     // warp 11 has no role (it completes the third warpgroup)
// Register split (setmaxnreg): the CTA is launched with kLaunchRegs per thread; the third
// warpgroup gives registers back and the softmax warpgroups take them.  The shares add up to the
// launch's total exactly (setmaxnreg.inc would wait forever for registers the launch never had,
// so the host checks the built kernel's register count before the first launch), and each SM
// sub-partition (warps w, w+4, w+8) fits its 16384 registers.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 192;
constexpr int kOtherRegs = 120;
static_assert(kLaunchRegs * kThreads == 256 * kSoftmaxRegs + 128 * kOtherRegs, "register split");
static_assert(32 * (2 * kSoftmaxRegs + kOtherRegs) <= 16384, "sub-partition register file");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
// Claim counters: the host hands each launch one of kSchedSlots counters, and a launch that
// reuses a counter is ordered after the counter's previous launch, so no two launches executing
// at the same time share one.  CTA c takes item c first, then claims items gridDim.x + 0, 1, 2,
// ... from the counter until a claim falls past the end; so a launch makes exactly `items`
// claims, and the CTA whose claim returns items - 1 (the last one) zeroes the counter for the
// next launch that gets it.  A launch without a counter (sched == nullptr: one captured into a
// CUDA graph, whose replays the host cannot order) uses a static schedule instead: in round r
// CTA c takes item r * gridDim.x + c, or r * gridDim.x + gridDim.x - 1 - c in odd rounds (a snake
// over the heaviest-first item order, so the rounds' heavy and light items even out).
constexpr int kSchedSlots = 64;

// The next item after this worker's first one (item `first`, of `workers` working in parallel:
// CTAs, or CTA pairs), or -1 past the end; `round` counts this worker's items so far, `done` is
// set by the claim past the end.
__device__ __forceinline__ int claim_next_item(unsigned int* sched, int items, int& round,
                                               bool& done, unsigned int first,
                                               unsigned int workers) {
    const unsigned int n = static_cast<unsigned int>(items);
    if (sched == nullptr) {
        const unsigned int r = static_cast<unsigned int>(++round);
        const unsigned int it = r * workers + ((r & 1u) ? workers - 1u - first : first);
        if (it < n) return static_cast<int>(it);
        done = true;
        return -1;
    }
    const unsigned int c = atomicAdd(sched, 1u);
    const unsigned int it = c + workers;
    if (it < n) return static_cast<int>(it);
    done = true;
    if (c == n - 1u) atomicExch(sched, 0u);
    return -1;
}

struct AttnParams {
    int B, Hq, Hkv, N;
    int group;         // Hq / Hkv
    int causal;
    int n_tiles;       // ceil(N / 128): number of Q tiles and of KV tiles per head
    int n_pairs;       // work items per (b, hq): ceil(n_tiles / 2), or n_tiles with one Q tile each
    float scale_log2;  // sm_scale * log2(e)
    int kv_block;      // (batch, KV head) pairs per scheduling block (their K/V fit in L2)
    float* lse;        // [B, Hq, N] fp32
    // split-KV partials (split instantiation only): KV tiles [s*split_tiles, (s+1)*split_tiles)
    int n_splits;
    int split_tiles;
    float* ws_o;       // [n_splits, B*Hq, N, D] fp32, O of each split normalised by its own l
    float* ws_lse;     // [n_splits, B*Hq, N] fp32, natural-log LSE of each split
    // Test hook (-1 normally): the producer withholds K/V ring entry `stall_item` of every CTA,
    // so the waits on it expire and the failure is reported through the status word.
    int stall_item;
    int items;             // work items of the launch (Q-tile pairs x splits)
    unsigned int* sched;   // this launch's claim counter, zero at launch (nullptr: static schedule)
    // O for the two-tile kernel's own stores: base, element strides of batch, head and row, and
    // the head dimension (columns at and past it are padding, not part of O)
    __nv_bfloat16* out;
    long long o_sb, o_sh, o_sn;
    int d_out;
};

template <int D>
struct SmemLayout {
    static constexpr int kPanelBytes = kBM * 64 * 2;        // 128 rows x 64 bf16 (one 128B-swizzle panel)
    static constexpr int kTileBytes = kBM * D * 2;          // 128 x D bf16 = D/64 panels
    static constexpr int kQ = 0;                            // Q tiles
    static constexpr int kKV = kQ + kQTiles * kTileBytes;   // K/V ring
    static constexpr int kP1 = kKV + kStages * kTileBytes;  // P keys 64..127 / O staging, [2 tiles]
    static constexpr int kP1Bytes = kBM * 64 * 2;           // one 128B-swizzle panel
    static constexpr int kBars = kP1 + 2 * kP1Bytes;
    // barrier indices
    static constexpr int kBarQFull = 0;                       // [2 tiles]
    static constexpr int kBarQFree = kBarQFull + 2;           // [2 tiles]: last S of an item done
    static constexpr int kBarKvFull = kBarQFree + 2;
    static constexpr int kBarKvEmpty = kBarKvFull + kStages;
    static constexpr int kBarSFull = kBarKvEmpty + kStages;   // [2]
    static constexpr int kBarPReady = kBarSFull + 2;          // [2 tiles][2 key halves]
    static constexpr int kBarPVDone = kBarPReady + 4;         // [2]: a step's P.V completed
    static constexpr int kBarODone = kBarPVDone + 2;          // [2]
    static constexpr int kBarTurn = kBarODone + 2;            // [2 groups][2]: exp2 turn tokens
    static constexpr int kBarItemFull = kBarTurn + 4;         // [2]: item ring slot written
    static constexpr int kBarItemEmpty = kBarItemFull + 2;    // [2]: item ring slot read by all
    static constexpr int kNumBars = kBarItemEmpty + 2;
    static constexpr int kItems = kBars + kNumBars * 8;       // int[2]: the item ring
    static constexpr int kTmemSlot = kItems + 8;
    static constexpr int kAbort = kTmemSlot + 8;
    static constexpr int kBytes = kAbort + 8;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
    // producer lanes: K panels, V panels
    static constexpr int kLoadLanes = 2 * (D / 64);
    // readers of an item ring slot besides the claiming lane: the other producer lanes, the two
    // issuer warps and the eight softmax warps (one arrival per warp)
    static constexpr int kItemReaders = kLoadLanes - 1 + 2 + 8;
};

// TMEM column map: S_t at 128*t (P_t aliases the first 64 columns of S_t), O_t at 256 + 128*t.
__device__ __forceinline__ uint32_t tmem_s_col(int t) { return 128u * t; }
__device__ __forceinline__ uint32_t tmem_o_col(int t) { return 256u + 128u * t; }

// One work item: a pair of Q tiles of one (batch, query head), and for the split instantiation
// one range of KV tiles.
struct FwdWork {
    int b, hkv, hq, bh, tile0, split;
    int kv_begin;      // first KV tile of the item
    int last0, last1;  // last KV tile of Q tile 0 / 1 (the diagonal under the causal mask)
    int kv_end;        // one past the last KV tile the item loads
    bool part0, part1;  // Q tile t takes part (its KV range is not empty)
};

// Item order: blocks of kv_block (batch, KV head) pairs whose K/V fit in L2 together; within a
// block, Q-tile pairs heaviest (latest) first, then the KV heads, then the query heads sharing
// each KV head.  Items are claimed in this order, so the CTAs working at any time read K/V of one
// block (which stays in L2), and every block (and so the launch) ends on its lightest causal pairs.
template <bool kSplit, bool kOne>
__device__ __forceinline__ FwdWork decode_work(const AttnParams& p, int item) {
    FwdWork w;
    w.split = 0;
    if constexpr (kSplit) {
        w.split = item % p.n_splits;
        item /= p.n_splits;
    }
    const int per_kv = p.n_pairs * p.group;
    const int blk = item / (p.kv_block * per_kv);
    const int in_blk = item % (p.kv_block * per_kv);
    const int kvs = min(p.kv_block, p.B * p.Hkv - blk * p.kv_block);  // KV heads in this block
    const int bh_kv = blk * p.kv_block + (in_blk % (kvs * p.group)) / p.group;
    const int rem = in_blk % p.group;
    const int pair = p.n_pairs - 1 - in_blk / (kvs * p.group);
    w.b = bh_kv / p.Hkv;
    w.hkv = bh_kv % p.Hkv;
    w.hq = w.hkv * p.group + rem;
    w.bh = w.b * p.Hq + w.hq;
    w.tile0 = kOne ? pair : 2 * pair;
    // Each Q tile t uses [kv_begin, last_t]; under the causal mask its last tile is its diagonal
    // (BM == BN, so it has the Q tile's index).  A Q tile takes part if that range is not empty
    // (always, unless a later split starts past it).
    w.kv_begin = kSplit ? w.split * p.split_tiles : 0;
    const int kv_limit = kSplit ? min(w.kv_begin + p.split_tiles, p.n_tiles) : p.n_tiles;
    w.last0 = min(kv_limit - 1, p.causal ? w.tile0 : p.n_tiles - 1);
    w.last1 = min(kv_limit - 1, p.causal ? w.tile0 + 1 : p.n_tiles - 1);
    w.part0 = w.last0 >= w.kv_begin;
    w.part1 = !kOne && w.tile0 + 1 < p.n_tiles && w.last1 >= w.kv_begin;
    w.kv_end = (w.part1 ? w.last1 : w.last0) + 1;
    return w;
}

// Index invariants of a decoded work item (checked in debug builds).
__device__ __forceinline__ bool work_in_range(const AttnParams& p, const FwdWork& w) {
    return w.b >= 0 && w.b < p.B && w.hq >= 0 && w.hq < p.Hq && w.hkv >= 0 && w.hkv < p.Hkv &&
           w.hkv == w.hq / p.group && w.tile0 >= 0 && w.tile0 < p.n_tiles && w.kv_begin >= 0 &&
           w.kv_end <= p.n_tiles && w.split >= 0 && w.split < p.n_splits;
}

// Up to this many splits of a work item run as one thread-block cluster and merge through
// distributed shared memory (cluster dimensions up to 8 are portable; with 4 a merging thread
// keeps two rows' loads from every split in registers at once).
constexpr int kMaxClusterSplits = 4;

// Split partials staged for the cluster merge, in the CTA's own shared memory once its MMAs are
// done: O_s of Q tile t (fp32, normalised by its own l) over the K/V ring at t * 128 * D * 4 bytes,
// row r at r * D * 4, its 16-byte chunk c at (c ^ (r & (D/4 - 1))) * 16 (so that a warp's 32 rows
// written at once spread over all banks); LSE_s of the 2 x 128 rows (natural log; -inf where the
// tile took no part in this split) in the first P panel, and the merge's weights of the rows
// this CTA combines after them.
template <int D>
__device__ __forceinline__ uint32_t cluster_o_stage(int t, int r, int c) {
    return static_cast<uint32_t>(SmemLayout<D>::kKV + t * kBM * D * 4 + r * D * 4 +
                                 ((c ^ (r & (D / 4 - 1))) << 4));
}
template <int D>
__device__ __forceinline__ uint32_t cluster_lse_stage(int t, int r) {
    return static_cast<uint32_t>(SmemLayout<D>::kP1 + (t * kBM + r) * 4);
}
// weight of split s for the i-th row this CTA merges (i < 128: both tiles' rows, at most 2 x 64)
template <int D>
__device__ __forceinline__ uint32_t cluster_weight(int i, int s) {
    return static_cast<uint32_t>(SmemLayout<D>::kP1 + 2 * kBM * 4 + (i * kMaxClusterSplits + s) * 4);
}
static_assert(kStages >= 4, "O staging (2 x 128 x D fp32) fits in the K/V ring (kStages x 128 x D bf16)");
static_assert(2 * kBM * 4 + kBM * kMaxClusterSplits * 4 <= 2 * kBM * 64 * 2,
              "LSE staging and weights fit in the P panels");

// The softmax warps (warp w: Q tile w / 4, TMEM lane quarter w % 4) stage their rows.
template <int D>
__device__ __forceinline__ void cluster_stage_split(uint32_t sbase, uint32_t tmem, int warp,
                                                    int lane, float m, float l, bool have) {
    const int t = warp >> 2, quarter = warp & 3, row = quarter * 32 + lane;
    const uint32_t o_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + tmem_o_col(t);
    if (have) {  // uniform over the warp (the tile's four warps agree on the item)
        tc_fence_after();
        const float inv_l = 1.0f / l;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(o_addr + cc * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
                st_shared_v4(sbase + cluster_o_stage<D>(t, row, cc * 8 + i),
                             __float_as_uint(__uint_as_float(r[4 * i]) * inv_l),
                             __float_as_uint(__uint_as_float(r[4 * i + 1]) * inv_l),
                             __float_as_uint(__uint_as_float(r[4 * i + 2]) * inv_l),
                             __float_as_uint(__uint_as_float(r[4 * i + 3]) * inv_l));
        }
    }
    const float lse = have ? (m + __log2f(l)) * kLn2 : -INFINITY;
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + cluster_lse_stage<D>(t, row)), "f"(lse)
                 : "memory");
}

// The merge of section 2.4's split-T inside the cluster: CTA s combines rows s*R .. s*R + R - 1
// (R = 128 / splits, rounded up) of each Q tile of the work item, reading every CTA's staging
// through distributed shared memory: LSE = M + ln sum_s exp(LSE_s - M), O = sum_s exp(LSE_s -
// LSE) O_s, over the splits that hold visible keys (LSE_s > -inf).  First one thread per row
// reads the row's LSE_s, writes LSE and keeps the weights exp(LSE_s - LSE) in shared memory;
// then D/4 lanes per row read the O_s rows (16 bytes a lane from every split at once) and store
// O.  Every thread of the CTA calls this (it holds a CTA barrier).  If a CTA of the cluster gave
// up (its abort flag), nothing is merged; the expiry is in the status word.
template <int D, bool kOne>
__device__ __forceinline__ void cluster_merge_splits(const AttnParams& p, uint32_t sbase) {
    using L = SmemLayout<D>;
    const int n = p.n_splits;
    uint32_t peer[kMaxClusterSplits];
    bool aborted = false;
#pragma unroll
    for (int s = 0; s < kMaxClusterSplits; ++s) {
        peer[s] = s < n ? dsmem_addr(sbase, static_cast<uint32_t>(s)) : 0u;
        if (s < n) aborted |= ld_dsmem_u32(peer[s] + L::kAbort) != 0u;
    }
    if (aborted) return;  // uniform over the cluster: every thread read the same flags
    const FwdWork w = decode_work<true, kOne>(p, static_cast<int>(blockIdx.x));
    constexpr int kTiles = kOne ? 1 : 2;
    const int per = (kBM + n - 1) / n;
    const int r0 = static_cast<int>(cluster_ctarank()) * per;
    const int rows = min(per, kBM - r0);  // rows of each tile this CTA merges
    auto q_of = [&](int i) { return (w.tile0 + i / rows) * kBM + r0 + i % rows; };
    // Only the softmax warps (threads 0..255) work here: they run with the larger register budget.
    constexpr int kWorkers = 256;
    const int tid = static_cast<int>(threadIdx.x);
    // 1. weights and LSE, one thread per row
    if (tid < kWorkers) {
        for (int i = tid; i < kTiles * rows; i += kWorkers) {
            const int q = q_of(i);
            if (q >= p.N) continue;
            const int t = i / rows, r = r0 + i % rows;
            float ls[kMaxClusterSplits];
            float mx = -INFINITY;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) {
                ls[s] = s < n ? __uint_as_float(ld_dsmem_u32(peer[s] + cluster_lse_stage<D>(t, r)))
                              : -INFINITY;
                mx = fmaxf(mx, ls[s]);
            }
            float sum = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) {
                ls[s] = ls[s] > -INFINITY ? expf(ls[s] - mx) : 0.f;
                sum += ls[s];
            }
            const float inv = 1.0f / sum;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s)
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + cluster_weight<D>(i, s)),
                             "f"(ls[s] * inv)
                             : "memory");
            if (ATTN_DCHECK(static_cast<size_t>(w.bh) * p.N + q <
                            static_cast<size_t>(p.B) * p.Hq * p.N))
                p.lse[static_cast<size_t>(w.bh) * p.N + q] = mx + logf(sum);
        }
    }
    __syncthreads();
    // 2. O: D/4 lanes per row, two rows per pass so that 2 x splits loads are in flight a lane
    if (tid < kWorkers) {
        constexpr int kLanes = D / 4, kStep = kWorkers / kLanes;
        const int c = tid % kLanes, col = 4 * c;
        __nv_bfloat16* obase = p.out + w.b * p.o_sb + w.hq * p.o_sh;
        for (int i0 = tid / kLanes; i0 < kTiles * rows; i0 += 2 * kStep) {
            uint32_t v[2][kMaxClusterSplits][4];
            bool live[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * kStep;
                live[u] = i < kTiles * rows && q_of(i) < p.N;
                const int t = i / rows, r = r0 + i % rows;
#pragma unroll
                for (int s = 0; s < kMaxClusterSplits; ++s)
                    if (live[u] && s < n)
                        ld_dsmem_v4(peer[s] + cluster_o_stage<D>(t, r, c), v[u][s][0], v[u][s][1],
                                    v[u][s][2], v[u][s][3]);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (!live[u]) continue;
                const int i = i0 + u * kStep;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < kMaxClusterSplits; ++s) {
                    if (s < n) {
                        float wgt;
                        asm volatile("ld.shared.f32 %0, [%1];"
                                     : "=f"(wgt)
                                     : "r"(sbase + cluster_weight<D>(i, s))
                                     : "memory");
                        if (wgt != 0.f)  // a split without visible keys staged no O
#pragma unroll
                            for (int x = 0; x < 4; ++x)
                                acc[x] += wgt * __uint_as_float(v[u][s][x]);
                    }
                }
                if (col < p.d_out && ATTN_DCHECK(work_in_range(p, w))) {
                    uint2 o;
                    o.x = pack_bf16x2(acc[0], acc[1]);
                    o.y = pack_bf16x2(acc[2], acc[3]);
                    *reinterpret_cast<uint2*>(obase + static_cast<long long>(q_of(i)) * p.o_sn +
                                              col) = o;
                }
            }
        }
    }
}

// kSplit = false: the whole KV range, bf16 O and LSE written to the outputs.
// kSplit = true:  the KV range of one split (split index innermost in the item number); the fp32
//                 O of that range (normalised by its own denominator) and its LSE go to the
//                 workspace, and attn_splitkv_merge_kernel combines the splits.
// kOne = true:    one Q tile per work item (the second tile's issuer and softmax group idle),
//                 for launches whose pairs would leave most SMs idle.
// kCluster = true (with kSplit): the splits of one work item are one thread-block cluster, one
//                 CTA per split (launched with one work unit per CTA and no claim counter); at
//                 the end every CTA stages its O_s = acc / l and LSE_s in its own shared memory
//                 and the cluster combines them through distributed shared memory
//                 (cluster_merge_splits): no partial reaches global memory, no merge kernel runs.
template <int D, bool kSplit, bool kOne = false, bool kCluster = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const AttnParams p,
                    unsigned int* status_word) {
    using L = SmemLayout<D>;
    static_assert(D == 64 || D == 128, "head dim");
    constexpr int kPanels = D / 64;
    constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0);   // Q (K-major) x K (K-major)
    constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, 1);    // P (TMEM) x V (MN-major)

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
    // the split instantiation's merge kernel may be scheduled as soon as every CTA has started
    // (it waits for this kernel's partials itself)
    if constexpr (kSplit) griddep_launch_dependents();

    // ---- setup (once per CTA) ------------------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(L::kBarQFull + t), kPanels);  // one arrive (+ tx) per Q panel
            mbar_init(bar(L::kBarQFree + t), 1);
            mbar_init(bar(L::kBarSFull + t), 1);
            mbar_init(bar(L::kBarPReady + 2 * t + 0), 128);
            mbar_init(bar(L::kBarPReady + 2 * t + 1), 128);
            mbar_init(bar(L::kBarPVDone + t), 1);
            mbar_init(bar(L::kBarODone + t), 1);
            mbar_init(bar(L::kBarTurn + 2 * t + 0), 128);
            mbar_init(bar(L::kBarTurn + 2 * t + 1), 128);
            mbar_init(bar(L::kBarItemFull + t), 1);
            mbar_init(bar(L::kBarItemEmpty + t), L::kItemReaders);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(L::kBarKvFull + s), kPanels);  // one arrive (+ tx) per panel
            mbar_init(bar(L::kBarKvEmpty + s), 2);       // one release per issuer
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp0) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Item ring reader (every role but the claiming lane): the item number of the k-th item, or
    // -1 at the end (or after an abort).  Warps pass warp = true (one arrival per warp).
    auto read_item = [&](int k, bool whole_warp) -> int {
        const int slot = k & 1;
        const uint32_t ph = static_cast<uint32_t>(k >> 1) & 1u;
        bool ok;
        if (whole_warp)
            ok = mbar_wait_warp(bar(L::kBarItemFull + slot), ph, abort_flag, status_word);
        else
            ok = mbar_wait_bounded(bar(L::kBarItemFull + slot), ph, abort_flag, status_word);
        if (!ok) return -1;
        int item = item_ring[slot];
        if (whole_warp) {
            // redux.sync leaves its result in a uniform register, so everything a warp derives
            // from the item (ring indices, smem descriptors, barrier phases) stays in the
            // uniform datapath, as blockIdx-derived values would.
            item = __reduce_min_sync(0xffffffffu, item);
            mbar_arrive_warp(bar(L::kBarItemEmpty + slot));
        } else {
            mbar_arrive(bar(L::kBarItemEmpty + slot));
        }
        return item;
    };

    // kCluster: the softmax threads keep their tile's final m and l (one work item per CTA)
    float cl_m = -INFINITY, cl_l = 0.f;
    bool cl_have = false;  // this thread's Q tile took part in this CTA's split

    // Each role's code follows its warpgroup's register budget (setmaxnreg at the top of the
    // warpgroup's branch), so the compiler allocates the softmax code with kSoftmaxRegs.
    if (warp >= kMmaWarp0) {
    setmaxnreg_dec<kOtherRegs>();
    if (warp == kLoadWarp) {
        // ====================== TMA producer: one lane per 64-column panel stream ===============
        // One thread's bulk tensor copies are processed one after another (measured: ~29 bytes
        // per cycle per SM from one issuing thread, ~50 from two, ~85 from four), so lane h
        // streams panel h of every K tile and lane kPanels + h panel h of every V tile; each
        // lane arrives with its own panel's bytes.  (The Q tiles are loaded by their MMA
        // issuers.)  Lane 0 also claims the items.
        if (lane < L::kLoadLanes) {
            ArmedPhases kv_armed;        // this lane's loads, drained after an abort
            int ring = 0;                // K/V ring entries of the earlier items
            bool claims_done = false;    // lane 0: this CTA's claim past the end was made
            int claim_round = 0;         // lane 0: items this CTA has taken
            // One claim: the item number, or -1 past the end (the launch's last claim also
            // zeroes the counter).
            auto claim = [&]() -> int {
                return claim_next_item(p.sched, p.items, claim_round, claims_done, blockIdx.x,
                                       gridDim.x);
            };
            for (int k = 0;; ++k) {
                int item;
                if (lane == 0) {
                    const int slot = k & 1;
                    if (!mbar_wait_bounded(bar(L::kBarItemEmpty + slot),
                                           (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u, abort_flag,
                                           status_word))
                        break;
                    item = k == 0 ? static_cast<int>(blockIdx.x) : claim();
                    item_ring[slot] = item;
                    mbar_arrive(bar(L::kBarItemFull + slot));
                } else {
                    item = read_item(k, false);
                }
                if (item < 0) break;
                const FwdWork w = decode_work<kSplit, kOne>(p, item);
                if (lane == 0) (void)ATTN_DCHECK(item < p.items && work_in_range(p, w));
                if (!(w.part0 || w.part1)) continue;
                {  // K (kv = 0) or V (kv = 1), panel h
                    const int kv = lane / kPanels, h = lane % kPanels;
                    const CUtensorMap* map = kv ? &tmap_v : &tmap_k;
                    bool ok = true;
                    for (int j = w.kv_begin; j < w.kv_end; ++j) {
                        const int idx = ring + 2 * (j - w.kv_begin) + kv;
                        const int slot = idx % kStages;
                        const uint32_t ph = (idx / kStages) & 1;
                        ok = mbar_wait_bounded(bar(L::kBarKvEmpty + slot), ph ^ 1u, abort_flag,
                                               status_word);
                        if (!ok) break;
                        if (idx == p.stall_item) continue;  // test hook: never deliver this entry
                        mbar_arrive_expect_tx(bar(L::kBarKvFull + slot), L::kPanelBytes);
                        kv_armed.arm(slot, ph);
                        tma_load_4d(sbase + L::kKV + slot * L::kTileBytes + h * L::kPanelBytes,
                                    map, bar(L::kBarKvFull + slot), h * 64, j * kBN, w.hkv, w.b);
                    }
                    if (!ok) break;
                }
                ring += 2 * (w.kv_end - w.kv_begin);
            }
            // After an abort, still make this CTA's claims up to the one past the end, so the
            // launch's claim count (and the counter's reset) stays exact.
            if (lane == 0)
                while (!claims_done) (void)claim();
            if (*abort_flag) kv_armed.drain(bar(L::kBarKvFull), globaltimer_ns() + kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
        // ============ MMA issuers: warp 8 for Q tile 0, warp 9 for Q tile 1 ======================
        // One issuing thread starts a tcgen05.mma only every ~95 cycles (warp-uniform loop,
        // elected lane), more than the 64 tensor cycles of an M=128, N=128, K=16 MMA; two issuers
        // with independent accumulators keep the tensor core fed, also while the other tile's
        // issuer waits for its softmax.  Every K/V ring entry gets one release per issuer: after
        // its MMAs, or (an entry this tile does not use) as soon as it has landed, so every slot
        // phase gets exactly two releases and never completes early.
        const int t = warp - kMmaWarp0;
        const uint32_t s_tmem = tmem + tmem_s_col(t);
        const uint32_t o_tmem = tmem + tmem_o_col(t);
        const uint32_t qa = sbase + L::kQ + t * L::kTileBytes;
        auto kv_slot = [](int idx) { return idx % kStages; };
        auto kv_phase = [](int idx) { return static_cast<uint32_t>((idx / kStages) & 1); };
        auto wait_full = [=](int idx) {
            return mbar_wait_warp(bar(L::kBarKvFull + kv_slot(idx)), kv_phase(idx), abort_flag,
                                  status_word);
        };
        // S_t = Q_t . K^T  (8 MMAs of K = 16 at D = 128)
        auto s_mma = [=](int kslot) {
            const uint32_t ka = sbase + L::kKV + kslot * L::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
                mma_bf16_ss_warp(s_tmem, smem_desc_sw128(qa + off, 16, 1024),
                                 smem_desc_sw128(ka + off, 16, 1024), kIdescS, kk > 0);
            }
        };
        // O_t += P_t . V in two halves.  Keys 0-63 of P_t arrive in TMEM over S_t (TS form);
        // keys 64-127 arrive in a swizzled smem panel (SS form).  Because the second half does
        // not live in TMEM, S_t(j+1) can be issued right after the first half's MMAs and computes
        // while the softmax still works on the second half.
        const uint32_t p1a = sbase + L::kP1 + t * L::kP1Bytes;
        auto pv_first = [=](int vslot, bool accumulate_first) {
            const uint32_t va = sbase + L::kKV + vslot * L::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ts_warp(o_tmem, s_tmem + kk * 8,
                                 smem_desc_sw128(va + kk * 2048, L::kPanelBytes, 1024), kIdescPV,
                                 (accumulate_first || kk > 0) ? 1u : 0u);
        };
        auto pv_second = [=](int vslot) {
            const uint32_t va = sbase + L::kKV + vslot * L::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss_warp(o_tmem, smem_desc_sw128(p1a + kk * 32, 16, 1024),
                                 smem_desc_sw128(va + (4 + kk) * 2048, L::kPanelBytes, 1024),
                                 kIdescPV, 1u);
        };

        ArmedPhases q_armed;   // this lane's Q loads, drained after an abort
        int ring = 0;          // K/V ring entries of the earlier items
        uint32_t steps = 0;    // KV steps this tile ran in earlier items (P-ready phases)
        uint32_t q_items = 0;  // items this tile took part in (Q-full phases)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = read_item(k, true);
            if (item < 0) break;
            const FwdWork w = decode_work<kSplit, kOne>(p, item);
            if (!(w.part0 || w.part1)) continue;
            const bool part = t == 0 ? w.part0 : w.part1;
            const int last = part ? (t == 0 ? w.last0 : w.last1) : w.kv_begin - 1;
            if (part) {
                // this tile's Q for the item: lane h loads panel h once the previous item's last
                // S MMA (which this warp issued) has read the buffer
                if (lane < kPanels) {
                    bool qok = q_items == 0 ||
                               mbar_wait_bounded(bar(L::kBarQFree + t), (q_items - 1) & 1u,
                                                 abort_flag, status_word);
                    if (qok) {
                        mbar_arrive_expect_tx(bar(L::kBarQFull + t), L::kPanelBytes);
                        q_armed.arm(t, q_items);
                        tma_load_4d(qa + lane * L::kPanelBytes, &tmap_q, bar(L::kBarQFull + t),
                                    lane * 64, (w.tile0 + t) * kBM, w.hq, w.b);
                    }
                }
                __syncwarp();
                ok = mbar_wait_warp(bar(L::kBarQFull + t), q_items & 1u, abort_flag, status_word);
                if (ok) ok = wait_full(ring);
                if (ok) {
                    tc_fence_after();
                    s_mma(kv_slot(ring));
                    mma_commit_warp(bar(L::kBarSFull + t));
                    mma_commit_warp(bar(L::kBarKvEmpty + kv_slot(ring)));
                    if (last == w.kv_begin) mma_commit_warp(bar(L::kBarQFree + t));
                }
                for (int j = w.kv_begin; ok && j <= last; ++j) {
                    const int vidx = ring + 2 * (j - w.kv_begin) + 1;  // V_j
                    const int kidx = vidx + 1;                         // K_{j+1}
                    ok = wait_full(vidx);
                    // (the issuers' and the softmax groups' long waits suspend instead of polling,
                    // leaving the issue slots of the SM sub-partition to the softmax warps that
                    // share it: measured 2-4 % faster than polling at N = 8192-16384)
                    if (ok) ok = mbar_wait_warp<true>(bar(L::kBarPReady + 2 * t + 0), steps & 1u,
                                                      abort_flag, status_word);
                    if (!ok) break;
                    tc_fence_after();
                    pv_first(kv_slot(vidx), j > w.kv_begin);
                    if (j + 1 <= last) {  // S_t(j+1) overwrites the first half of P_t(j)
                        ok = wait_full(kidx);
                        if (!ok) break;
                        tc_fence_after();
                        s_mma(kv_slot(kidx));
                        mma_commit_warp(bar(L::kBarSFull + t));
                        mma_commit_warp(bar(L::kBarKvEmpty + kv_slot(kidx)));
                        if (j + 1 == last) mma_commit_warp(bar(L::kBarQFree + t));
                    }
                    ok = mbar_wait_warp<true>(bar(L::kBarPReady + 2 * t + 1), steps & 1u,
                                              abort_flag, status_word);
                    if (!ok) break;
                    tc_fence_after();
                    pv_second(kv_slot(vidx));
                    ++steps;
                    mma_commit_warp(bar(L::kBarPVDone + t));
                    if (j == last) mma_commit_warp(bar(L::kBarODone + t));
                    mma_commit_warp(bar(L::kBarKvEmpty + kv_slot(vidx)));
                }
                ++q_items;
            }
            // K/V tiles of this item that this Q tile does not need (under the causal mask, the
            // last one for Q tile 0; all of them if the tile takes no part)
            for (int j = last + 1; ok && j < w.kv_end; ++j) {
                for (int kv = 0; ok && kv < 2; ++kv) {
                    const int idx = ring + 2 * (j - w.kv_begin) + kv;
                    ok = wait_full(idx);
                    if (ok) mbar_arrive_warp(bar(L::kBarKvEmpty + kv_slot(idx)));
                }
            }
            ring += 2 * (w.kv_end - w.kv_begin);
        }
        if (*abort_flag) q_armed.drain(bar(L::kBarQFull), globaltimer_ns() + kDrainLimitNs);
        __syncwarp();
    }
    } else {
        setmaxnreg_inc<kSoftmaxRegs>();
        // =========================== softmax + epilogue (warps 0-7) ============================
        const int t = warp >> 2;          // which Q tile
        const int quarter = warp & 3;     // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;  // row within the Q tile
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + tmem_s_col(t);
        const uint32_t o_addr = tmem + lane_base + tmem_o_col(t);
        const uint32_t p1 = sbase + L::kP1 + t * L::kP1Bytes;  // P keys 64..127, O staging
        const float c = p.scale_log2;
        // Barrier phases, one bit each: S-full / P.V-done step parity, O-done parity.
        constexpr uint32_t kPhStep = 1u, kPhODone = 4u;
        uint32_t ph = 0;
        uint32_t tok = 0;  // this group's exp2 phases that take part in the ping-pong so far
        bool ok = true;
        // The four warps of a group leave the item loop together (they share named barriers):
        // they agree on every item they read and on the outcome of every item's waits.
        for (int k = 0;; ++k) {
            const int item = read_item(k, true);
            if (!named_barrier_and(1 + t, 128, item >= 0)) break;
            int n, lim, tok_until;
            bool mask_last;
            {
                const FwdWork w = decode_work<kSplit, kOne>(p, item);
                if (!(t == 0 ? w.part0 : w.part1)) continue;
                const bool pingpong = w.part0 && w.part1;
                const int q_tile = w.tile0 + t;
                const int last = t == 0 ? w.last0 : w.last1;
                n = last - w.kv_begin + 1;  // KV steps of this tile
                // Only the last step can need a mask: the causal diagonal tile, or the ragged
                // last key tile (non-causal).  lim = first masked key of this row.
                mask_last = p.causal ? last == q_tile
                                     : (last == p.n_tiles - 1 && (p.N % kBN) != 0);
                lim = p.causal ? row + 1 : p.N - last * kBN;
                // Ping-pong through turn tokens: group 1's exp2 phase number x waits for group
                // 0's number x, group 0's number x for group 1's number x-2, so the phases
                // alternate in the steady state while group 0 may run up to two ahead, e.g. into
                // the next item while group 1 finishes its item's last (diagonal) step and
                // epilogue.  Tokens go to two barriers per group by the parity of x, so neither
                // barrier ever holds two pending phases.  Steps i <= tok_until take part: both
                // groups' steps up to tile 0's last one, in items where both tiles take part.
                tok_until = !pingpong ? -1 : (t == 0 ? n - 1 : w.last0 - w.kv_begin);
            }
            float m = -INFINITY;  // running max of c*s (log2 units)
            float l = 0.f;        // running denominator
            for (int i = 0; i < n; ++i) {
                ok = mbar_wait_warp<true>(bar(L::kBarSFull + t), ph & kPhStep, abort_flag,
                                          status_word);
                if (!ok) break;
                tc_fence_after();
                // Masks are applied in TMEM before the row is loaded, so the common unmasked step
                // carries no mask code.
                if (mask_last && i == n - 1) {
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
                // row maximum: 8 independent chains of 3-input max
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
                const float alpha = ex2_approx(m - m_new);  // 1 if unchanged, 0 on the first tile
                const bool rescale = i > 0 && __any_sync(0xffffffffu, m_new != m);
                m = m_new;
                const float neg_m = -m;
                if (i <= tok_until && (t == 1 || tok >= 2)) {
                    const uint32_t x = t == 0 ? tok - 2 : tok;  // the other group's token
                    ok = mbar_wait_warp<true>(bar(L::kBarTurn + 2 * t + (x & 1)), (x >> 1) & 1u,
                                              abort_flag, status_word);
                    if (!ok) break;
                }
                // p = exp2(c*s - m).  Keys 0-63 go to TMEM (over S) and are published first; keys
                // 64-127 go to this tile's smem panel, which the previous step's second-half P.V
                // must have finished reading (pv_done).  That P.V also had to land before the
                // O correction (O_row *= alpha, rare thanks to the lazy maximum).
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                auto exp_half = [&](int h, uint32_t (&pk)[32]) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int col = h * 64 + 2 * i;
                        float x0, x1;
                        ffma2(x0, x1, s[col], s[col + 1], c, c, neg_m, neg_m);
                        const float p0 = ex2_approx(x0);
                        const float p1v = ex2_approx(x1);
                        const int a = (i & 1) * 2;
                        fadd2(acc[a], acc[a + 1], acc[a], acc[a + 1], p0, p1v);
                        pk[i] = pack_bf16x2(p0, p1v);
                    }
                };
                const bool prev_pv = i > 0;  // a previous step's P.V is in flight
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
                    mbar_arrive(bar(L::kBarPReady + 2 * t + 0));
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
                    fence_proxy_async_smem();  // generic-proxy stores -> the MMA's async reads
                    mbar_arrive(bar(L::kBarPReady + 2 * t + 1));
                }
                l = l * alpha + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
                if (i <= tok_until) {  // token number `tok` to the other group
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
            // The epilogue's coordinates, decoded again from an opaque copy of the item number so
            // that they are not kept in registers through the step loop.
            const FwdWork we = decode_work<kSplit, kOne>(p, opaque_int(item));
            const int row_g = (we.tile0 + t) * kBM + row;
            const float inv_l = 1.0f / l;
            if constexpr (kCluster) {
                // ---- staged in the teardown, once every MMA of the CTA has completed ----------
                cl_m = m;
                cl_l = l;
                cl_have = true;
                (void)row_g;
                (void)inv_l;
            } else if constexpr (kSplit) {
                // ---- split epilogue: O_s = acc / l (fp32) and LSE_s to the workspace ----------
                const size_t prow =
                    (static_cast<size_t>(we.split) * p.B * p.Hq + we.bh) * p.N + row_g;
                float* dst = p.ws_o + prow * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t r[32];
                    tmem_ld32(o_addr + cc * 32, r);  // warp-collective: every lane loads
                    tmem_wait_ld();
                    if (row_g < p.N && ATTN_DCHECK(work_in_range(p, we))) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            st_global_v4f(dst + cc * 32 + 4 * i, __uint_as_float(r[4 * i]) * inv_l,
                                          __uint_as_float(r[4 * i + 1]) * inv_l,
                                          __uint_as_float(r[4 * i + 2]) * inv_l,
                                          __uint_as_float(r[4 * i + 3]) * inv_l);
                    }
                }
                if (row_g < p.N &&
                    ATTN_DCHECK(prow < static_cast<size_t>(p.n_splits) * p.B * p.Hq * p.N))
                    p.ws_lse[prow] = (m + __log2f(l)) * kLn2;
            } else {
                // ---- epilogue: O = acc / l -> bf16, one 64-column panel at a time through this
                // tile's P panel (free: O-done follows the last P.V), out with coalesced 16-byte
                // stores (each warp instruction writes four 128-byte row segments); LSE.
                const int q_row0 = (we.tile0 + t) * kBM;
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
                            const int chunk = cc * 4 + c16;  // 16-byte chunk within the 128B row
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
                    named_barrier_sync(1 + t, 128);  // the panel may be written again
                }
                if (row_g < p.N &&
                    ATTN_DCHECK(static_cast<size_t>(we.bh) * p.N + row_g <
                                static_cast<size_t>(p.B) * p.Hq * p.N))
                    p.lse[static_cast<size_t>(we.bh) * p.N + row_g] = (m + __log2f(l)) * kLn2;
            }
        }
        __syncwarp();
    }

    // ---- teardown ------------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if constexpr (kCluster) {
        // (after an abort the K/V ring may still be a TMA destination: nothing is staged)
        if (warp < 8) cluster_stage_split<D>(sbase, tmem, warp, lane, cl_m, cl_l,
                                             cl_have && *abort_flag == 0);
        cluster_sync_all();  // every CTA's partials are staged (and visible to the cluster)
        cluster_merge_splits<D, kOne>(p, sbase);
        cluster_sync_all();  // no CTA leaves while another may still read its staging
    }
    if (warp == kMmaWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Split-KV merge ("Attention Kernel 实现与正确性验证" section 2.4, the split-T pattern: partial
// results per split of the key axis, then a safe-softmax combination), fused into one kernel.
// For query row i of head bh, the splits s that hold keys visible to it (all those starting at or
// before its last visible key tile) are combined as
//   LSE = M + ln sum_s exp(LSE_s - M),  M = max_s LSE_s,   O = sum_s exp(LSE_s - LSE) * O_s.
// One warp per row; lane k owns D/32 consecutive columns (coalesced 16-byte loads per split).
// D is the padded width of the partials; only the first d_out columns of each row go to `out`:
// rows of d_out elements one after another, or (kStrided) rows addressed through element strides
// (batch o_sb, head o_sh, row o_sn; each a multiple of 8).  The contiguous instantiation keeps
// its index arithmetic (and registers, so the blocks in flight of this memory-streaming kernel)
// to the row number alone.
template <int D, bool kStrided>
__global__ void __launch_bounds__(256)
    attn_splitkv_merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                              __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int BH,
                              int Hq, int N, int d_out, long long o_sb, long long o_sh,
                              long long o_sn, int n_tiles, int causal, int n_splits,
                              int split_tiles) {
    constexpr int kCols = D / 32;
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    griddep_wait();  // launched as the split kernel's dependant: its partials are complete
    if (row >= static_cast<long long>(BH) * N) return;
    const int i = static_cast<int>(row % N);
    const int last_kv = causal ? i / kBN : n_tiles - 1;
    const int n_valid = min(n_splits, last_kv / split_tiles + 1);
    (void)ATTN_DCHECK(n_valid >= 1 && n_valid <= n_splits && last_kv < n_tiles);
    const size_t plane = static_cast<size_t>(BH) * N;  // rows per split
    float mx = -INFINITY;
    for (int s = 0; s < n_valid; ++s) mx = fmaxf(mx, ws_lse[s * plane + row]);
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
    float wsum = 0.f;
    for (int s = 0; s < n_valid; ++s) {
        const float w = expf(ws_lse[s * plane + row] - mx);
        wsum += w;
        const float* src = ws_o + (s * plane + row) * D + lane * kCols;
        if constexpr (kCols == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            acc[0] += w * v.x; acc[1] += w * v.y;
        }
    }
    const float inv = 1.0f / wsum;
    const int c0 = lane * kCols;
    __nv_bfloat16* o;
    if constexpr (kStrided) {
        const int bh = static_cast<int>(row / N);  // BH < 2^31
        const int b = bh / Hq;
        o = out + b * o_sb + (bh - b * Hq) * o_sh + i * o_sn + c0;
    } else {
        (void)Hq;
        (void)o_sb;
        (void)o_sh;
        (void)o_sn;
        o = out + row * d_out + c0;
    }
    if (d_out == D) {  // full width: one 8-byte (D=128) or 4-byte (D=64) store per lane
        if constexpr (kCols == 4) {
            uint2 packed;
            packed.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            packed.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2*>(o) = packed;
        } else {
            *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
    } else {  // padded head dimension: the columns at and beyond d_out are not part of O
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            if (c0 + c < d_out) o[c] = __float2bfloat16_rn(acc[c] * inv);
    }
    if (lane == 0) lse[row] = mx + logf(wsum);
}

}  // namespace gb300attn
