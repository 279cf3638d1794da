// attn_api.cu - C ABI of the GB300 exact-attention forward (validation, TMA descriptors, launch).
//
// Interface follows the problem statement of the pages: inputs Q [B,Hq,N,D], K/V [B,Hkv,N,D]
// contiguous bf16 ("Triton-CUDA Attention", skillmd.com: (B, H, L, D) layout, contiguous inputs,
// GQA grid over the query heads), a causal flag ("Flash Attention 与 Kernel 优化",
// fangpin.github.io: FlashAttention.apply(q, k, v, is_causal)), outputs O and the per-row LSE.
// The split-KV entry point follows the split-T pattern of "Attention Kernel 实现与正确性验证"
// (walkerchi.com), section 2.4: partial results per split of the key axis, then a fused
// safe-softmax merge.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <functional>
#include <mutex>
#include <utility>
#include <vector>

#include "attn.h"
#include "attn_bwd_kernel.cuh"
#include "attn_fwd_d256_kernel.cuh"
#include "attn_fwd_kernel.cuh"
#include "attn_fwd_pair_kernel.cuh"
#include "mla_decode_kernel.cuh"

using namespace gb300attn;

// The device status word (g_attn_status_word, ptx.cuh): kernels OR failure flags into it; the
// host reads and clears it in attn_debug_status.
// Claim counters of the persistent kernels, handed to launches round robin; each launch leaves
// its counter at zero, and a launch that reuses a counter waits for the counter's previous launch.
__device__ unsigned int g_fwd_sched[gb300attn::kSchedSlots] = {};

// attn_fwd's own split-KV partials (when its cost model picks the workspace path): a fixed device
// buffer of kFwdScratchSlots slots, leased to one launch at a time like the claim counters, so
// that attn_fwd never allocates and never shares partials between launches that overlap.
constexpr int kFwdScratchSlots = 2;
constexpr size_t kFwdScratchBytes = size_t(64) << 20;  // per slot
__device__ __align__(256) unsigned char g_fwd_scratch[kFwdScratchSlots * kFwdScratchBytes];

namespace {

constexpr int kMaxSplits = 64;
constexpr int kMergeThreads = 256;

thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return ATTN_ERR_CUDA;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Element strides of a [B, H, N, D] bf16 tensor whose D axis is contiguous.
struct Strides {
    int64_t n, h, b;
};

Strides contiguous_strides(int64_t H, int64_t N, int64_t D) { return {D, N * D, H * N * D}; }

// 4-D view [B, H, N, D] (innermost D); box = 64 (D) x box_rows (rows) x 1 x 1, 128B swizzle.
// Rows >= N of a head are out of bounds: zero-filled on load, dropped on store.
bool make_tile_map(CUtensorMap* map, const void* base, int64_t B, int64_t H, int64_t N, int64_t D,
                   const Strides& st, int box_rows) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n * 2),
                                   static_cast<cuuint64_t>(st.h * 2),
                                   static_cast<cuuint64_t>(st.b * 2)};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
    const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
               box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Encoded tensor maps depend only on (address, sizes, strides); repeated calls on the same buffers
// (the usual case in a serving or training loop) reuse them from a small per-thread cache.
struct MapKey {
    const void* base;
    int64_t B, H, N, D, sn, sh, sb;
    int box_rows;
    bool operator==(const MapKey& o) const {
        return base == o.base && B == o.B && H == o.H && N == o.N && D == o.D && sn == o.sn &&
               sh == o.sh && sb == o.sb && box_rows == o.box_rows;
    }
};
struct MapCache {
    static constexpr int kEntries = 16;
    MapKey key[kEntries];
    CUtensorMap map[kEntries];
    bool valid[kEntries] = {};
    int next = 0;
};
thread_local MapCache t_maps;

bool cached_tile_map(CUtensorMap* map, const void* base, int64_t B, int64_t H, int64_t N,
                     int64_t D, const Strides& st, int box_rows = kBM) {
    const MapKey key{base, B, H, N, D, st.n, st.h, st.b, box_rows};
    for (int i = 0; i < MapCache::kEntries; ++i)
        if (t_maps.valid[i] && t_maps.key[i] == key) {
            *map = t_maps.map[i];
            return true;
        }
    if (!make_tile_map(map, base, B, H, N, D, st, box_rows)) return false;
    const int slot = t_maps.next;
    t_maps.next = (slot + 1) % MapCache::kEntries;
    t_maps.key[slot] = key;
    t_maps.map[slot] = *map;
    t_maps.valid[slot] = true;
    return true;
}

// One claim counter and the completion event of the last launch that used it.
struct SchedSlot {
    std::mutex lock;           // held from the wait on `done` until `done` is recorded again
    cudaEvent_t done = nullptr;
    bool recorded = false;
};

// Per-device one-time set-up: architecture check, SM count, status-word address, smem opt-in.
constexpr int kMaxDevices = 64;
struct DeviceState {
    std::once_flag once;
    int status = ATTN_OK;
    int cuda_error = 0;
    int num_sms = 0;
    unsigned int* status_word = nullptr;
    unsigned int* sched = nullptr;  // g_fwd_sched
    std::atomic<unsigned int> sched_next{0};
    SchedSlot slots[kSchedSlots];
    int pair_clusters = 0;  // CTA pairs of the pair kernel that fit on the device at once
    unsigned char* fwd_scratch = nullptr;  // g_fwd_scratch
    std::atomic<unsigned int> scratch_next{0};
    SchedSlot scratch_slots[kFwdScratchSlots];
    // clusters of n split CTAs (n = 2..kMaxClusterSplits) that fit on the device at once, for
    // D <= 64 ([0]) and D <= 128 ([1])
    int cluster_fit[2][kMaxClusterSplits + 1] = {};
};
DeviceState g_devices[kMaxDevices];

// Opt in to the large shared-memory carve-out, and check that the kernel was built with the
// per-thread register count its setmaxnreg split assumes (a launch with fewer registers would
// leave the softmax warpgroups waiting for registers that do not exist).
template <int D, bool kSplit, bool kOne = false, bool kCluster = false>
cudaError_t opt_in_smem(bool* regs_ok) {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, attn_fwd_kernel<D, kSplit, kOne, kCluster>);
    if (e != cudaSuccess) return e;
    if (a.numRegs != kLaunchRegs) *regs_ok = false;
    return cudaFuncSetAttribute(attn_fwd_kernel<D, kSplit, kOne, kCluster>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SmemLayout<D>::kAlloc);
}

// The pair kernel: shared-memory opt-in, its register count, and how many CTA pairs fit on the
// device at once (a pair needs two SMs of one GPC).
cudaError_t opt_in_pair(bool* regs_ok, int* clusters) {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, attn_fwd_pair_kernel);
    if (e != cudaSuccess) return e;
    if (a.numRegs != kLaunchRegs) *regs_ok = false;
    e = cudaFuncSetAttribute(attn_fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairSmem::kAlloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = PairSmem::kAlloc;
    *clusters = 0;
    // If the device cannot say (or fits no pair), the forward runs on single CTAs only.
    if (cudaOccupancyMaxActiveClusters(clusters, attn_fwd_pair_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        *clusters = 0;
    }
    return cudaSuccess;
}

// How many clusters of n CTAs of the cluster-merge split kernel fit on the device at once (a
// cluster needs n SMs of one GPC).  If the device cannot say, none: the split-KV path then
// always uses its workspace and merge kernel.
template <int D>
void query_cluster_fit(int* fit) {
    for (int n = 2; n <= kMaxClusterSplits; ++n) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned int>(n));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = SmemLayout<D>::kAlloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned int>(n);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        fit[n] = 0;
        if (cudaOccupancyMaxActiveClusters(&fit[n], attn_fwd_kernel<D, true, false, true>, &cfg) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            fit[n] = 0;
        }
    }
}

template <int D>
cudaError_t opt_in_bwd_smem() {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DkdvSmem<D>::kAlloc);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, DqSmem<D>::kAlloc);
    return e;
}

int device_state(int dev, DeviceState** out) {
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    DeviceState& st = g_devices[dev];
    std::call_once(st.once, [&st, dev] {
        int major = 0, minor = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) { st.status = ATTN_ERR_CUDA; st.cuda_error = e; return; }
        if (major != 10 || minor != 3) { st.status = ATTN_ERR_ARCH; return; }
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status_word), g_attn_status_word);
        if (e == cudaSuccess)
            e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.sched), g_fwd_sched);
        if (e == cudaSuccess)
            e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.fwd_scratch), g_fwd_scratch);
        bool regs_ok = true;
        if (e == cudaSuccess) e = opt_in_smem<64, false>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_smem<128, false>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_smem<64, true>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_smem<128, true>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_smem<64, false, true>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_smem<128, false, true>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_smem<64, true, false, true>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_smem<128, true, false, true>(&regs_ok);
        if (e == cudaSuccess) e = opt_in_bwd_smem<64>();
        if (e == cudaSuccess) e = opt_in_bwd_smem<128>();
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     MlaSmem::kAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_fwd_d256_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Fwd256Smem::kAlloc);
        if (e == cudaSuccess) e = opt_in_pair(&regs_ok, &st.pair_clusters);
        if (e == cudaSuccess) {
            query_cluster_fit<64>(st.cluster_fit[0]);
            query_cluster_fit<128>(st.cluster_fit[1]);
        }
        if (e != cudaSuccess) { st.status = ATTN_ERR_CUDA; st.cuda_error = e; return; }
        if (!regs_ok) st.status = ATTN_ERR_ARCH;
    });
    if (st.status == ATTN_ERR_CUDA) t_last_cuda_error = st.cuda_error;
    *out = &st;
    return st.status;
}

int current_device_state(DeviceState** out) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    return device_state(dev, out);
}

int check_memory(const void* ptr, int dev) {
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return ATTN_ERR_MEMORY;
    }
    if (a.type == cudaMemoryTypeManaged) return ATTN_OK;
    if (a.type == cudaMemoryTypeDevice && a.device == dev) return ATTN_OK;
    return ATTN_ERR_MEMORY;
}

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

// Everything about one call that the entry points share.
struct Problem {
    const void *q, *k, *v;
    void* out;
    float* lse;
    int B, Hq, Hkv, N, D, causal;
    float sm_scale;
    int64_t bh, bh_kv, n_tiles, n_pairs, items;
    int64_t q_bytes, kv_bytes, lse_bytes;  // byte spans: [ptr, ptr + bytes) covers each tensor
    bool strided = false;                   // strides below given by the caller
    Strides sq{}, sk{}, sv{}, so{};
};

// Byte span of a strided [B, H, N, D] bf16 tensor (from its first to one past its last element).
int64_t span_bytes(int64_t B, int64_t H, int64_t N, int64_t D, const Strides& st) {
    return ((B - 1) * st.b + (H - 1) * st.h + (N - 1) * st.n + D) * 2;
}

// TMA needs every stride to be a positive multiple of 16 bytes (8 bf16) and below 2^40 bytes.
bool strides_ok(const Strides& st) {
    for (int64_t x : {st.n, st.h, st.b})
        if (x <= 0 || (x % 8) != 0 || x >= (int64_t(1) << 39)) return false;
    return true;
}

// Host-side validation; returns ATTN_OK with *empty set for an empty problem.  Nothing is
// launched or written when this fails.
int validate(Problem& P, bool* empty) {
    *empty = false;
    if (P.B < 0 || P.N < 0 || P.Hq <= 0 || P.Hkv <= 0) return ATTN_ERR_SHAPE;
    if (P.Hq % P.Hkv != 0) return ATTN_ERR_HEADS;
    if (P.D % 8 != 0 || P.D < 8 || P.D > 256) return ATTN_ERR_HEADDIM;
    if (!std::isfinite(P.sm_scale) || !(P.sm_scale > 0.f)) return ATTN_ERR_SCALE;
    if (P.B == 0 || P.N == 0) {  // empty problem: nothing to read or write
        *empty = true;
        return ATTN_OK;
    }
    if (!P.q || !P.k || !P.v || !P.out || !P.lse) return ATTN_ERR_NULL;
    const uintptr_t align_bits =
        reinterpret_cast<uintptr_t>(P.q) | reinterpret_cast<uintptr_t>(P.k) |
        reinterpret_cast<uintptr_t>(P.v) | reinterpret_cast<uintptr_t>(P.out) |
        reinterpret_cast<uintptr_t>(P.lse);
    if (align_bits & 15u) return ATTN_ERR_ALIGN;

    P.bh = static_cast<int64_t>(P.B) * P.Hq;
    P.bh_kv = static_cast<int64_t>(P.B) * P.Hkv;
    P.n_tiles = (static_cast<int64_t>(P.N) + kBM - 1) / kBM;
    P.n_pairs = (P.n_tiles + 1) / 2;
    P.items = (P.D > 128 ? P.n_tiles : P.n_pairs) * P.bh;  // one or two Q tiles per CTA
    if (P.items > 0x7fffffffLL || P.bh > 0x7fffffffLL) return ATTN_ERR_SHAPE;

    if (!P.strided) {
        P.sq = P.so = contiguous_strides(P.Hq, P.N, P.D);
        P.sk = P.sv = contiguous_strides(P.Hkv, P.N, P.D);
    } else if (!strides_ok(P.sq) || !strides_ok(P.sk) || !strides_ok(P.sv) || !strides_ok(P.so)) {
        return ATTN_ERR_STRIDE;
    }
    P.q_bytes = span_bytes(P.B, P.Hq, P.N, P.D, P.sq);
    P.kv_bytes = std::max(span_bytes(P.B, P.Hkv, P.N, P.D, P.sk),
                          span_bytes(P.B, P.Hkv, P.N, P.D, P.sv));
    P.lse_bytes = P.bh * P.N * 4;
    const int64_t o_bytes = span_bytes(P.B, P.Hq, P.N, P.D, P.so);
    if (overlaps(P.out, o_bytes, P.q, P.q_bytes) || overlaps(P.out, o_bytes, P.k, P.kv_bytes) ||
        overlaps(P.out, o_bytes, P.v, P.kv_bytes) || overlaps(P.out, o_bytes, P.lse, P.lse_bytes) ||
        overlaps(P.lse, P.lse_bytes, P.q, P.q_bytes) ||
        overlaps(P.lse, P.lse_bytes, P.k, P.kv_bytes) ||
        overlaps(P.lse, P.lse_bytes, P.v, P.kv_bytes))
        return ATTN_ERR_ALIAS;
    return ATTN_OK;
}

// (batch, KV head) pairs per scheduling block: at most as many as keep their K and V within
// 16 MB (measured: blocks of 50-67 MB of K/V, a die's share of the 129 MB L2, made the CTAs in
// flight read K/V from DRAM about twice), spread evenly over the blocks so that no block is much
// smaller than the others (each block starts on its heaviest causal tiles, so a small last block
// would leave a long tail).
int kv_block_for(const Problem& P) {
    const int64_t d_pad = P.D <= 64 ? 64 : (P.D <= 128 ? 128 : 256);
    const int64_t kv_bytes = std::max<int64_t>(1, 2 * static_cast<int64_t>(P.N) * d_pad * 2);
    const int64_t budget = int64_t(16) << 20;
    const int64_t most = std::max<int64_t>(1, std::min<int64_t>(P.bh_kv, budget / kv_bytes));
    const int64_t blocks = (P.bh_kv + most - 1) / most;
    return static_cast<int>((P.bh_kv + blocks - 1) / blocks);
}

// Device checks and TMA descriptors; fills the kernel parameters common to both entry points.
int prepare(const Problem& P, DeviceState** ds, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv,
            CUtensorMap* mo, AttnParams* prm) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    // A host thread that has not used CUDA yet (e.g. an autograd worker) has no current context,
    // and the driver's tensor-map encoder needs one: bind the current device's primary context.
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const int st = device_state(dev, ds);
    if (st != ATTN_OK) return st;
    for (const void* ptr :
         {P.q, P.k, P.v, static_cast<const void*>(P.out), static_cast<const void*>(P.lse)})
        if (check_memory(ptr, dev) != ATTN_OK) return ATTN_ERR_MEMORY;
    if (!cached_tile_map(mq, P.q, P.B, P.Hq, P.N, P.D, P.sq) ||
        !cached_tile_map(mk, P.k, P.B, P.Hkv, P.N, P.D, P.sk) ||
        !cached_tile_map(mv, P.v, P.B, P.Hkv, P.N, P.D, P.sv) ||
        !cached_tile_map(mo, P.out, P.B, P.Hq, P.N, P.D, P.so))
        return cuda_fail(cudaErrorInvalidValue);
    prm->B = P.B;
    prm->Hq = P.Hq;
    prm->Hkv = P.Hkv;
    prm->N = P.N;
    prm->group = P.Hq / P.Hkv;
    prm->causal = P.causal ? 1 : 0;
    prm->n_tiles = static_cast<int>(P.n_tiles);
    prm->n_pairs = static_cast<int>(P.n_pairs);
    prm->scale_log2 = P.sm_scale * 1.4426950408889634f;  // log2(e)
    prm->kv_block = kv_block_for(P);
    prm->lse = P.lse;
    prm->n_splits = 1;
    prm->split_tiles = prm->n_tiles;
    prm->ws_o = nullptr;
    prm->ws_lse = nullptr;
    prm->stall_item = -1;
    prm->items = static_cast<int>(P.items);
    prm->out = static_cast<__nv_bfloat16*>(P.out);
    prm->o_sb = P.so.b;
    prm->o_sh = P.so.h;
    prm->o_sn = P.so.n;
    prm->d_out = P.D;
    prm->sched = nullptr;  // set by with_claim_counter around the launch
    return ATTN_OK;
}

// Runs launch() on stream `s` holding `slot`: the stream first waits for the event recorded
// after the slot's previous launch, so two launches that hold one slot never run at the same
// time, however many streams or host threads launch; the slot's lock is held until that event is
// recorded again, so two host threads never interleave on one slot.  The event is recorded
// whatever the launch returned: a chain that failed part-way may have enqueued a kernel that uses
// the slot, and the slot's next launch must wait for it.
template <class Launch>
int on_slot(SchedSlot& slot, cudaStream_t s, Launch&& launch) {
    std::lock_guard<std::mutex> guard(slot.lock);
    cudaError_t e = cudaSuccess;
    if (slot.done == nullptr) {
        e = cudaEventCreateWithFlags(&slot.done, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            slot.done = nullptr;
            return cuda_fail(e);
        }
    }
    if (slot.recorded) {
        e = cudaStreamWaitEvent(s, slot.done, 0);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    const int st = launch();
    e = cudaEventRecord(slot.done, s);
    if (e == cudaSuccess) slot.recorded = true;
    if (st != ATTN_OK) return st;
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Runs launch(counter) with a claim counter that no other executing launch holds: one of the
// device's kSchedSlots, taken round robin and held as on_slot describes.  While the stream is
// being captured into a CUDA graph the host cannot order the graph's future replays against
// other launches, so a captured launch gets no counter (nullptr) and the kernel uses its static
// schedule.
template <class Launch>
int with_claim_counter(DeviceState* ds, cudaStream_t s, Launch&& launch) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e);
    if (cap != cudaStreamCaptureStatusNone) return launch(static_cast<unsigned int*>(nullptr));
    const unsigned int idx = ds->sched_next.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots;
    return on_slot(ds->slots[idx], s, [&]() { return launch(ds->sched + idx); });
}

// The persistent two-tile kernel: one CTA per SM (or per item, if fewer), each claiming items
// until all `items` are taken.
// `after` (if given) launches what must follow the kernel directly on the stream (the split
// kernel's merge), inside the claim counter's scope.
int no_follow_up() { return ATTN_OK; }

template <int D, bool kSplit, bool kOne = false, class After = int (*)()>
int launch_fwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
               const AttnParams& p, DeviceState* ds, int64_t items, cudaStream_t stream,
               After&& after = no_follow_up) {
    AttnParams prm = p;
    prm.items = static_cast<int>(items);
    const int64_t grid = std::min<int64_t>(items, std::max(1, ds->num_sms));
    return with_claim_counter(ds, stream, [&](unsigned int* counter) {
        prm.sched = counter;
        attn_fwd_kernel<D, kSplit, kOne><<<static_cast<unsigned int>(grid), kThreads,
                                           SmemLayout<D>::kAlloc, stream>>>(mq, mk, mv, prm,
                                                                            ds->status_word);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
        return after();
    });
}

// The single pass runs on the one-CTA kernel for every shape: measured on GB300 the pair kernel
// is slower wherever it can run (0.62-0.85x at N = 512-32768), its M = 256 MMAs issuing more
// slowly per SM and each step's handshakes crossing between the two SMs; attn_fwd_test_kernel
// still runs it.

// The pair kernel over all quads of the problem: min(quads, pairs that fit) clusters of two CTAs,
// each pair claiming quads until all are taken.  K and V are read in half tiles (64-row boxes).
int launch_pair(const Problem& P, const CUtensorMap& mq, const AttnParams& p_in, DeviceState* ds,
                cudaStream_t stream) {
    CUtensorMap mk64, mv64;
    if (!cached_tile_map(&mk64, P.k, P.B, P.Hkv, P.N, P.D, P.sk, 64) ||
        !cached_tile_map(&mv64, P.v, P.B, P.Hkv, P.N, P.D, P.sv, 64))
        return cuda_fail(cudaErrorInvalidValue);
    AttnParams prm = p_in;
    const int64_t quads = (P.n_tiles + 3) / 4;
    const int64_t items = quads * P.bh;
    if (items > 0x7fffffffLL) return ATTN_ERR_SHAPE;
    prm.n_pairs = static_cast<int>(quads);
    prm.items = static_cast<int>(items);
    const int64_t pairs = std::min<int64_t>(items, ds->pair_clusters);
    return with_claim_counter(ds, stream, [&](unsigned int* counter) {
        prm.sched = counter;
        attn_fwd_pair_kernel<<<static_cast<unsigned int>(2 * pairs), kThreads, PairSmem::kAlloc,
                               stream>>>(mq, mk64, mv64, prm, ds->status_word);
        const cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
    });
}

// The single-pass forward for head dimension D: two Q tiles per work item up to D = 128 (one if
// `one_tile`), one Q tile per CTA above.
int launch_single(int D, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                  const CUtensorMap& mo, const AttnParams& p, DeviceState* ds, int64_t grid,
                  cudaStream_t stream, bool one_tile = false) {
    if (D <= 64)
        return one_tile ? launch_fwd<64, false, true>(mq, mk, mv, p, ds, grid, stream)
                        : launch_fwd<64, false>(mq, mk, mv, p, ds, grid, stream);
    if (D <= 128)
        return one_tile ? launch_fwd<128, false, true>(mq, mk, mv, p, ds, grid, stream)
                        : launch_fwd<128, false>(mq, mk, mv, p, ds, grid, stream);
    attn_fwd_d256_kernel<<<static_cast<unsigned int>(grid), kW256Threads, Fwd256Smem::kAlloc,
                           stream>>>(mq, mk, mv, mo, p, ds->status_word);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Launches `kernel` right behind the previous kernel on `stream` with programmatic dependent
// launch: it may be scheduled before that kernel has finished (once all of that kernel's CTAs
// have started) and waits for it itself (griddep_wait) before it reads that kernel's results,
// so its launch and set-up overlap the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int D>
int launch_merge(const AttnParams& p, __nv_bfloat16* out, int d_out, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.N;
    const int64_t blocks = (rows + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
    const bool contiguous = p.o_sn == d_out && p.o_sh == static_cast<long long>(p.N) * d_out &&
                            p.o_sb == static_cast<long long>(p.Hq) * p.N * d_out;
    const cudaError_t e = launch_dependent(
        contiguous ? attn_splitkv_merge_kernel<D, false> : attn_splitkv_merge_kernel<D, true>,
        dim3(static_cast<unsigned int>(blocks)), dim3(kMergeThreads),
        0, stream, static_cast<const float*>(p.ws_o), static_cast<const float*>(p.ws_lse), out,
        p.lse, p.B * p.Hq, p.Hq, p.N, d_out, p.o_sb, p.o_sh, p.o_sn, p.n_tiles, p.causal,
        p.n_splits, p.split_tiles);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Split-KV with 2..kMaxClusterSplits splits: the splits of a work item are one thread-block
// cluster, one work unit per CTA (so no claim counter), and they merge their partials through
// distributed shared memory at the end: no workspace, no merge kernel.
template <int D>
int launch_cluster_split(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const AttnParams& p, DeviceState* ds, int64_t units,
                         cudaStream_t stream) {
    AttnParams prm = p;
    prm.items = static_cast<int>(units);
    prm.sched = nullptr;
    prm.ws_o = nullptr;
    prm.ws_lse = nullptr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned int>(units));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SmemLayout<D>::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned int>(p.n_splits);  // the item's splits
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D, true, false, true>, mq, mk,
                                             mv, prm, ds->status_word);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Whether `items` work items split n ways run as clusters that all fit on the device at once.
bool cluster_fits(const DeviceState* ds, int D, int64_t items, int n) {
    return n >= 2 && n <= kMaxClusterSplits && D <= 128 && items <= ds->cluster_fit[D > 64][n];
}

// Effective split layout for a requested count: tiles per split and the number of non-empty
// splits (every split but the last holds split_tiles KV tiles).
void split_layout(int64_t n_tiles, int requested, int* split_tiles, int* n_splits) {
    const int64_t want = requested < 1 ? 1 : (requested > kMaxSplits ? kMaxSplits : requested);
    const int64_t tps = (n_tiles + want - 1) / want;
    *split_tiles = static_cast<int>(tps);
    *n_splits = static_cast<int>((n_tiles + tps - 1) / tps);
}

// The kernels compute on D padded to 64 or 128 columns (the TMA zero-fills the rest), so the
// fp32 partials are D_pad wide.
int64_t padded_dim(int64_t D) { return D <= 64 ? 64 : 128; }

int64_t workspace_bytes_for(int64_t bh, int64_t N, int64_t D, int n_splits) {
    return static_cast<int64_t>(n_splits) * bh * N * (padded_dim(D) + 1) * 4;
}

// ---- split choice: a cost model of the forward's launches -------------------------------------
// Estimated time (us) of a launch, calibrated on GB300 against CUDA-event times of 80 problems
// (B = 1, Hq 1-8, N 1024-16384, D 64 and 128, causal or not; cold L2) for the single pass and for
// 2-4 splits on either split path; it ranks the choices within ~7 % RMS:
//   kLaunchUs        launch, start-up and tail of a persistent or one-unit-per-CTA launch
//   kPairStepUs      a key tile of a work unit in which both of its Q tiles take part
//   kLoneStepUs      a key tile of a unit with one Q tile taking part (one-tile items; the
//                    causal diagonal's extra step)
//   kUnitUs          a unit's Q load and epilogue
//   kMergeUs + traffic / kMergeBytesPerUs   the workspace path: fp32 partials written by the split
//                    kernel and read by the merge kernel (n_splits x rows x (D_pad + 1) x 4 bytes,
//                    both ways), the merge's own launch hidden behind the split kernel's tail
//   kClusterLaunchUs the cluster path's launch, start-up and in-cluster merge (staging O and LSE
//                    in shared memory and reading the peers' rows through distributed shared
//                    memory)
// The persistent launches claim units heaviest first, so their makespan is that of list
// scheduling in claim order over min(units, SMs) workers; a cluster launch runs every unit at
// once (one wave), so its makespan is its longest unit.
constexpr double kLaunchUs = 10.0, kPairStepUs = 1.2, kLoneStepUs = 1.0, kUnitUs = 0.5;
constexpr double kSkipUnitUs = 0.2;  // a unit whose Q tiles see none of its split's keys
constexpr double kMergeUs = 2.0, kMergeBytesPerUs = 3.0e6;
constexpr double kClusterLaunchUs = 17.5;
constexpr int kModelMaxSplits = 16;

struct ForwardShape {
    int64_t bh, n_tiles;
    int D;
    bool causal;
};

// What the model needs of the device: its SM count and how many clusters of n split CTAs fit at
// once (for the shape's head dimension).
struct SplitDevice {
    int num_sms;
    int cluster_fit[kMaxClusterSplits + 1];
    bool fits(int64_t items, int n) const {
        return n >= 2 && n <= kMaxClusterSplits && items <= cluster_fit[n];
    }
};
SplitDevice split_device(const DeviceState* ds, int D) {
    SplitDevice d{ds->num_sms, {}};
    for (int n = 0; n <= kMaxClusterSplits; ++n) d.cluster_fit[n] = ds->cluster_fit[D > 64][n];
    return d;
}

// Key-tile steps of Q tiles 2p and 2p + 1 (s0, s1) within KV tiles [kb, ke).
inline void unit_steps(const ForwardShape& f, int64_t p, int64_t kb, int64_t ke, int64_t* s0,
                       int64_t* s1) {
    const int64_t t0 = 2 * p, t1 = 2 * p + 1;
    const int64_t l0 = std::min(ke - 1, f.causal ? t0 : f.n_tiles - 1);
    const int64_t l1 = std::min(ke - 1, f.causal ? t1 : f.n_tiles - 1);
    *s0 = std::max<int64_t>(0, l0 - kb + 1);
    *s1 = t1 < f.n_tiles ? std::max<int64_t>(0, l1 - kb + 1) : 0;
}

inline double unit_cost(int64_t s0, int64_t s1) {
    if (s0 == 0 && s1 == 0) return kSkipUnitUs;
    return kUnitUs + kPairStepUs * static_cast<double>(std::min(s0, s1)) +
           kLoneStepUs * static_cast<double>(std::max(s0, s1) - std::min(s0, s1));
}

// List scheduling over `workers`, units in claim order: each goes to the earliest-free worker.
class Makespan {
  public:
    explicit Makespan(int64_t workers) : free_(static_cast<size_t>(workers), 0.0) {}
    void add(double cost) {
        std::pop_heap(free_.begin(), free_.end(), std::greater<double>());
        free_.back() += cost;
        std::push_heap(free_.begin(), free_.end(), std::greater<double>());
    }
    double value() const { return *std::max_element(free_.begin(), free_.end()); }

  private:
    std::vector<double> free_;  // min-heap of the workers' finishing times
};

// The single pass: pairs of Q tiles, or single Q tiles when pairs would leave more than half of
// the SMs idle (as prefer_single_tiles decides).
double estimate_single(const ForwardShape& f, int num_sms) {
    const int64_t pairs = (f.n_tiles + 1) / 2;
    const bool one = 2 * pairs * f.bh <= num_sms;
    const int64_t items = (one ? f.n_tiles : pairs) * f.bh;
    Makespan ms(std::min<int64_t>(items, num_sms));
    if (one) {
        for (int64_t t = f.n_tiles - 1; t >= 0; --t) {
            const double c = kUnitUs + kLoneStepUs * static_cast<double>(f.causal ? t + 1 : f.n_tiles);
            for (int64_t h = 0; h < f.bh; ++h) ms.add(c);
        }
    } else {
        for (int64_t p = pairs - 1; p >= 0; --p) {
            int64_t s0, s1;
            unit_steps(f, p, 0, f.n_tiles, &s0, &s1);
            const double c = unit_cost(s0, s1);
            for (int64_t h = 0; h < f.bh; ++h) ms.add(c);
        }
    }
    return kLaunchUs + ms.value();
}

// n splits of tps key tiles each; `cluster`: merged inside one-wave clusters, else through the
// workspace and the merge kernel.
double estimate_split(const ForwardShape& f, int tps, int n, bool cluster, int num_sms) {
    const int64_t pairs = (f.n_tiles + 1) / 2;
    if (cluster) {  // one wave: the longest unit (the last pair's, or the first split's)
        double longest = 0.0;
        for (int64_t p = pairs - 1; p >= std::max<int64_t>(0, pairs - 2); --p)
            for (int k = 0; k < n; ++k) {
                int64_t s0, s1;
                unit_steps(f, p, int64_t(k) * tps, std::min<int64_t>(f.n_tiles, int64_t(k + 1) * tps),
                           &s0, &s1);
                longest = std::max(longest, unit_cost(s0, s1));
            }
        return kClusterLaunchUs + longest;
    }
    Makespan ms(std::min<int64_t>(pairs * f.bh * n, num_sms));
    for (int64_t p = pairs - 1; p >= 0; --p) {
        double c[kMaxSplits];
        for (int k = 0; k < n; ++k) {
            int64_t s0, s1;
            unit_steps(f, p, int64_t(k) * tps, std::min<int64_t>(f.n_tiles, int64_t(k + 1) * tps),
                       &s0, &s1);
            c[k] = unit_cost(s0, s1);
        }
        for (int64_t h = 0; h < f.bh; ++h)
            for (int k = 0; k < n; ++k) ms.add(c[k]);
    }
    const double traffic = 2.0 * n * static_cast<double>(f.bh) * f.n_tiles * kBM *
                           (padded_dim(f.D) + 1) * 4.0;
    return kLaunchUs + ms.value() + kMergeUs + traffic / kMergeBytesPerUs;
}

// The split count with the lowest estimate: the single pass or 2..kModelMaxSplits splits
// (cluster_only: only splits that merge inside one-wave clusters, as attn_fwd can run without a
// workspace; max_ws: the largest workspace a workspace-path candidate may need).  Problems with at
// least twice as many Q-tile pairs as SMs are not split: their single pass already fills the SMs
// in balanced waves.  A split must beat the single pass by kSplitMarginUs.
constexpr double kSplitMarginUs = 1.0;
int choose_splits(const ForwardShape& f, const SplitDevice& dev, bool cluster_only,
                  int64_t max_ws) {
    const int64_t pairs = (f.n_tiles + 1) / 2;
    const int64_t items = pairs * f.bh;
    if (f.D > 128 || f.n_tiles < 2 || items >= 2 * static_cast<int64_t>(dev.num_sms)) return 1;
    int best = 1;
    double best_us = estimate_single(f, dev.num_sms) - kSplitMarginUs;
    int last_n = 1;
    for (int want = 2; want <= (cluster_only ? kMaxClusterSplits : kModelMaxSplits); ++want) {
        int tps = 0, n = 0;
        split_layout(f.n_tiles, want, &tps, &n);
        if (n == last_n) continue;  // the same layout as a smaller request
        last_n = n;
        const bool cluster = dev.fits(items, n);
        if (cluster_only && !cluster) continue;
        if (!cluster_only && workspace_bytes_for(f.bh, f.n_tiles * kBM, f.D, n) > max_ws) continue;
        const double us = estimate_split(f, tps, n, cluster, dev.num_sms);
        if (us < best_us) {
            best = n;
            best_us = us;
        }
    }
    return best;
}

// attn_fwd_splitkv's default split count, cached per shape (the list-scheduling estimate of a
// few thousand units takes up to a few milliseconds of host time).
struct SplitCacheKey {
    int64_t bh, n_tiles, max_ws;
    int dev, D, causal, cluster_only;
    bool operator==(const SplitCacheKey& o) const {
        return bh == o.bh && n_tiles == o.n_tiles && max_ws == o.max_ws && dev == o.dev &&
               D == o.D && causal == o.causal && cluster_only == o.cluster_only;
    }
};
std::mutex g_split_cache_lock;
std::vector<std::pair<SplitCacheKey, int>> g_split_cache;  // small; cleared when it grows

int default_splits(int64_t bh, int64_t N, int D, bool causal, int64_t max_ws,
                   const DeviceState* ds, int dev, bool cluster_only = false) {
    const ForwardShape f{bh, (N + kBM - 1) / kBM, D <= 64 ? 64 : 128, causal};
    // the cases choose_splits settles at once (most problems) skip the cache
    if (D > 128 || f.n_tiles < 2 || (f.n_tiles + 1) / 2 * bh >= 2 * int64_t(ds->num_sms)) return 1;
    const SplitCacheKey key{bh, f.n_tiles, max_ws, dev, f.D, causal ? 1 : 0, cluster_only ? 1 : 0};
    {
        std::lock_guard<std::mutex> guard(g_split_cache_lock);
        for (const auto& e : g_split_cache)
            if (e.first == key) return e.second;
    }
    const int n = choose_splits(f, split_device(ds, D), cluster_only, max_ws);
    std::lock_guard<std::mutex> guard(g_split_cache_lock);
    if (g_split_cache.size() >= 1024) g_split_cache.clear();
    g_split_cache.emplace_back(key, n);
    return n;
}

// attn_fwd's own split.  Outside a graph capture both split paths are candidates (the workspace
// path's partials in a leased slot of g_fwd_scratch); while the stream is being captured (the
// host cannot order a graph's replays against other users of a slot), only splits that merge
// inside one-wave clusters.
int auto_splits(const Problem& P, const DeviceState* ds, bool cluster_only) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return default_splits(P.bh, P.N, P.D, P.causal != 0,
                          cluster_only ? 0 : static_cast<int64_t>(kFwdScratchBytes), ds, dev,
                          cluster_only);
}

// Runs launch(scratch) with one of the device's kFwdScratchSlots slots of g_fwd_scratch that no
// other executing launch holds: taken round robin and held as on_slot describes.  Not for
// streams being captured.
template <class Launch>
int with_scratch(DeviceState* ds, cudaStream_t s, Launch&& launch) {
    const unsigned int idx =
        ds->scratch_next.fetch_add(1u, std::memory_order_relaxed) % kFwdScratchSlots;
    unsigned char* scratch = ds->fwd_scratch + static_cast<size_t>(idx) * kFwdScratchBytes;
    return on_slot(ds->scratch_slots[idx], s, [&]() { return launch(scratch); });
}

}  // namespace

// With fewer Q-tile pairs than half the SMs, one Q tile per work item, so that twice as many SMs
// work: a pair hides the S -> softmax -> P.V latency of one tile behind the other's, but when
// pairs would leave most SMs idle the extra SMs gain more.  (Single-pass launches only; the
// split-KV path fills the SMs with splits instead.)
static bool prefer_single_tiles(Problem& P, const DeviceState* ds, AttnParams* prm) {
    if (P.D > 128 || P.n_tiles < 2 || 2 * P.items > ds->num_sms) return false;
    prm->n_pairs = static_cast<int>(P.n_tiles);
    P.items = P.n_tiles * P.bh;
    prm->items = static_cast<int>(P.items);
    return true;
}

// The forward of a validated, non-empty problem: the single pass, or (allow_split) the split
// that auto_splits picks.
static int run_forward(Problem& P, bool allow_split, cudaStream_t s) {
    DeviceState* ds = nullptr;
    CUtensorMap mq, mk, mv, mo;
    AttnParams prm;
    int st = prepare(P, &ds, &mq, &mk, &mv, &mo, &prm);
    if (st != ATTN_OK) return st;
    int n = 1;
    if (allow_split) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        const cudaError_t e = cudaStreamIsCapturing(s, &cap);
        if (e != cudaSuccess) return cuda_fail(e);
        n = auto_splits(P, ds, cap != cudaStreamCaptureStatusNone);
    }
    if (n > 1) {
        split_layout(P.n_tiles, n, &prm.split_tiles, &prm.n_splits);
        const int64_t units = P.items * prm.n_splits;
        if (cluster_fits(ds, P.D, P.items, prm.n_splits))
            return P.D <= 64 ? launch_cluster_split<64>(mq, mk, mv, prm, ds, units, s)
                             : launch_cluster_split<128>(mq, mk, mv, prm, ds, units, s);
        // the workspace path (auto_splits allowed it: not capturing, partials within one scratch
        // slot)
        return with_scratch(ds, s, [&](unsigned char* scratch) {
            prm.ws_o = reinterpret_cast<float*>(scratch);
            prm.ws_lse = prm.ws_o + static_cast<int64_t>(prm.n_splits) * P.bh * P.N *
                                        padded_dim(P.D);
            auto* o = static_cast<__nv_bfloat16*>(P.out);
            auto after = [&]() {
                return P.D <= 64 ? launch_merge<64>(prm, o, P.D, s)
                                 : launch_merge<128>(prm, o, P.D, s);
            };
            return P.D <= 64 ? launch_fwd<64, true>(mq, mk, mv, prm, ds, units, s, after)
                             : launch_fwd<128, true>(mq, mk, mv, prm, ds, units, s, after);
        });
    }
    const bool one_tile = prefer_single_tiles(P, ds, &prm);
    return launch_single(P.D, mq, mk, mv, mo, prm, ds, P.items, s, one_tile);
}

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                        int Hq, int Hkv, int N, int D, int causal, float sm_scale, void* stream) {
    Problem P{q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale};
    bool empty = false;
    const int st = validate(P, &empty);
    if (st != ATTN_OK || empty) return st;
    return run_forward(P, true, static_cast<cudaStream_t>(stream));
}

extern "C" int attn_fwd_num_splits(int B, int Hq, int N, int D, int causal) {
    if (B <= 0 || Hq <= 0 || N <= 0 || D % 8 != 0 || D < 8 || D > 256) return 1;
    DeviceState* ds = nullptr;
    if (current_device_state(&ds) != ATTN_OK) return 1;
    Problem P{};
    P.D = D;
    P.causal = causal;
    P.bh = static_cast<int64_t>(B) * Hq;
    P.n_tiles = (static_cast<int64_t>(N) + kBM - 1) / kBM;
    P.items = (P.n_tiles + 1) / 2 * P.bh;
    P.N = N;
    return auto_splits(P, ds, false);
}

extern "C" int attn_fwd_strided(const void* q, const void* k, const void* v, void* out,
                                float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                                float sm_scale, const long long* q_strides,
                                const long long* k_strides, const long long* v_strides,
                                const long long* o_strides, void* stream) {
    if (!q_strides || !k_strides || !v_strides || !o_strides) return ATTN_ERR_NULL;
    Problem P{q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale};
    P.strided = true;
    // caller order per tensor: {batch, head, row} strides in elements
    P.sq = {q_strides[2], q_strides[1], q_strides[0]};
    P.sk = {k_strides[2], k_strides[1], k_strides[0]};
    P.sv = {v_strides[2], v_strides[1], v_strides[0]};
    P.so = {o_strides[2], o_strides[1], o_strides[0]};
    bool empty = false;
    const int st = validate(P, &empty);
    if (st != ATTN_OK || empty) return st;
    return run_forward(P, true, static_cast<cudaStream_t>(stream));
}

extern "C" int attn_fwd_test_stall(const void* q, const void* k, const void* v, void* out,
                                   float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                                   float sm_scale, int stall_item, void* stream) {
    if (D > 128) return ATTN_ERR_HEADDIM;  // the hook lives in the two-tile kernel
    Problem P{q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale};
    bool empty = false;
    int st = validate(P, &empty);
    if (st != ATTN_OK || empty) return st;
    if (stall_item < 0) return ATTN_ERR_SHAPE;
    DeviceState* ds = nullptr;
    CUtensorMap mq, mk, mv, mo;
    AttnParams prm;
    st = prepare(P, &ds, &mq, &mk, &mv, &mo, &prm);
    if (st != ATTN_OK) return st;
    prm.stall_item = stall_item;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return D <= 64 ? launch_fwd<64, false>(mq, mk, mv, prm, ds, P.items, s)
                   : launch_fwd<128, false>(mq, mk, mv, prm, ds, P.items, s);
}

extern "C" int attn_fwd_test_kernel(const void* q, const void* k, const void* v, void* out,
                                    float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                                    float sm_scale, int kernel, int stall_item, void* stream) {
    if (kernel < 1 || kernel > 3) return ATTN_ERR_SHAPE;
    if (stall_item < -1) return ATTN_ERR_SHAPE;
    if (D > 128 || (kernel == 2 && D <= 64)) return ATTN_ERR_HEADDIM;
    Problem P{q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale};
    bool empty = false;
    int st = validate(P, &empty);
    if (st != ATTN_OK || empty) return st;
    DeviceState* ds = nullptr;
    CUtensorMap mq, mk, mv, mo;
    AttnParams prm;
    st = prepare(P, &ds, &mq, &mk, &mv, &mo, &prm);
    if (st != ATTN_OK) return st;
    prm.stall_item = stall_item;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kernel == 2) {
        if (ds->pair_clusters < 1) return ATTN_ERR_ARCH;
        return launch_pair(P, mq, prm, ds, s);
    }
    if (kernel == 3) {  // two key-axis splits merged inside clusters
        split_layout(P.n_tiles, 2, &prm.split_tiles, &prm.n_splits);
        if (prm.n_splits != 2 || !cluster_fits(ds, D, P.items, 2)) return ATTN_ERR_SHAPE;
        return D <= 64 ? launch_cluster_split<64>(mq, mk, mv, prm, ds, P.items * 2, s)
                       : launch_cluster_split<128>(mq, mk, mv, prm, ds, P.items * 2, s);
    }
    return D <= 64 ? launch_fwd<64, false>(mq, mk, mv, prm, ds, P.items, s)
                   : launch_fwd<128, false>(mq, mk, mv, prm, ds, P.items, s);
}

extern "C" int attn_fwd_test_split_choice(int B, int Hq, int N, int D, int causal, int num_sms,
                                          const int* cluster_fit, int cluster_only,
                                          long long max_ws) {
    if (B <= 0 || Hq <= 0 || N <= 0 || D % 8 != 0 || D < 8 || D > 256 || num_sms <= 0 ||
        !cluster_fit || max_ws < 0)
        return ATTN_ERR_SHAPE;
    SplitDevice dev{num_sms, {}};
    for (int n = 2; n <= kMaxClusterSplits; ++n) dev.cluster_fit[n] = cluster_fit[n - 2];
    const int64_t bh = static_cast<int64_t>(B) * Hq;
    const int64_t n_tiles = (static_cast<int64_t>(N) + kBM - 1) / kBM;
    const ForwardShape f{bh, n_tiles, D, causal != 0};
    const int n = choose_splits(f, dev, cluster_only != 0, max_ws);
    int tps = 0, eff = 0;
    split_layout(n_tiles, n, &tps, &eff);
    return eff;
}

namespace {
// The default split count for these sizes on the current device (1 on any failure), limited to
// splits whose workspace fits max_ws bytes.
int splitkv_default(int B, int Hq, int N, int D, int causal, int64_t max_ws) {
    if (B <= 0 || Hq <= 0 || N <= 0 || D % 8 != 0 || D < 8 || D > 128) return 1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    DeviceState* ds = nullptr;
    if (device_state(dev, &ds) != ATTN_OK) return 1;
    const int n = default_splits(static_cast<int64_t>(B) * Hq, N, D, causal != 0, max_ws, ds, dev);
    int tps = 0, eff = 0;
    split_layout((static_cast<int64_t>(N) + kBM - 1) / kBM, n, &tps, &eff);
    return eff;
}
}  // namespace

extern "C" int attn_fwd_splitkv_num_splits(int B, int Hq, int N, int D, int causal) {
    return splitkv_default(B, Hq, N, D, causal, INT64_MAX);
}

extern "C" size_t attn_fwd_splitkv_workspace_bytes(int B, int Hq, int N, int D, int num_splits) {
    if (B <= 0 || Hq <= 0 || N <= 0 || D % 8 != 0 || D < 8 || D > 256) return 0;
    if (D > 128) return 0;  // single pass
    const int64_t n_tiles = (static_cast<int64_t>(N) + kBM - 1) / kBM;
    const int64_t bh = static_cast<int64_t>(B) * Hq;
    auto bytes = [&](int requested) -> int64_t {
        int tps = 0, n = 0;
        split_layout(n_tiles, requested, &tps, &n);
        return n <= 1 ? 0 : workspace_bytes_for(bh, N, D, n);
    };
    // The default count depends on the causal mask, which this query does not take: enough for
    // either.
    if (num_splits == 0)
        return static_cast<size_t>(std::max(bytes(attn_fwd_splitkv_num_splits(B, Hq, N, D, 0)),
                                            bytes(attn_fwd_splitkv_num_splits(B, Hq, N, D, 1))));
    return static_cast<size_t>(bytes(num_splits));
}

extern "C" int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* out,
                                float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                                float sm_scale, int num_splits, void* workspace,
                                size_t workspace_bytes, void* stream) {
    if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_SPLITS;
    Problem P{q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale};
    bool empty = false;
    int st = validate(P, &empty);
    if (st != ATTN_OK || empty) return st;
    if (num_splits == 0) num_splits = attn_fwd_splitkv_num_splits(B, Hq, N, D, causal);
    int split_tiles = 0, n_splits = 0;
    split_layout(P.n_tiles, num_splits, &split_tiles, &n_splits);
    if (D > 128) n_splits = 1;  // the wide-head kernel has no split variant
    if (n_splits <= 1)  // one split is the single pass; the workspace is not touched
        return run_forward(P, false, static_cast<cudaStream_t>(stream));

    // The workspace is checked the same way whichever path runs below, so the call's result
    // does not depend on how many clusters the device fits.
    const int64_t need = workspace_bytes_for(P.bh, N, D, n_splits);
    if (!workspace) return ATTN_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return ATTN_ERR_ALIGN;
    if (static_cast<int64_t>(workspace_bytes) < need) return ATTN_ERR_WORKSPACE;
    if (overlaps(workspace, need, q, P.q_bytes) || overlaps(workspace, need, k, P.kv_bytes) ||
        overlaps(workspace, need, v, P.kv_bytes) || overlaps(workspace, need, out, P.q_bytes) ||
        overlaps(workspace, need, lse, P.lse_bytes))
        return ATTN_ERR_ALIAS;
    if (P.items * n_splits > 0x7fffffffLL) return ATTN_ERR_SHAPE;

    DeviceState* ds = nullptr;
    CUtensorMap mq, mk, mv, mo;
    AttnParams prm;
    st = prepare(P, &ds, &mq, &mk, &mv, &mo, &prm);
    if (st != ATTN_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || check_memory(workspace, dev) != ATTN_OK)
        return ATTN_ERR_MEMORY;
    prm.n_splits = n_splits;
    prm.split_tiles = split_tiles;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t items = P.items * n_splits;
    // Splits whose clusters all fit on the device at once merge inside their cluster (the
    // workspace stays untouched); otherwise the persistent split kernel writes the partials to
    // the workspace and the merge kernel combines them (its dynamic claims balance the uneven
    // causal splits over several waves, which a one-unit-per-CTA cluster launch cannot).
    if (cluster_fits(ds, D, P.items, n_splits))
        return D <= 64 ? launch_cluster_split<64>(mq, mk, mv, prm, ds, items, s)
                       : launch_cluster_split<128>(mq, mk, mv, prm, ds, items, s);
    prm.ws_o = static_cast<float*>(workspace);
    prm.ws_lse = prm.ws_o + static_cast<int64_t>(n_splits) * P.bh * N * padded_dim(D);
    auto* o = static_cast<__nv_bfloat16*>(out);
    // the merge kernel follows the split kernel directly (programmatic dependent launch): the
    // claim counter's completion event is recorded after both
    auto after = [&]() {
        return D <= 64 ? launch_merge<64>(prm, o, D, s) : launch_merge<128>(prm, o, D, s);
    };
    return D <= 64 ? launch_fwd<64, true>(mq, mk, mv, prm, ds, items, s, after)
                   : launch_fwd<128, true>(mq, mk, mv, prm, ds, items, s, after);
}

// ------------------------------------------------------------------------------------------------
// Backward
// ------------------------------------------------------------------------------------------------
namespace {

template <int D>
int launch_bwd(const Problem& P, const CUtensorMap& mq, const CUtensorMap& mk,
               const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mdk,
               const CUtensorMap& mdv, const BwdParams& bp_in, const void* out, const void* dout,
               float* delta, DeviceState* ds, cudaStream_t s) {
    BwdParams bp = bp_in;
    unsigned int* status_word = ds->status_word;
    const int num_sms = ds->num_sms;
    const long long rows = P.bh * P.N;
    // persistent dQ: one CTA per SM (or per item, if fewer)
    const int64_t dq_grid = std::min<int64_t>(bp.items, std::max(1, num_sms));
    // Delta, then dK/dV and dQ each launched directly behind the previous kernel (programmatic
    // dependent launch: each waits for its predecessor before reading what it wrote); the claim
    // counter (dQ's) covers the whole chain, so nothing else separates them on the stream.
    return with_claim_counter(ds, s, [&](unsigned int* counter) {
        bp.sched = counter;
        attn_bwd_delta_kernel<<<static_cast<unsigned int>((rows + 7) / 8), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout),
            delta, rows, P.D);
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess)
            e = launch_dependent(attn_bwd_dkdv_kernel<D>,
                                 dim3(static_cast<unsigned int>(P.n_tiles * P.bh_kv)),
                                 dim3(kBwdThreads), DkdvSmem<D>::kAlloc, s, mq, mk, mv, mdo, mdk,
                                 mdv, bp, status_word);
        if (e == cudaSuccess)
            e = launch_dependent(attn_bwd_dq_kernel<D>, dim3(static_cast<unsigned int>(dq_grid)),
                                 dim3(kBwdThreads), DqSmem<D>::kAlloc, s, mq, mk, mv, mdo, bp,
                                 status_word);
        return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
    });
}

}  // namespace

extern "C" size_t attn_bwd_workspace_bytes(int B, int Hq, int N) {
    if (B <= 0 || Hq <= 0 || N <= 0) return 0;
    return static_cast<size_t>(B) * Hq * N * 4;
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                        int Hq, int Hkv, int N, int D, int causal, float sm_scale,
                        void* workspace, size_t workspace_bytes, void* stream) {
    if (D > 128) return ATTN_ERR_HEADDIM;  // the backward kernels hold at most 128 columns
    // the forward's checks cover q, k, v, out (here an input) and lse
    Problem P{q, k, v, const_cast<void*>(out), const_cast<float*>(lse), B, Hq, Hkv, N, D, causal,
              sm_scale};
    bool empty = false;
    int st = validate(P, &empty);
    if (st != ATTN_OK || empty) return st;
    if (!dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_NULL;
    const uintptr_t align_bits =
        reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv) |
        reinterpret_cast<uintptr_t>(workspace);
    if (align_bits & 15u) return ATTN_ERR_ALIGN;
    const int64_t ws_need = P.bh * N * 4;
    if (static_cast<int64_t>(workspace_bytes) < ws_need) return ATTN_ERR_WORKSPACE;
    // outputs (dq, dk, dv, workspace) must not overlap any input or each other
    const void* ins[] = {q, k, v, out, lse, dout};
    const int64_t in_bytes[] = {P.q_bytes, P.kv_bytes, P.kv_bytes, P.q_bytes, P.lse_bytes,
                                P.q_bytes};
    const void* outs[] = {dq, dk, dv, workspace};
    const int64_t out_bytes[] = {P.q_bytes, P.kv_bytes, P.kv_bytes, ws_need};
    for (int a = 0; a < 4; ++a) {
        for (int x = 0; x < 6; ++x)
            if (overlaps(outs[a], out_bytes[a], ins[x], in_bytes[x])) return ATTN_ERR_ALIAS;
        for (int c = a + 1; c < 4; ++c)
            if (overlaps(outs[a], out_bytes[a], outs[c], out_bytes[c])) return ATTN_ERR_ALIAS;
    }
    DeviceState* ds = nullptr;
    CUtensorMap mq, mk, mv, mo_unused;
    AttnParams prm;
    st = prepare(P, &ds, &mq, &mk, &mv, &mo_unused, &prm);
    if (st != ATTN_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    for (const void* ptr : {dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                            static_cast<const void*>(dv), static_cast<const void*>(workspace)})
        if (check_memory(ptr, dev) != ATTN_OK) return ATTN_ERR_MEMORY;
    CUtensorMap mdo, mdk, mdv;
    if (!cached_tile_map(&mdo, dout, B, Hq, N, D, P.sq) ||
        !cached_tile_map(&mdk, dk, B, Hkv, N, D, P.sk) ||
        !cached_tile_map(&mdv, dv, B, Hkv, N, D, P.sv))
        return cuda_fail(cudaErrorInvalidValue);
    BwdParams bp;
    bp.B = B;
    bp.Hq = Hq;
    bp.Hkv = Hkv;
    bp.N = N;
    bp.group = Hq / Hkv;
    bp.causal = causal ? 1 : 0;
    bp.n_tiles = static_cast<int>(P.n_tiles);
    bp.scale_log2 = sm_scale * 1.4426950408889634f;
    bp.sm_scale = sm_scale;
    bp.lse = lse;
    bp.delta = static_cast<const float*>(workspace);
    if (P.n_tiles * P.bh > 0x7fffffffLL) return ATTN_ERR_SHAPE;
    bp.items = static_cast<int>(P.n_tiles * P.bh);
    bp.sched = nullptr;  // set by with_claim_counter around the dQ launch
    bp.dq = static_cast<__nv_bfloat16*>(dq);
    bp.d_out = D;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* delta = static_cast<float*>(workspace);
    return D <= 64 ? launch_bwd<64>(P, mq, mk, mv, mdo, mdk, mdv, bp, out, dout, delta, ds, s)
                   : launch_bwd<128>(P, mq, mk, mv, mdo, mdk, mdv, bp, out, dout, delta, ds, s);
}

// ------------------------------------------------------------------------------------------------
// Absorbed MLA decode ("Attention Kernel 实现与正确性验证", walkerchi.com, sections 2.1-2.4)
// ------------------------------------------------------------------------------------------------
namespace {

// 3-D view [B, rows, 576] of a contiguous bf16 tensor; box = 64 columns x box_rows rows, 128B
// swizzle.  Rows past `rows` are zero-filled on load.
bool make_mla_map(CUtensorMap* map, const void* base, int64_t B, int64_t rows, int box_rows) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kMlaDqk), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kMlaDqk * 2),
                                   static_cast<cuuint64_t>(rows * kMlaDqk * 2)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

int64_t mla_items(int B, int H) {
    return static_cast<int64_t>(B) * ((H + kMlaHeads - 1) / kMlaHeads) * 2;
}

int64_t mla_tiles(int T) { return (static_cast<int64_t>(T) + kMlaBN - 1) / kMlaBN; }

// Splits of the token axis, from a cost model in units of one 64-token tile per CTA (about
// 1.8 us): CTAs run in waves of one per SM, and a split run also writes each split's fp32
// partial rows (2 KiB per head) and merges them, about 0.57 tile per thousand partial rows
// plus half a tile for the merge launch.  The least costly count wins (fewest splits on ties).
// (With 2-4 splits the merge runs inside a cluster and costs less than this; the model was
// fitted to the global-memory merge and still picks the faster count at B = 16 and 32.)
int mla_heuristic_splits(int64_t items, int64_t n_tiles, int64_t rows, int num_sms) {
    const int64_t max_s = std::min<int64_t>(n_tiles, kMaxSplits);
    int best = 1;
    int64_t best_cost = -1;
    for (int64_t s = 1; s <= max_s; ++s) {
        const int64_t waves = (items * s + num_sms - 1) / num_sms;
        int64_t cost = 1000 * waves * ((n_tiles + s - 1) / s);  // milli-tiles
        if (s > 1) cost += 500 + s * rows * 57 / 100;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = static_cast<int>(s);
        }
    }
    return best;
}

// fp32 O_s and LSE_s of every split, for the merge kernel (2..kMlaMaxClusterSplits splits merge
// inside a cluster and need none)
int64_t mla_workspace_for(int B, int H, int n_splits) {
    if (n_splits <= kMlaMaxClusterSplits) return 0;
    return static_cast<int64_t>(n_splits) * B * H * (kMlaDc + 1) * 4;
}

}  // namespace

extern "C" int attn_mla_decode_num_splits(int B, int H, int T) {
    if (B <= 0 || H <= 0 || T <= 0) return 1;
    DeviceState* ds = nullptr;
    if (current_device_state(&ds) != ATTN_OK) return 1;
    return mla_heuristic_splits(mla_items(B, H), mla_tiles(T), static_cast<int64_t>(B) * H,
                                ds->num_sms);
}

extern "C" size_t attn_mla_decode_workspace_bytes(int B, int H, int T, int num_splits) {
    if (B <= 0 || H <= 0 || T <= 0 || num_splits < 0 || num_splits > kMaxSplits) return 0;
    if (num_splits == 0) num_splits = attn_mla_decode_num_splits(B, H, T);
    num_splits = static_cast<int>(std::min<int64_t>(num_splits, mla_tiles(T)));
    return static_cast<size_t>(mla_workspace_for(B, H, num_splits));
}

namespace {

int mla_decode_run(const void* q, const void* kv, void* out, float* lse, int B, int H, int T,
                   int d_c, int d_r, float sm_scale, int num_splits, void* workspace,
                   size_t workspace_bytes, void* stream, int stall_tile) {
    if (B < 0 || H <= 0 || T <= 0) return ATTN_ERR_SHAPE;
    if (d_c != kMlaDc || d_r != kMlaDr) return ATTN_ERR_HEADDIM;
    if (!std::isfinite(sm_scale) || !(sm_scale > 0.f)) return ATTN_ERR_SCALE;
    if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_SPLITS;
    if (B == 0) return ATTN_OK;
    if (!q || !kv || !out || !lse) return ATTN_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) |
         reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(lse)) & 15u)
        return ATTN_ERR_ALIGN;
    const int64_t n_ht = (H + kMlaHeads - 1) / kMlaHeads;
    const int64_t n_tiles = mla_tiles(T);
    const int64_t items = mla_items(B, H);
    const int64_t q_bytes = static_cast<int64_t>(B) * H * kMlaDqk * 2;
    const int64_t kv_bytes = static_cast<int64_t>(B) * T * kMlaDqk * 2;
    const int64_t o_bytes = static_cast<int64_t>(B) * H * kMlaDc * 2;
    const int64_t lse_bytes = static_cast<int64_t>(B) * H * 4;
    if (overlaps(out, o_bytes, q, q_bytes) || overlaps(out, o_bytes, kv, kv_bytes) ||
        overlaps(out, o_bytes, lse, lse_bytes) || overlaps(lse, lse_bytes, q, q_bytes) ||
        overlaps(lse, lse_bytes, kv, kv_bytes))
        return ATTN_ERR_ALIAS;

    // An explicit split count is checked against the workspace before any CUDA call; the
    // default one needs the SM count first.
    auto check_workspace = [&](int n_splits) {
        if (items * n_splits > 0x7fffffffLL) return ATTN_ERR_SHAPE;
        const int64_t need = mla_workspace_for(B, H, n_splits);
        if (need == 0) return ATTN_OK;
        if (!workspace) return ATTN_ERR_NULL;
        if (reinterpret_cast<uintptr_t>(workspace) & 15u) return ATTN_ERR_ALIGN;
        if (static_cast<int64_t>(workspace_bytes) < need) return ATTN_ERR_WORKSPACE;
        if (overlaps(workspace, need, q, q_bytes) || overlaps(workspace, need, kv, kv_bytes) ||
            overlaps(workspace, need, out, o_bytes) || overlaps(workspace, need, lse, lse_bytes))
            return ATTN_ERR_ALIAS;
        return ATTN_OK;
    };
    int n_splits = static_cast<int>(std::min<int64_t>(num_splits, n_tiles));
    int st = num_splits > 0 ? check_workspace(n_splits) : ATTN_OK;
    if (st != ATTN_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceState* ds = nullptr;
    st = device_state(dev, &ds);
    if (st != ATTN_OK) return st;
    if (num_splits == 0) {
        n_splits = mla_heuristic_splits(items, n_tiles, static_cast<int64_t>(B) * H, ds->num_sms);
        st = check_workspace(n_splits);
        if (st != ATTN_OK) return st;
    }
    for (const void* ptr : {q, kv, static_cast<const void*>(out), static_cast<const void*>(lse)})
        if (check_memory(ptr, dev) != ATTN_OK) return ATTN_ERR_MEMORY;
    const bool cluster = n_splits > 1 && n_splits <= kMlaMaxClusterSplits;
    if (n_splits > 1 && !cluster && check_memory(workspace, dev) != ATTN_OK) return ATTN_ERR_MEMORY;

    CUtensorMap mq, mkv;
    if (!make_mla_map(&mq, q, B, H, kMlaHeads) || !make_mla_map(&mkv, kv, B, T, kMlaBN))
        return cuda_fail(cudaErrorInvalidValue);
    MlaParams prm;
    prm.B = B;
    prm.H = H;
    prm.T = T;
    prm.n_ht = static_cast<int>(n_ht);
    prm.n_tiles = static_cast<int>(n_tiles);
    prm.n_splits = n_splits;
    prm.scale_log2 = sm_scale * 1.4426950408889634f;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    // With a few splits the CTAs of a group form a cluster and merge through distributed shared
    // memory (no partials in global memory, no second launch); with more, the partials go to the
    // workspace and the merge kernel spreads the rows over the GPU.
    prm.cluster_merge = cluster ? 1 : 0;
    prm.ws_o = n_splits > 1 && !cluster ? static_cast<float*>(workspace) : nullptr;
    prm.ws_lse = prm.ws_o ? prm.ws_o + static_cast<int64_t>(n_splits) * B * H * kMlaDc : nullptr;
    prm.stall_tile = stall_tile;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cluster) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned int>(items * n_splits));
        cfg.blockDim = dim3(kMlaThreads);
        cfg.dynamicSmemBytes = MlaSmem::kAlloc;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned int>(n_splits);  // the group's splits
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, mq, mkv, prm, ds->status_word);
    } else {
        mla_decode_kernel<<<static_cast<unsigned int>(items * n_splits), kMlaThreads,
                            MlaSmem::kAlloc, s>>>(mq, mkv, prm, ds->status_word);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return cuda_fail(e);
    if (n_splits > 1 && !cluster) {
        const int64_t rows = static_cast<int64_t>(B) * H;
        const int64_t rows_per_block = 4 / mla_merge_groups(n_splits);
        e = launch_dependent(
            mla_merge_kernel,
            dim3(static_cast<unsigned int>((rows + rows_per_block - 1) / rows_per_block)),
            dim3(kMlaMergeThreads), 0, s, static_cast<const float*>(prm.ws_o),
            static_cast<const float*>(prm.ws_lse), prm.out, lse, static_cast<int>(rows), n_splits);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return ATTN_OK;
}

}  // namespace

extern "C" int attn_mla_decode(const void* q, const void* kv, void* out, float* lse, int B, int H,
                               int T, int d_c, int d_r, float sm_scale, int num_splits,
                               void* workspace, size_t workspace_bytes, void* stream) {
    return mla_decode_run(q, kv, out, lse, B, H, T, d_c, d_r, sm_scale, num_splits, workspace,
                          workspace_bytes, stream, -1);
}

extern "C" int attn_mla_decode_test_stall(const void* q, const void* kv, void* out, float* lse,
                                          int B, int H, int T, int d_c, int d_r, float sm_scale,
                                          int num_splits, void* workspace,
                                          size_t workspace_bytes, int stall_tile, void* stream) {
    if (stall_tile < 0) return ATTN_ERR_SHAPE;
    return mla_decode_run(q, kv, out, lse, B, H, T, d_c, d_r, sm_scale, num_splits, workspace,
                          workspace_bytes, stream, stall_tile);
}

extern "C" const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL: return "a required pointer is NULL";
        case ATTN_ERR_SHAPE: return "invalid or overflowing shape (B, Hq, Hkv, N)";
        case ATTN_ERR_HEADS: return "Hq is not a multiple of Hkv";
        case ATTN_ERR_HEADDIM:
            return "unsupported head dimension (attention: D a multiple of 8 in [8, 256], "
                   "backward [8, 128]; MLA decode: d_c = 512 and d_r = 64)";
        case ATTN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case ATTN_ERR_SCALE: return "sm_scale must be finite and positive";
        case ATTN_ERR_ARCH:
            return "the device is not sm_103 (GB300), its shared memory is misaligned, or a kernel "
                   "was built with an unexpected register count";
        case ATTN_ERR_CUDA: return "a CUDA call failed (see attn_last_cuda_error)";
        case ATTN_ERR_TIMEOUT: return "a device-side bounded wait expired";
        case ATTN_ERR_MEMORY: return "a pointer is not device memory of the current device";
        case ATTN_ERR_ALIAS: return "out/lse/workspace overlap an input or each other";
        case ATTN_ERR_SPLITS: return "num_splits must be in [0, 64]";
        case ATTN_ERR_WORKSPACE:
            return "workspace smaller than the entry point's *_workspace_bytes() figure";
        case ATTN_ERR_STRIDE:
            return "a stride is not a positive multiple of 8 elements (16 bytes) below 2^39";
        case ATTN_ERR_SCRATCH:
            return "problem needs more split-KV scratch than the built-in buffer "
                   "(attn_fwd_splitkv_noalloc_max_bytes)";
        case ATTN_ERR_RANGE:
            return "an index check of the debug build failed (the access was skipped)";
        default: return "unknown status";
    }
}

extern "C" int attn_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int attn_debug_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int word = 0;
    const unsigned int zero = 0;
    e = cudaMemcpyFromSymbolAsync(&word, g_attn_status_word, sizeof word, 0,
                                  cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_attn_status_word, &zero, sizeof zero, 0,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (word & kDevTimeout) return ATTN_ERR_TIMEOUT;
    if (word & kDevRange) return ATTN_ERR_RANGE;
    return (word & kDevSmemAlign) ? ATTN_ERR_ARCH : ATTN_OK;
}

// ------------------------------------------------------------------------------------------------
// Split-KV forward without any device allocation.
//
// Some callers cannot allocate device memory when they call us: a plug-in whose host application
// owns the whole device-memory budget, or a latency-critical serving loop that forbids
// allocation after start-up.  For them the split partials live in this fixed, file-scope device
// buffer instead of a caller-provided workspace.  Every GPU that loads the library holds it
// (kNoAllocScratchBytes) until the process exits.
// ------------------------------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_splitkv_scratch[kNoAllocScratchBytes];

// In host code `g_splitkv_scratch` only names a host-side stand-in for the device array, so the
// device address is looked up per device (with that device current) and cached once the lookup
// has succeeded.  A failed lookup (for instance one attempted while a stream capture forbids it)
// is not cached: the next call tries again.
struct ScratchState {
    std::mutex lock;
    void* ptr = nullptr;
};
ScratchState g_scratch[kMaxDevices];

int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    ScratchState& st = g_scratch[dev];
    std::lock_guard<std::mutex> guard(st.lock);
    if (st.ptr == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_splitkv_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        st.ptr = ptr;
    }
    *out = st.ptr;
    return ATTN_OK;
}

}  // namespace

extern "C" size_t attn_fwd_splitkv_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* out,
                                        float* lse, int B, int Hq, int Hkv, int N, int D,
                                        int causal, float sm_scale, int num_splits,
                                        void* stream) {
    if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_SPLITS;
    Problem P{q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale};
    bool empty = false;
    const int st = validate(P, &empty);
    if (st != ATTN_OK || empty) return st;
    // the default: the best split count whose partials fit the buffer
    if (num_splits == 0)
        num_splits = splitkv_default(B, Hq, N, D, causal,
                                     static_cast<int64_t>(kNoAllocScratchBytes));
    int split_tiles = 0, n_splits = 0;
    split_layout(P.n_tiles, num_splits, &split_tiles, &n_splits);
    if (D > 128) n_splits = 1;
    if (n_splits > 1 && workspace_bytes_for(P.bh, N, D, n_splits) >
                            static_cast<int64_t>(kNoAllocScratchBytes))
        return ATTN_ERR_SCRATCH;  // checked before anything touches the device
    void* scratch = nullptr;
    const int sa = scratch_address(&scratch);
    if (sa != ATTN_OK) return sa;
    // The split kernel writes every partial the merge reads, so nothing has to start at zero.
    return attn_fwd_splitkv(q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale, num_splits,
                            scratch, kNoAllocScratchBytes, stream);
}
