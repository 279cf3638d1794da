// attn_api.cu - C ABI of the GB300 exact-attention forward (validation, TMA descriptors, launch).
//
// Interface follows the problem statement of the pages: inputs Q [B,Hq,N,D], K/V [B,Hkv,N,D]
// contiguous bf16 ("Triton-CUDA Attention", skillmd.com: (B, H, L, D) layout, contiguous inputs,
// GQA grid over the query heads), a causal flag ("Flash Attention 与 Kernel 优化",
// fangpin.github.io: FlashAttention.apply(q, k, v, is_causal)), outputs O and the per-row LSE.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "attn_fwd_kernel.cuh"

using namespace gb300attn;

// Device status word: kernels OR failure flags into it (see attn_debug_status).
__device__ unsigned int g_attn_status_word = 0;

namespace {

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

// 3-D view [BH, N, D] of a contiguous bf16 tensor; box = 64 (D) x 128 (rows) x 1, 128B swizzle.
// Rows >= N of a head are out of bounds: zero-filled on load, dropped on store.
bool make_tile_map(CUtensorMap* map, const void* base, int64_t BH, int64_t N, int64_t D) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2),
                                   static_cast<cuuint64_t>(N * D * 2)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBM), 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Per-device one-time set-up: architecture check, status-word address, smem opt-in.
constexpr int kMaxDevices = 64;
struct DeviceState {
    std::once_flag once;
    int status = ATTN_OK;
    int cuda_error = 0;
    unsigned int* status_word = nullptr;
};
DeviceState g_devices[kMaxDevices];

int device_state(int dev, DeviceState** out) {
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    DeviceState& st = g_devices[dev];
    std::call_once(st.once, [&st, dev] {
        int major = 0, minor = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) { st.status = ATTN_ERR_CUDA; st.cuda_error = e; return; }
        if (major != 10 || minor != 3) { st.status = ATTN_ERR_ARCH; return; }
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status_word), g_attn_status_word);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_fwd_kernel<64>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SmemLayout<64>::kAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_fwd_kernel<128>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SmemLayout<128>::kAlloc);
        if (e != cudaSuccess) { st.status = ATTN_ERR_CUDA; st.cuda_error = e; }
    });
    if (st.status == ATTN_ERR_CUDA) t_last_cuda_error = st.cuda_error;
    *out = &st;
    return st.status;
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

template <int D>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
           const CUtensorMap& mo, const AttnParams& p, unsigned int* status_word, int64_t grid,
           cudaStream_t stream) {
    attn_fwd_kernel<D><<<static_cast<unsigned int>(grid), kThreads, SmemLayout<D>::kAlloc,
                         stream>>>(mq, mk, mv, mo, p, status_word);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                        int Hq, int Hkv, int N, int D, int causal, float sm_scale, void* stream) {
    // ---- host-side validation: nothing is launched or written on failure ---------------------
    if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0) return ATTN_ERR_SHAPE;
    if (Hq % Hkv != 0) return ATTN_ERR_HEADS;
    if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
    if (!std::isfinite(sm_scale) || !(sm_scale > 0.f)) return ATTN_ERR_SCALE;
    if (B == 0 || N == 0) return ATTN_OK;  // empty problem: nothing to read or write
    if (!q || !k || !v || !out || !lse) return ATTN_ERR_NULL;
    const uintptr_t align_bits = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                                 reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out) |
                                 reinterpret_cast<uintptr_t>(lse);
    if (align_bits & 15u) return ATTN_ERR_ALIGN;

    const int64_t bh = static_cast<int64_t>(B) * Hq;
    const int64_t bh_kv = static_cast<int64_t>(B) * Hkv;
    const int64_t n_tiles = (static_cast<int64_t>(N) + kBM - 1) / kBM;
    const int64_t n_pairs = (n_tiles + 1) / 2;
    const int64_t grid = n_pairs * bh;
    if (grid > 0x7fffffffLL || bh > 0x7fffffffLL) return ATTN_ERR_SHAPE;

    const int64_t q_bytes = bh * N * D * 2, kv_bytes = bh_kv * N * D * 2, lse_bytes = bh * N * 4;
    if (overlaps(out, q_bytes, q, q_bytes) || overlaps(out, q_bytes, k, kv_bytes) ||
        overlaps(out, q_bytes, v, kv_bytes) || overlaps(out, q_bytes, lse, lse_bytes) ||
        overlaps(lse, lse_bytes, q, q_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
        overlaps(lse, lse_bytes, v, kv_bytes))
        return ATTN_ERR_ALIAS;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceState* ds = nullptr;
    const int st = device_state(dev, &ds);
    if (st != ATTN_OK) return st;
    for (const void* ptr : {q, k, v, static_cast<const void*>(out), static_cast<const void*>(lse)})
        if (check_memory(ptr, dev) != ATTN_OK) return ATTN_ERR_MEMORY;

    // ---- TMA descriptors (passed by value as __grid_constant__ kernel parameters) -------------
    CUtensorMap mq, mk, mv, mo;
    if (!make_tile_map(&mq, q, bh, N, D) || !make_tile_map(&mk, k, bh_kv, N, D) ||
        !make_tile_map(&mv, v, bh_kv, N, D) || !make_tile_map(&mo, out, bh, N, D))
        return cuda_fail(cudaErrorInvalidValue);

    AttnParams p;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.N = N;
    p.group = Hq / Hkv;
    p.causal = causal ? 1 : 0;
    p.n_tiles = static_cast<int>(n_tiles);
    p.n_pairs = static_cast<int>(n_pairs);
    p.scale_log2 = sm_scale * 1.4426950408889634f;  // log2(e)
    p.lse = lse;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return D == 64 ? launch<64>(mq, mk, mv, mo, p, ds->status_word, grid, s)
                   : launch<128>(mq, mk, mv, mo, p, ds->status_word, grid, s);
}

extern "C" const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL: return "a required pointer is NULL";
        case ATTN_ERR_SHAPE: return "invalid or overflowing shape (B, Hq, Hkv, N)";
        case ATTN_ERR_HEADS: return "Hq is not a multiple of Hkv";
        case ATTN_ERR_HEADDIM: return "unsupported head dimension (D must be 64 or 128)";
        case ATTN_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
        case ATTN_ERR_SCALE: return "sm_scale must be finite and positive";
        case ATTN_ERR_ARCH: return "the current device is not sm_103 (GB300)";
        case ATTN_ERR_CUDA: return "a CUDA call failed (see attn_last_cuda_error)";
        case ATTN_ERR_TIMEOUT: return "a device-side bounded wait expired";
        case ATTN_ERR_MEMORY: return "a pointer is not device memory of the current device";
        case ATTN_ERR_ALIAS: return "out/lse overlap an input or each other";
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
    return (word & kDevTimeout) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}
