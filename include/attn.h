/*
 * attn.h - C ABI of the GB300 (sm_103a) exact-attention forward library (libgb300attn.so).
 *
 * The operation.  For Q [B, Hq, N, D] and K, V [B, Hkv, N, D] (bf16), every query row i of head
 * (b, hq) gets
 *     O[b,hq,i,:]  = sum_{j in J(i)} softmax_j(sm_scale * Q[b,hq,i,:] . K[b,hkv,j,:]) V[b,hkv,j,:]
 *     LSE[b,hq,i]  = ln sum_{j in J(i)} exp(sm_scale * Q[b,hq,i,:] . K[b,hkv,j,:])
 * with hkv = hq * Hkv / Hq (integer division) and J(i) = {0..i} under the causal mask (top-left
 * aligned, key j visible to query i iff j <= i), else {0..N-1}.
 * Sources: "Attention Kernel 实现与正确性验证" (walkerchi.com), section 1.1 (tiling + online softmax,
 * the score matrix never written to memory) and section 1.2 (the GQA-aware forward kernel and its
 * causal condition); "Triton-CUDA Attention" (skillmd.com), the standard forward with its
 * (B, H, L, D) contiguous layout and sm_scale = 1/sqrt(D), and the GQA/MQA variants (heads map by
 * integer division, grid over the query heads); "Flash Attention 与 Kernel 优化"
 * (fangpin.github.io), the interface section (inputs already projected, no RoPE inside) and the
 * saved per-row log-sum-exp statistic.
 *
 * Ownership.  Every tensor pointer is a DEVICE pointer (cudaMalloc / cudaMallocManaged memory of the
 * current device), owned by the caller.  The library never allocates, frees or retains them, and
 * allocates no device memory of its own per call.
 *
 * Errors.  Argument validation happens before anything is launched; on any validation failure the
 * call returns a negative attn_status_t and writes nothing.  Kernel execution is asynchronous on
 * `stream`: a return of ATTN_OK means "enqueued".  Device-side bounded waits that expire (which a
 * correct build never hits) are recorded in a device status word read by attn_debug_status().
 *
 * Thread safety.  Calls from several host threads are safe; the only mutable host state is the
 * per-thread last CUDA error.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = -1,     /* a required pointer is NULL */
    ATTN_ERR_SHAPE = -2,    /* B, Hq, Hkv or N negative, Hq or Hkv zero, or sizes overflow */
    ATTN_ERR_HEADS = -3,    /* Hq is not a multiple of Hkv */
    ATTN_ERR_HEADDIM = -4,  /* D not a multiple of 8 in [8, 256] ([8, 128] for the backward) */
    ATTN_ERR_ALIGN = -5,    /* a tensor pointer is not 16-byte aligned */
    ATTN_ERR_SCALE = -6,    /* sm_scale is not finite and positive */
    ATTN_ERR_ARCH = -7,     /* the device is not sm_103, its shared memory is misaligned, or the
                               library was built with an unexpected register count */
    ATTN_ERR_CUDA = -8,     /* a CUDA runtime/driver call failed; see attn_last_cuda_error() */
    ATTN_ERR_TIMEOUT = -9,  /* a device-side bounded wait expired (reported by attn_debug_status) */
    ATTN_ERR_MEMORY = -10,  /* a pointer is not device memory of the current device */
    ATTN_ERR_ALIAS = -11,   /* out, lse or the workspace overlaps q, k, v or each other */
    ATTN_ERR_SPLITS = -12,  /* num_splits outside [0, 64] */
    ATTN_ERR_WORKSPACE = -13, /* workspace smaller than attn_fwd_splitkv_workspace_bytes() */
    ATTN_ERR_SCRATCH = -14, /* attn_fwd_splitkv_noalloc: more scratch needed than it has */
    ATTN_ERR_STRIDE = -15,  /* attn_fwd_strided: a stride is not usable by the TMA */
    ATTN_ERR_RANGE = -16    /* debug build only: an index check failed (reported by
                               attn_debug_status; the access was skipped) */
} attn_status_t;

/*
 * attn_fwd - fused exact-attention forward (tiled, online softmax, O and LSE).
 *
 *   q        bf16 [B, Hq,  N, D], contiguous (row-major, D innermost)
 *   k        bf16 [B, Hkv, N, D], contiguous
 *   v        bf16 [B, Hkv, N, D], contiguous
 *   out      bf16 [B, Hq,  N, D], contiguous; written (round-to-nearest-even); must not overlap
 *            q, k, v or lse
 *   lse      fp32 [B, Hq, N]; written with the natural-log LSE of the scaled, masked scores
 *   B, Hq, Hkv, N, D   sizes; Hq % Hkv == 0 (MQA is Hkv == 1); D a multiple of 8 in [8, 256]
 *            (computed on D padded to 64, 128 or 256 with zeros, as "Triton-CUDA Attention" pads
 *            D to a power of two; the padding is never read from or written to memory; D > 128
 *            runs a one-Q-tile-per-CTA kernel, since its output fills the tensor memory);
 *            B == 0 or N == 0 is a valid empty problem (returns ATTN_OK, launches nothing; the pointers may then
 *            be NULL, as zero-size allocations often are)
 *   causal   0: every key visible; nonzero: key j visible to query i iff j <= i
 *   sm_scale score scale (callers usually pass 1/sqrt(D)); finite and > 0
 *   stream   a cudaStream_t of the current device, passed as void* (NULL = legacy default stream)
 *
 * Returns ATTN_OK once its kernels are enqueued on `stream`, else a negative attn_status_t.
 *
 * Scheduling: up to D = 128 the kernel is persistent (one CTA per SM); a work item is a pair of
 * 128-row Q tiles of one head, or a single Q tile when pairs would leave more than half of the
 * SMs idle (the results are the same bits either way).  When the Q tiles leave SMs idle and the
 * key axis is long, attn_fwd splits the key axis instead, as attn_fwd_splitkv describes
 * (attn_fwd_num_splits() says how many ways; the result then differs from the single pass by
 * rounding only): the splits of each pair of Q tiles either run as a thread-block cluster whose
 * CTAs merge through distributed shared memory, or the persistent split kernel writes its
 * partials to one of two 64 MiB slots of a device buffer compiled into the library and a merge
 * kernel follows.  A slot is leased to one launch at a time (a later launch's stream waits for
 * the slot's previous launch, as for the claim counters below), so overlapping calls stay
 * correct; while the stream is being captured into a CUDA graph only the cluster form is used.  The persistent kernels' CTAs claim work items
 * from a device counter that the library hands to each launch from a pool of 64 (round robin,
 * per device, shared with attn_fwd_strided, the split-KV entry points and the backward's dQ
 * kernel).  Each launch returns its counter to zero, and before a launch reuses a counter its
 * stream waits (cudaStreamWaitEvent) for the counter's previous launch to finish, so any number
 * of launches from any streams or host threads may overlap.  A launch made while its stream is
 * being captured into a CUDA graph takes no counter: its CTAs follow a static schedule instead
 * (a few per cent slower on long causal problems), so graphs may replay on any streams, also
 * concurrently with each other.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int N, int D, int causal, float sm_scale, void* stream);

/* Key-axis splits attn_fwd uses for these sizes on the current device (outside a graph
 * capture): 1 (single pass) unless the cost model of attn_fwd_splitkv_num_splits(), limited to
 * workspaces of one 64 MiB scratch slot, gives a split a margin of at least 1 us; also 1 for
 * invalid sizes. */
int attn_fwd_num_splits(int B, int Hq, int N, int D, int causal);

/* attn_fwd_test_split_choice - test hook: the split count the library's cost model picks for
 * these sizes on a device described by the arguments, touching no device: num_sms SMs and
 * cluster_fit[0..2] clusters of 2, 3 and 4 split CTAs fitting on it at once.  cluster_only != 0
 * gives the choice among splits that merge inside clusters only (attn_fwd's while its stream is
 * captured), else the choice among the counts whose workspace is at most
 * max_ws bytes (attn_fwd's with 64 MiB, attn_fwd_splitkv_num_splits's with LLONG_MAX; uncached).
 * Returns the count, or ATTN_ERR_SHAPE for invalid arguments. */
int attn_fwd_test_split_choice(int B, int Hq, int N, int D, int causal, int num_sms,
                               const int* cluster_fit, int cluster_only, long long max_ws);

/*
 * attn_fwd_strided - attn_fwd for tensors that are not contiguous, e.g. the [B, N, H, D] layout
 * that projections usually produce.  "Triton-CUDA Attention" (skillmd.com) asks callers to
 * transpose and make such inputs contiguous first (its common-errors table); here the TMA tensor
 * maps take the strides directly, so no copy is needed.
 *
 *   q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale, stream: as for attn_fwd, except that
 *     q, k, v and out are [B, H, N, D] tensors addressed through strides (D still contiguous);
 *     lse is contiguous [B, Hq, N].
 *   q_strides, k_strides, v_strides, o_strides: host arrays of 3 element strides each,
 *     {batch, head, row}; each must be a positive multiple of 8 elements (16 bytes) below 2^39,
 *     else ATTN_ERR_STRIDE.  A contiguous tensor has {H*N*D, N*D, D}; a [B, N, H, D] one has
 *     {N*H*D, D, H*D}.  out must not overlap any input (checked over each tensor's byte span).
 */
int attn_fwd_strided(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int Hq, int Hkv, int N, int D, int causal, float sm_scale,
                     const long long* q_strides, const long long* k_strides,
                     const long long* v_strides, const long long* o_strides, void* stream);

/*
 * attn_fwd_splitkv - the same forward, with the key axis of every query tile cut into splits.
 *
 * The split-T pattern of "Attention Kernel 实现与正确性验证" (walkerchi.com), section 2.4: each
 * split of the key axis produces a partial result (here: O over that split's keys, normalised by
 * that split's own denominator, in fp32, and that split's natural-log LSE), and a safe-softmax
 * merge combines them: LSE = M + ln sum_s exp(LSE_s - M) with M = max_s LSE_s, and
 * O = sum_s exp(LSE_s - LSE) O_s.  With 2-4 splits whose clusters all fit on the device at once
 * (one wave), the splits of each work item run as a thread-block cluster and merge through
 * distributed shared memory at the end of the kernel; otherwise the persistent split kernel
 * writes the partials to `workspace` and a merge kernel follows on the same stream (its dynamic
 * claims balance uneven causal splits over several waves).  This raises the number of CTAs for
 * problems whose query tiles alone do not fill the GPU (short sequences, few heads); the result
 * equals attn_fwd's up to rounding.
 *
 *   q, k, v, out, lse, B, Hq, Hkv, N, D, causal, sm_scale, stream: as for attn_fwd.
 *   num_splits       requested number of key-axis splits, 0..64; 0 picks
 *                    attn_fwd_splitkv_num_splits().  Splits hold ceil(ceil(N/128)/num_splits)
 *                    key tiles of 128, so fewer splits may be used.  One split is
 *                    attn_fwd's single pass (never split further);
 *                    D > 128 always runs as one split (the wide-head kernel has no split form).
 *   workspace        device memory of at least attn_fwd_splitkv_workspace_bytes(B, Hq, N, D,
 *                    num_splits) bytes, 16-byte aligned, owned by the caller; its previous
 *                    contents are ignored and it holds partial results afterwards (it is
 *                    checked, but left untouched, when the splits merge inside clusters).  It
 *                    must not overlap the inputs or outputs, and calls that run concurrently on
 *                    the GPU must not share it.  May be NULL when the call resolves to one split.
 *   workspace_bytes  size of `workspace` in bytes.
 *
 * Returns ATTN_OK once its kernels are enqueued, else a negative attn_status_t (nothing written).
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int Hq, int Hkv, int N, int D, int causal, float sm_scale, int num_splits,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes attn_fwd_splitkv needs for these sizes (0 if the call resolves to one split or
 * the sizes are invalid).  num_splits == 0: enough for attn_fwd_splitkv_num_splits()'s count,
 * with or without the causal mask (the larger of the two). */
size_t attn_fwd_splitkv_workspace_bytes(int B, int Hq, int N, int D, int num_splits);

/* Suggested split count for the current device (attn_fwd_splitkv's default): the count, from 1
 * (single pass) to 16, with the lowest estimated time under a cost model calibrated on GB300
 * (launch, per-unit and per-key-tile costs; the heaviest-first claim order simulated as list
 * scheduling over the SMs; the workspace path's partial traffic, or the cluster path's in-cluster
 * merge).  A split must win by 1 us; problems with at least twice as many Q-tile pairs as SMs are
 * not split.  The result is cached per shape (its first evaluation takes up to a few ms). */
int attn_fwd_splitkv_num_splits(int B, int Hq, int N, int D, int causal);

/*
 * attn_fwd_splitkv_noalloc - attn_fwd_splitkv for callers that cannot allocate device memory.
 *
 * No counterpart in the pages: this is a convenience of this library.  Some callers cannot hand
 * us a workspace because they may not allocate device memory at call time (a plug-in whose host
 * application owns the whole device-memory budget, or a serving loop that forbids allocation
 * after start-up).  This entry point keeps the split partials in a fixed device buffer compiled
 * into the library (attn_fwd_splitkv_noalloc_max_bytes() bytes, held on every GPU that loads the
 * library until the process exits) and calls no allocator of any kind.
 *
 *   Arguments, outputs and result: as attn_fwd_splitkv, without the workspace arguments.
 *   A problem whose partials need more than the buffer holds (attn_fwd_splitkv_workspace_bytes()
 *   > attn_fwd_splitkv_noalloc_max_bytes()) returns ATTN_ERR_SCRATCH before any launch.  With an
 *   explicit num_splits the check runs before any CUDA call.  With num_splits = 0 the default is
 *   the split count attn_fwd_splitkv_num_splits() would choose among those whose partials fit
 *   the buffer (the choice needs the device's SM count: the same one-time device query every
 *   entry point makes), so it never returns ATTN_ERR_SCRATCH.
 *   The buffer's device address is looked up the first time this is called on a device (with that
 *   device current); make that first call before capturing any stream.  A lookup that fails is
 *   not remembered: the next call on that device tries again.
 *   All calls share the one buffer, and it keeps the last call's partials (nothing in it needs to
 *   start at zero).  Calls that overlap on the GPU - on different streams, or from several host
 *   threads without ordering - race on it and may return wrong results; serialise them.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                             int B, int Hq, int Hkv, int N, int D, int causal, float sm_scale,
                             int num_splits, void* stream);

/* Size in bytes of the fixed buffer attn_fwd_splitkv_noalloc uses. */
size_t attn_fwd_splitkv_noalloc_max_bytes(void);

/* Static, human-readable text for an attn_status_t value (never NULL). */
const char* attn_status_string(int status);

/* The cudaError_t behind this thread's most recent ATTN_ERR_CUDA (0 if none). */
int attn_last_cuda_error(void);

/*
 * attn_debug_status - synchronise `stream`, then read and clear the device status word.
 * Returns ATTN_OK if no kernel of this library recorded a failure since the last call,
 * ATTN_ERR_TIMEOUT if a device-side bounded wait expired, ATTN_ERR_RANGE if (in the debug build,
 * compiled with ATTN_DEBUG) a kernel's index check failed, ATTN_ERR_ARCH if a kernel found its
 * dynamic shared memory not 1024-byte aligned (it then did no work), or ATTN_ERR_CUDA if the
 * synchronisation itself failed.  The status word is shared by all streams of the device.
 * The debug build checks, before each store whose address it computes, that the indices behind
 * it are in range (the decoded work item: batch, heads, tiles, split; rows of O, LSE, dQ, Delta
 * and the split partials); a failed check records ATTN_ERR_RANGE and skips the store.  It stands
 * in for a memory checker: it never traps.
 */
int attn_debug_status(void* stream);

/*
 * attn_bwd - gradients of attn_fwd by recompute (no stored probability matrix).
 *
 * The pages train through this attention by recomputing the scores and the probabilities from
 * the saved log-sum-exp ("Attention Kernel 实现与正确性验证" (walkerchi.com), section 1.1, the third
 * FA-2 idea; "Flash Attention 与 Kernel 优化" (fangpin.github.io), autograd and backward: rebuild
 * s = qk^T * scale, the causal mask and p = softmax(s), then dv, dp, ds, dq, dk).  For query row
 * i and visible key j: p_ij = exp(sm_scale q_i.k_j - LSE_i), dp_ij = dO_i.v_j,
 * ds_ij = p_ij (dp_ij - dO_i.O_i); dQ_i = sm_scale sum_j ds_ij k_j, dK_j = sm_scale sum ds_ij q_i
 * and dV_j = sum p_ij dO_i, the last two summed over the query heads that share the KV head.
 *
 *   q, k, v, B, Hq, Hkv, N, D, causal, sm_scale: as passed to attn_fwd (contiguous); D at most
 *                128 here (ATTN_ERR_HEADDIM above).
 *   out, lse     attn_fwd's outputs O [B,Hq,N,D] bf16 and LSE [B,Hq,N] fp32 (inputs here).
 *   dout         dL/dO, bf16 [B, Hq, N, D], contiguous.
 *   dq           bf16 [B, Hq, N, D]; dk, dv bf16 [B, Hkv, N, D]: written (contiguous).
 *   workspace    device memory of at least attn_bwd_workspace_bytes(B, Hq, N) bytes, 16-byte
 *                aligned, owned by the caller (holds dO . O per row); contents ignored.
 *   No output may overlap an input or another output.  Three kernels run on `stream`.
 *
 * Returns ATTN_OK once enqueued, else a negative attn_status_t (nothing written).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int D,
             int causal, float sm_scale, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes attn_bwd needs (B * Hq * N * 4; 0 for invalid sizes). */
size_t attn_bwd_workspace_bytes(int B, int Hq, int N);

/*
 * attn_mla_decode - absorbed multi-head latent attention (MLA), one decode query per head.
 *
 * "Attention Kernel 实现与正确性验证" (walkerchi.com), section 2.1: W_uk is folded into the query
 * (q_abs = q_nope W_uk), so the scores are taken in the compressed space against the cached c_kv
 * plus the decoupled RoPE key k_pe, and no K or V is rebuilt; section 2.2 gives the reference
 * (softmax over all cached tokens, no mask, output c_kv-weighted, then W_uv); section 2.4 splits
 * the token axis (split-T) and merges with a safe softmax.  For batch b, head h, token t:
 *   s_t = sm_scale * (q[b,h,0:d_c] . kv[b,t,0:d_c] + q[b,h,d_c:] . kv[b,t,d_c:])
 *   out[b,h,:] = sum_t softmax_t(s) kv[b,t,0:d_c]        lse[b,h] = ln sum_t exp(s_t)
 * The query absorption and the up-projection out W_uv^T are the caller's matrix products, like
 * the projections around attn_fwd.
 *
 *   q         bf16 [B, H, d_c + d_r] contiguous: q_abs then q_pe per head.
 *   kv        bf16 [B, T, d_c + d_r] contiguous: c_kv then k_pe per cached token (all heads).
 *   out       bf16 [B, H, d_c] contiguous (written, compressed space).
 *   lse       fp32 [B, H] (written, natural log).
 *   d_c, d_r  must be 512 and 64 (the page's DeepSeek-V3 widths), else ATTN_ERR_HEADDIM.
 *   sm_scale  finite, > 0; the un-absorbed head width sets it (1/sqrt(d_nope + d_r)).
 *   num_splits  token-axis splits in [0, 64]; 0 picks attn_mla_decode_num_splits(B, H, T).
 *               Clamped to the number of 64-token tiles.  With one split the workspace is unused.
 *   workspace   device memory, 16-byte aligned, of at least
 *               attn_mla_decode_workspace_bytes(B, H, T, num_splits) bytes when that is nonzero
 *               (per-split fp32 partials and LSEs, needed above 4 splits); owned by the
 *               caller, contents ignored.
 *   T >= 1 and H >= 1; B == 0 is a no-op.  Outputs, inputs and the workspace must not overlap.
 *   Pointers are device pointers of the current device, owned by the caller.
 *
 * Returns ATTN_OK once enqueued, else a negative attn_status_t and nothing is written.  One
 * kernel runs; with 2-4 splits the split CTAs of each (batch, 128-head tile, value half) form a
 * thread-block cluster and merge through distributed shared memory; with more splits the
 * partials go to the workspace and a merge kernel follows.  Device-side wait expiries go to
 * attn_debug_status.
 */
int attn_mla_decode(const void* q, const void* kv, void* out, float* lse, int B, int H, int T,
                    int d_c, int d_r, float sm_scale, int num_splits, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Split count attn_mla_decode picks for num_splits == 0 (1 for invalid sizes). */
int attn_mla_decode_num_splits(int B, int H, int T);

/* Workspace bytes attn_mla_decode needs for `num_splits` (0 = its own choice); 0 if none. */
size_t attn_mla_decode_workspace_bytes(int B, int H, int T, int num_splits);

/*
 * attn_fwd_test_stall - test hook for the failure-reporting path (not for computing anything).
 *
 * Runs attn_fwd, except that every CTA's producer withholds item `stall_item` (>= 0) of its K/V
 * load ring (item 2j is K tile j, 2j+1 is V tile j, counted from the CTA's first tile), so the
 * bounded waits on it expire after about one second.  The CTA then stops all its roles, frees its
 * tensor memory and returns; out and lse hold garbage, the device status word records the
 * expiry (attn_debug_status returns ATTN_ERR_TIMEOUT) and the CUDA context stays usable.  An
 * item past the CTA's last one stalls nothing.  Use tiny problems: each CTA waits ~1 s.
 */
int attn_fwd_test_stall(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                        int Hq, int Hkv, int N, int D, int causal, float sm_scale, int stall_item,
                        void* stream);

/*
 * attn_fwd_test_kernel - test and benchmark hook: attn_fwd on a chosen forward kernel.
 *
 * Runs the problem (arguments as attn_fwd, contiguous tensors) on the kernel named by `kernel`,
 * so that tests can check each kernel on any shape and benchmarks can time them side by side:
 *   kernel = 1  the one-CTA kernel, two 128-row Q tiles per work item (D <= 128), the kernel
 *               attn_fwd runs up to D = 128;
 *   kernel = 2  the CTA-pair kernel: a cluster of two CTAs on two SMs shares every tcgen05 MMA
 *               (cta_group::2, M = 256), each SM loading and reading half of every K and V tile;
 *               four Q tiles per work item (64 < D <= 128; ATTN_ERR_HEADDIM otherwise,
 *               ATTN_ERR_ARCH if no CTA pair fits on the device).  Measured slower than kernel 1
 *               on GB300, so attn_fwd does not use it;
 *   kernel = 3  the one-CTA kernel over two key-axis splits whose CTA pairs are clusters that
 *               merge through distributed shared memory (D <= 128; ATTN_ERR_SHAPE unless the
 *               key axis has at least two tiles and all the clusters fit on the device at once).
 * stall_item: -1, or a K/V ring entry to withhold as in attn_fwd_test_stall (on CTA pairs both
 * CTAs withhold their halves of it; in split clusters every CTA withholds it, and no cluster
 * merges).
 * The results are those of attn_fwd (the same definition; fp32 accumulation may group the work
 * differently).  Any other value of `kernel` returns ATTN_ERR_SHAPE.
 */
int attn_fwd_test_kernel(const void* q, const void* k, const void* v, void* out, float* lse,
                         int B, int Hq, int Hkv, int N, int D, int causal, float sm_scale,
                         int kernel, int stall_item, void* stream);

/*
 * attn_mla_decode_test_stall - the same test hook for attn_mla_decode (arguments as there).
 *
 * The producer of every CTA whose token range holds 64-token tile `stall_tile` (>= 0) withholds
 * that tile's cache panels, so those CTAs' bounded waits expire after about one second and they
 * stop, free their tensor memory and return.  A cluster with such a CTA is not merged: out and
 * lse hold garbage there, the status word records the expiry, and the next call computes
 * correctly.  Use tiny problems.
 */
int attn_mla_decode_test_stall(const void* q, const void* kv, void* out, float* lse, int B, int H,
                               int T, int d_c, int d_r, float sm_scale, int num_splits,
                               void* workspace, size_t workspace_bytes, int stall_tile,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
