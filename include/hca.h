/*
 * hca.h -- C ABI of libhca: DeepSeek-V4 Heavily Compressed Attention (HCA),
 * forward and backward, on NVIDIA GB300 (sm_103a).
 *
 * The operation.  Single-KV-head (MQA) attention in which the one shared kv
 * tensor is both key and value ("[DeepSeek-V4] Implement Compressed Attention
 * Layers", review suggestions on the logits and output einsums: k = v = kv,
 * broadcast over the query heads).  Query position i of batch row b attends,
 * under one softmax, to
 *   - the raw kv rows t with i-W < t <= i (causal sliding window), and
 *   - the compressed entries ckv[j] whose length-m window [j*m, (j+1)*m-1]
 *     has completed, (j+1)*m <= i+1,
 * ("Add HCA Static Compilation for Splash Attention [Deepseek v4]",
 * Description: the HCA pattern is the local sliding window plus the completed
 * earlier compression windows), restricted to keys of the query's own packed
 * document: raw rows with the same segment id, compressed entries whose whole
 * window carries that id (same page, packing and segment-id bullet; "DSV4:
 * Route compressed and sliding train attention onto the splash kernels",
 * segment-mask review suggestion).  Sequence lengths need not be multiples of
 * any tile size (same page, unaligned-length bullet).  No mask tensor is ever
 * written: visibility is computed from coordinates inside the kernels.
 *
 * Conventions shared by every entry point.
 *   Layout   q, out, dq, dout: [B,H,S,D]; kv, dkv: [B,S,D];
 *            ckv, dckv: [B,Sc,D] with Sc = ceil(S/m); seg: [B,S] int32;
 *            lse: [B,H,S] fp32.  All contiguous, row-major.
 *   dtype    HCA_BF16: q/kv/ckv/out/dout/dq/dkv/dckv are bfloat16, the
 *            arithmetic is bf16 tensor-core products with fp32 accumulation
 *            and fp32 softmax; D = 64 or 128 (other D: HCA_ERR_UNSUPPORTED).
 *            HCA_F32: everything fp32, fp32 arithmetic, any D.
 *            lse is fp32 in both.
 *   seg      NULL means one segment per batch row.  Otherwise non-negative
 *            ids must be non-decreasing along S and negative ids (padding)
 *            must form a suffix of each row; padded positions are neither
 *            queries nor keys (out = 0, lse = -inf, dq = 0).  This ordering
 *            is checked on the device; a violation is reported through
 *            hca_workspace_status and the outputs of that call are NaN.
 *   Memory   Every pointer is a device pointer owned by the caller.  Tensor
 *            base pointers must be 16-byte aligned and D * element size must
 *            be a multiple of 16 bytes.  The library allocates and frees
 *            nothing; scratch comes from the caller's workspace (at least
 *            hca_workspace_size bytes, 256-byte aligned).
 *   Streams  Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *            default stream) and the call returns without synchronising.
 *   Errors   Every entry returns an hca_status.  Argument errors are
 *            detected on the host before anything is enqueued; launch
 *            failures return HCA_ERR_CUDA.  Nothing aborts the process.
 */
#ifndef HCA_H_
#define HCA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HCA_API __attribute__((visibility("default")))
#else
#define HCA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HCA_OK = 0,
  HCA_ERR_NULL = 1,        /* a required pointer is NULL                       */
  HCA_ERR_SHAPE = 2,       /* B, H, S or D out of range                        */
  HCA_ERR_DTYPE = 3,       /* unknown dtype code                               */
  HCA_ERR_ALIGN = 4,       /* pointer not 16-byte aligned, or D*elt % 16 != 0  */
  HCA_ERR_ARG = 5,         /* W < 1, m < 1, scale not finite, bad tile size    */
  HCA_ERR_SEG = 6,         /* segment ids out of order (device-side check)     */
  HCA_ERR_WORKSPACE = 7,   /* workspace NULL, misaligned or too small          */
  HCA_ERR_UNSUPPORTED = 8, /* no kernel for this dtype / D combination (bf16
                              runs on tensor cores only, for D = 64 or 128)  */
  HCA_ERR_CUDA = 9,        /* a CUDA runtime call or launch failed             */
  HCA_ERR_TIMEOUT = 10     /* a bounded on-device wait gave up                 */
} hca_status;

typedef enum { HCA_BF16 = 0, HCA_F32 = 1 } hca_dtype;

/* Human-readable name of a status code (static string, never NULL). */
HCA_API const char *hca_status_string(int status);

/* ABI version of this library (increases when an entry point changes). */
HCA_API int hca_version(void);

/* Bytes of caller-provided workspace that hca_attn_fwd (for_backward = 0)
 * or hca_attn_bwd (for_backward = 1) needs for these sizes; 0 when the
 * arguments are invalid.  Grows as O(B*S + B*H*S + Sc*D): never O(S^2). */
HCA_API size_t hca_workspace_size(int B, int H, int S, int D, int W, int m, int dtype, int for_backward);

/* Number of consecutive query positions the forward kernel packs into one
 * 128-row tile for H heads (the tile holds Pq positions of 128 / Pq heads,
 * the largest power of two dividing both H and 128), i.e. the Pq argument
 * that makes hca_tile_map describe the forward's own tiles; 1 for fp32. */
HCA_API int hca_query_tile_positions(int H, int D, int dtype);

/* Forward.  out[B,H,S,D] = softmax-weighted sum of the visible keys;
 * lse[B,H,S] = natural-log logsumexp of the scaled visible logits
 * (scale * <q, key>).  Cited passage: see the header comment.
 * Returns HCA_OK once the work is enqueued. */
HCA_API int hca_attn_fwd(const void *q, const void *kv, const void *ckv, const int32_t *seg,
                 void *out, float *lse,
                 int B, int H, int S, int D, int W, int m, float scale, int dtype,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Backward of hca_attn_fwd for the cotangent dout = dL/dout, given the
 * forward's out and lse.  dq[B,H,S,D]; dkv[B,S,D] and dckv[B,Sc,D] each sum
 * the key-role and the value-role gradient of the shared rows over every
 * head and visible query ("[DeepSeek-V4] Implement Compressed Attention
 * Layers": k and v are the same tensor).  dq, dkv and dckv are fully
 * overwritten. */
HCA_API int hca_attn_bwd(const void *q, const void *kv, const void *ckv, const int32_t *seg,
                 const void *out, const float *lse, const void *dout,
                 void *dq, void *dkv, void *dckv,
                 int B, int H, int S, int D, int W, int m, float scale, int dtype,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Visible (query, key) pairs per head of every batch row, from the same
 * interval arithmetic the attention kernels use: raw_pairs[B] over raw kv
 * rows and comp_pairs[B] over compressed entries (device int64 arrays,
 * overwritten).  Needs hca_workspace_size(B,1,S,16,W,m,HCA_F32,0) bytes. */
HCA_API int hca_visible_pairs(const int32_t *seg, int B, int S, int W, int m,
                      int64_t *raw_pairs, int64_t *comp_pairs,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Per query tile of Pq consecutive positions, the half-open key ranges the
 * kernels visit: map[B][ceil(S/Pq)][4] = {raw_lo, raw_hi, comp_lo, comp_hi}
 * (device int32, overwritten; 0,0 = no key of that kind).  Keys outside
 * these ranges are never loaded.  Same workspace as hca_visible_pairs. */
HCA_API int hca_tile_map(const int32_t *seg, int B, int S, int W, int m, int Pq, int32_t *map,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Synchronises `stream` and returns the status the device recorded in this
 * workspace during the last call that used it (HCA_OK, HCA_ERR_SEG or
 * HCA_ERR_TIMEOUT), or HCA_ERR_CUDA if the synchronisation failed.  This is
 * the one entry point that blocks the host. */
HCA_API int hca_workspace_status(const void *workspace, void *stream);

/* Local sliding-window attention (the LOCAL_SLIDING layers of "DSV4: Route
 * compressed and sliding train attention onto the splash kernels", local
 * sliding mask: window plus segment ids, no compressed set).  Query i
 * attends under one softmax to the raw kv rows t with i - W < t <= i of its
 * own document and to nothing else.  Arguments, layouts, ownership and
 * errors are those of hca_attn_fwd / hca_attn_bwd without ckv, dckv and m;
 * the same kernels run with the compressed set empty.  The workspace size
 * comes from hca_local_workspace_size (for_backward as in
 * hca_workspace_size); dq and dkv are fully overwritten. */
HCA_API size_t hca_local_workspace_size(int B, int H, int S, int D, int W, int dtype, int for_backward);
HCA_API int hca_local_attn_fwd(const void *q, const void *kv, const int32_t *seg, void *out, float *lse,
                               int B, int H, int S, int D, int W, float scale, int dtype,
                               void *workspace, size_t workspace_bytes, void *stream);
HCA_API int hca_local_attn_bwd(const void *q, const void *kv, const int32_t *seg,
                               const void *out, const float *lse, const void *dout, void *dq, void *dkv,
                               int B, int H, int S, int D, int W, float scale, int dtype,
                               void *workspace, size_t workspace_bytes, void *stream);

/* Forward for callers that cannot allocate device memory.  The paper has no
 * counterpart: this is a convenience of this library.  Plugin hooks of
 * inference runtimes, real-time loops that cannot afford cudaMalloc's implicit
 * synchronisation, and hosts without an allocator can call it with only their
 * inputs and outputs; arguments, layouts, outputs and errors are those of
 * hca_attn_fwd.  Its scratch is a fixed array inside the library (every GPU
 * that loads the library keeps it until exit, about 4 MB), which caps B * S at
 * HCA_NOALLOC_MAX_POSITIONS; larger problems return HCA_ERR_WORKSPACE before
 * anything is enqueued.  The first call on a device looks the array up (make
 * it before any stream capture).  All calls share the array: calls that
 * overlap on the GPU race and must be serialised by the caller.  A segment
 * ordering error poisons that call's outputs with NaN (there is no workspace
 * to read a status from).  A bounded on-device wait that gives up (see
 * HCA_ERR_TIMEOUT) leaves that call's outputs undefined, and this entry point
 * cannot report it: callers that need to detect it use hca_attn_fwd with a
 * workspace.  Nothing is allocated or freed. */
#define HCA_NOALLOC_MAX_POSITIONS (1 << 20)
HCA_API int hca_attn_fwd_noalloc(const void *q, const void *kv, const void *ckv, const int32_t *seg,
                                 void *out, float *lse,
                                 int B, int H, int S, int D, int W, int m, float scale, int dtype, void *stream);

/* Compressed sparse attention (CSA): HCA's two sets with the compressed
 * entries narrowed to a per-query selection ("Add HCA Static Compilation
 * for Splash Attention [Deepseek v4]", Description: CSA, compress ratio 4,
 * needs a top-k step and runtime indexer masks that keep or discard (query,
 * compressed entry) pairs; "DSV4: Route compressed and sliding train
 * attention onto the splash kernels", indexer-mask review).  Query i attends
 * under one softmax to its raw window (as hca_attn_fwd) and to the entries
 * j listed in sel[b,i,:] that hca_attn_fwd would let it see (window complete
 * at i, inside i's document).  Entries outside that set, repeats and
 * negative ids (padding) in sel are ignored, so sel can be the output of
 * hca_indexer_topk directly.
 *   sel   [B,S,k] int32 (device), k >= 1
 * Other arguments, layouts and outputs as hca_attn_fwd / hca_attn_bwd; dckv
 * rows of entries nobody selected are 0.  bf16 only, D = 128, H a multiple
 * of 32 and 2*Pq*k <= 32768 (Pq = hca_query_tile_positions); anything else
 * returns HCA_ERR_UNSUPPORTED.  Workspace: hca_csa_workspace_size bytes
 * (for_backward as in hca_workspace_size); 0 for unsupported sizes.  The
 * backward's dckv is summed with fp32 atomics (reproducible only up to
 * summation order); dq and dkv are deterministic. */
HCA_API size_t hca_csa_workspace_size(int B, int H, int S, int D, int W, int m, int k, int dtype, int for_backward);
HCA_API int hca_csa_attn_fwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const int32_t *sel,
                             void *out, float *lse, int B, int H, int S, int D, int W, int m, int k, float scale,
                             int dtype, void *workspace, size_t workspace_bytes, void *stream);
HCA_API int hca_csa_attn_bwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const int32_t *sel,
                             const void *out, const float *lse, const void *dout, void *dq, void *dkv, void *dckv,
                             int B, int H, int S, int D, int W, int m, int k, float scale, int dtype,
                             void *workspace, size_t workspace_bytes, void *stream);

/* HCA compressor: pooling of length-m windows of rows into compressed
 * entries ("[DeepSeek-V4] Implement Compressed Attention Layers",
 * Description: the compressors pool with a causal block bias; "Add HCA Static
 * Compilation for Splash Attention [Deepseek v4]": compressed entries are
 * the length-m windows).  For window j of batch row b and its positions
 * t = j*m + r (r < m) that exist and are not padding (seg >= 0):
 *   a = softmax_r(g[b,t] + bias[r]),   ckv[b,j,:] = sum_r a_r x[b,t,:];
 * a window with no such position gives a zero row.
 *   x     [B,S,D]  dtype (bf16 or fp32), D a multiple of 32, D <= 256
 *   g     [B,S]    fp32 gate logits;  bias [m] fp32 (offset in the block)
 *   seg   [B,S]    int32 or NULL (padding is skipped; documents are not:
 *                  a window that crosses documents is never visible to the
 *                  attention, whatever its value)
 *   ckv   [B,ceil(S/m),D] dtype, fully overwritten.
 * No workspace.  Errors as for hca_attn_fwd (HCA_ERR_UNSUPPORTED for D). */
HCA_API int hca_compress_fwd(const void *x, const float *g, const float *bias, const int32_t *seg, void *ckv,
                             int B, int S, int D, int m, int dtype, void *stream);

/* Backward of hca_compress_fwd for the cotangent dckv [B,ceil(S/m),D]:
 * dx [B,S,D] (dtype; 0 at padding), dg [B,S] fp32 (0 at padding), dbias [m]
 * fp32 (summed over every window in a fixed order, so run-to-run identical).
 * All three are fully overwritten.  Needs hca_compress_workspace_size(B,S,m)
 * bytes of workspace (one logit gradient per window position). */
HCA_API size_t hca_compress_workspace_size(int B, int S, int m);
HCA_API int hca_compress_bwd(const void *x, const float *g, const float *bias, const int32_t *seg,
                             const void *dckv, void *dx, float *dg, float *dbias,
                             int B, int S, int D, int m, int dtype,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Lightning Indexer with top-k selection, the step that feeds CSA
 * ("[DeepSeek-V4] Implement Compressed Attention Layers": the indexer's
 * per-head scores are the matmul of its queries with the transposed
 * compressed kv, and it masks with a sentinel; "Add HCA Static Compilation
 * for Splash Attention [Deepseek v4]", Description: CSA needs a top-k step).
 *   score[b,s,j] = sum_h w[b,s,h] <qi[b,s,h,:], ki[b,j,:]>   (bf16 inputs,
 *                  heads collapsed first in fp32, tensor-core products with
 *                  fp32 accumulation)
 * for the entries j that query s may see under the HCA compressed rule
 * (window complete at s, inside s's document); the others carry the
 * sentinel -inf and are never selected.  sel[b,s,:] receives the k entries
 * with the largest scores (ties: smaller index), in ascending entry order,
 * padded with -1 when fewer than k are visible.
 *   qi [B,S,Hi,Di] bf16, Di = 128;  ki [B,ceil(S/m),Di] bf16;  w [B,S,Hi] fp32
 *   seg [B,S] int32 or NULL;  sel [B,S,k] int32 (overwritten)
 *   scores [B,S,ceil(S/m)] fp32 or NULL: when given, every score with the
 *                  sentinel -inf outside the visible range (for checking)
 * ceil(S/m) must be at most 55296 and k at least 1.  Workspace:
 * hca_indexer_workspace_size(B,S,m) bytes (status word, document starts,
 * collapsed queries and a score buffer of at most 256 MB).  Segment ids out
 * of order are reported through hca_workspace_status (HCA_ERR_SEG) and that
 * call selects nothing (every entry of sel is -1). */
HCA_API size_t hca_indexer_workspace_size(int B, int S, int m);
HCA_API int hca_indexer_topk(const void *qi, const void *ki, const float *w, const int32_t *seg,
                             int32_t *sel, float *scores, int B, int S, int Hi, int Di, int m, int k,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Failure-path test hooks.  "Add HCA Static Compilation for Splash Attention
 * [Deepseek v4]" (Description, validation-guard bullet) wants unsupported or
 * failing cases reported as errors rather than crashes; the tests that check
 * this need failures on demand, and these hooks make them without faulting
 * the GPU.  `what` is one of
 *   HCA_INJECT_RESET          clear every injection below (value ignored);
 *   HCA_INJECT_LAUNCH_FAILURE the next `value` attention calls return
 *                             HCA_ERR_CUDA after checking their arguments and
 *                             before enqueuing anything;
 *   HCA_INJECT_STALL          in the next bf16 attention call, the kernels
 *                             named by the mask `value` (HCA_STALL_FWD,
 *                             HCA_STALL_DQ, HCA_STALL_DKV) start with their
 *                             MMA warp waiting on a barrier that nothing
 *                             arrives at: the wait gives up after the wait
 *                             limit, every CTA drains its own copies and
 *                             MMAs, frees its tensor memory and exits, later
 *                             kernels of the call see the error and poison
 *                             their outputs, and the call's workspace status
 *                             reads HCA_ERR_TIMEOUT;
 *   HCA_INJECT_WAIT_LIMIT_NS  limit of every bounded on-device wait, in ns,
 *                             for later launches (0 restores the default 2 s);
 *   HCA_INJECT_CSA_UNION      how later CSA calls build each query group's
 *                             union of selected entries: 0 picks the cheaper
 *                             of the two kernels (the default), 1 forces the
 *                             sorting kernel, a multiple of 64 up to 16384
 *                             forces the byte-mask kernel with chunks of that
 *                             many entries (so small cases reach its
 *                             several-chunk path).  Both give the same union.
 * The settings are process-wide.  Returns HCA_OK, or HCA_ERR_ARG for an
 * unknown `what`, a negative value or a value out of its range. */
#define HCA_INJECT_RESET 0
#define HCA_INJECT_LAUNCH_FAILURE 1
#define HCA_INJECT_STALL 2
#define HCA_INJECT_WAIT_LIMIT_NS 3
#define HCA_INJECT_CSA_UNION 4
#define HCA_STALL_FWD 1
#define HCA_STALL_DQ 2
#define HCA_STALL_DKV 4
HCA_API int hca_test_inject(int what, long long value);

/* Optional per-kernel timing.  hca_profile_enable(1) resets the counters and
 * makes every later kernel launch of the library record a pair of CUDA events
 * on its stream (0 stops recording).  hca_profile_read synchronises on the
 * recorded events and returns, for kernel id `kernel` (0 <= kernel <
 * hca_num_kernels()), the number of launches and their total device time in
 * milliseconds since the last enable.  hca_kernel_name gives the id's name. */
HCA_API int hca_profile_enable(int on);
HCA_API int hca_profile_read(int kernel, long long *launches, double *total_ms);
HCA_API int hca_num_kernels(void);
HCA_API const char *hca_kernel_name(int kernel);

#ifdef __cplusplus
}
#endif

#endif /* HCA_H_ */
