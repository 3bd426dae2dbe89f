// hca_api.cu -- the exported C ABI of libhca (see include/hca.h): argument
// validation, workspace carving and kernel dispatch.  Everything is enqueued
// on the caller's stream; nothing here allocates or synchronises except
// hca_workspace_status, whose job is to synchronise.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "hca_common.cuh"
#include "hca_internal.h"

using namespace hca;

namespace {

constexpr int kMaxD = 256;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elt_bytes(int dtype) { return dtype == HCA_F32 ? 4 : 2; }

// Common checks of sizes and scalar arguments.
int check_dims(int B, int H, int S, int D, int W, int m, int dtype) {
  if (dtype != HCA_BF16 && dtype != HCA_F32) return HCA_ERR_DTYPE;
  if (B < 0 || H < 1 || S < 0 || D < 1 || D > kMaxD) return HCA_ERR_SHAPE;
  // every flat index of the largest tensor must fit in 63 bits and every
  // position index in 31 bits
  if ((double)B * H * (double)S * D > 9.0e18 || S > (1 << 30) || H > (1 << 20)) return HCA_ERR_SHAPE;
  if (W < 1 || m < 1) return HCA_ERR_ARG;
  if ((D * elt_bytes(dtype)) % 16 != 0) return HCA_ERR_ALIGN;
  return HCA_OK;
}

size_t fwd_ws_bytes(int B, int S) { return kHeaderBytes + align_up((size_t)B * S * sizeof(int32_t)); }

size_t bwd_ws_bytes(int B, int H, int S, int D, int W, int m, int dtype, bool csa = false) {
  size_t n = fwd_ws_bytes(B, S) + align_up((size_t)B * H * S * sizeof(float));
  n += tc_bwd_scratch_bytes(B, H, S, D, W, m, dtype, csa);
  return n;
}

// CSA workspace: the attention's, then the union of selections (per forward
// pair of 2*Pq positions, or per dq tile of Pq), then (backward) the fp32
// dckv accumulator.
int csa_pq(int H) { return tc_query_tile_positions(H); }
size_t csa_fwd_ws_bytes(int B, int H, int S, int k) { return fwd_ws_bytes(B, S) + csa_union_bytes(B, S, 2 * csa_pq(H), k); }
size_t csa_bwd_ws_bytes(int B, int H, int S, int D, int W, int m, int k) {
  return bwd_ws_bytes(B, H, S, D, W, m, HCA_BF16, true) + csa_union_bytes(B, S, csa_pq(H), k) +
         csa_dckv_acc_bytes(B, (S + m - 1) / m);
}

struct Carve {
  char *p;
  int32_t *status;
  int32_t *sstart;
};

Carve carve_fwd(void *ws, int B, int S) {
  Carve c;
  c.p = static_cast<char *>(ws);
  c.status = reinterpret_cast<int32_t *>(c.p);
  c.sstart = reinterpret_cast<int32_t *>(c.p + kHeaderBytes);
  return c;
}

int check_ws(void *ws, size_t have, size_t need) {
  if (need == 0) return HCA_OK;
  if (ws == nullptr) return HCA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return HCA_ERR_WORKSPACE;
  if (have < need) return HCA_ERR_WORKSPACE;
  return HCA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? HCA_OK : HCA_ERR_CUDA; }

// bf16 runs on the tensor-core kernels only; fp32 on the CUDA-core kernels
bool supported(int H, int D, int dtype) { return dtype == HCA_F32 || tc_fwd_supported(H, D, dtype); }

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<long long> g_inject_launch_failures{0};
std::atomic<int> g_inject_stall_mask{0};
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_csa_union{0};

bool take_counter(std::atomic<long long> &c) {
  long long v = c.load();
  while (v > 0)
    if (c.compare_exchange_weak(v, v - 1)) return true;
  return false;
}

}  // namespace

namespace hca {
bool take_launch_failure() { return take_counter(g_inject_launch_failures); }
int take_stall_mask() { return g_inject_stall_mask.exchange(0); }
uint64_t wait_limit_ns() { return g_wait_ns.load(); }
int csa_union_setting() { return g_csa_union.load(); }
}  // namespace hca

extern "C" {

const char *hca_status_string(int s) {
  switch (s) {
    case HCA_OK: return "HCA_OK";
    case HCA_ERR_NULL: return "HCA_ERR_NULL: a required pointer is NULL";
    case HCA_ERR_SHAPE: return "HCA_ERR_SHAPE: B, H, S or D out of range";
    case HCA_ERR_DTYPE: return "HCA_ERR_DTYPE: unknown dtype";
    case HCA_ERR_ALIGN: return "HCA_ERR_ALIGN: pointer not 16-byte aligned or D*element size not a multiple of 16";
    case HCA_ERR_ARG: return "HCA_ERR_ARG: W < 1, m < 1, non-finite scale or bad tile size";
    case HCA_ERR_SEG: return "HCA_ERR_SEG: segment ids decrease or padding is not a suffix";
    case HCA_ERR_WORKSPACE: return "HCA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case HCA_ERR_UNSUPPORTED: return "HCA_ERR_UNSUPPORTED: no kernel for this dtype/D combination";
    case HCA_ERR_CUDA: return "HCA_ERR_CUDA: a CUDA call or launch failed";
    case HCA_ERR_TIMEOUT: return "HCA_ERR_TIMEOUT: an on-device wait gave up";
    default: return "HCA_ERR_UNKNOWN";
  }
}

int hca_version(void) { return 1; }

size_t hca_workspace_size(int B, int H, int S, int D, int W, int m, int dtype, int for_backward) {
  if (check_dims(B, H, S, D, W, m, dtype) != HCA_OK) return 0;
  return for_backward ? bwd_ws_bytes(B, H, S, D, W, m, dtype) : fwd_ws_bytes(B, S);
}

int hca_test_inject(int what, long long value) {
  if (value < 0) return HCA_ERR_ARG;
  switch (what) {
    case HCA_INJECT_RESET:
      g_inject_launch_failures = 0;
      g_inject_stall_mask = 0;
      g_wait_ns = kDefaultWaitNs;
      g_csa_union = 0;
      return HCA_OK;
    case HCA_INJECT_LAUNCH_FAILURE: g_inject_launch_failures = value; return HCA_OK;
    case HCA_INJECT_STALL:
      if (value > (HCA_STALL_FWD | HCA_STALL_DQ | HCA_STALL_DKV)) return HCA_ERR_ARG;
      g_inject_stall_mask = (int)value;
      return HCA_OK;
    case HCA_INJECT_WAIT_LIMIT_NS: g_wait_ns = value == 0 ? kDefaultWaitNs : (unsigned long long)value; return HCA_OK;
    case HCA_INJECT_CSA_UNION:
      if (value > 16384 || (value > 1 && value % 64 != 0)) return HCA_ERR_ARG;
      g_csa_union = (int)value;
      return HCA_OK;
    default: return HCA_ERR_ARG;
  }
}

size_t hca_compress_workspace_size(int B, int S, int m) {
  if (B < 0 || S < 0 || m < 1 || S > (1 << 30)) return 0;
  const size_t n = compress_workspace_bytes(B, S, m);
  return n ? n : kAlign;
}

static int compress_checks(const void *x, const float *g, const float *bias, const int32_t *seg, const void *out,
                           int B, int S, int D, int m, int dtype) {
  if (dtype != HCA_BF16 && dtype != HCA_F32) return HCA_ERR_DTYPE;
  if (B < 0 || S < 0 || D < 1 || S > (1 << 30) || (double)B * S * D > 9.0e18) return HCA_ERR_SHAPE;
  if (m < 1) return HCA_ERR_ARG;
  if (D % 32 != 0 || D > 256) return HCA_ERR_UNSUPPORTED;
  if (B * (long long)S == 0) return HCA_OK;
  if (!x || !g || !bias || !out) return HCA_ERR_NULL;
  if (!aligned16(x) || !aligned16(out) || (seg && !aligned16(seg))) return HCA_ERR_ALIGN;
  return HCA_OK;
}

int hca_compress_fwd(const void *x, const float *g, const float *bias, const int32_t *seg, void *ckv, int B, int S,
                     int D, int m, int dtype, void *stream) {
  int rc = compress_checks(x, g, bias, seg, ckv, B, S, D, m, dtype);
  if (rc != HCA_OK || B * (long long)S == 0) return rc;
  if (take_launch_failure()) return HCA_ERR_CUDA;
  return cuda_status(compress_fwd(x, g, bias, seg, ckv, B, S, D, m, dtype, static_cast<cudaStream_t>(stream)));
}

int hca_compress_bwd(const void *x, const float *g, const float *bias, const int32_t *seg, const void *dckv, void *dx,
                     float *dg, float *dbias, int B, int S, int D, int m, int dtype, void *workspace,
                     size_t workspace_bytes, void *stream) {
  int rc = compress_checks(x, g, bias, seg, dckv, B, S, D, m, dtype);
  if (rc != HCA_OK) return rc;
  if (!dbias) return HCA_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B * (long long)S == 0) return cuda_status(cudaMemsetAsync(dbias, 0, sizeof(float) * m, st));
  if (!dx || !dg) return HCA_ERR_NULL;
  if (!aligned16(dx)) return HCA_ERR_ALIGN;
  rc = check_ws(workspace, workspace_bytes, compress_workspace_bytes(B, S, m));
  if (rc != HCA_OK) return rc;
  if (take_launch_failure()) return HCA_ERR_CUDA;
  return cuda_status(compress_bwd(x, g, bias, seg, dckv, dx, dg, dbias, static_cast<float *>(workspace), B, S, D, m,
                                  dtype, st));
}

size_t hca_indexer_workspace_size(int B, int S, int m) {
  if (B < 0 || S < 0 || m < 1 || S > (1 << 30)) return 0;
  return indexer_workspace_bytes(B, S, m);
}

int hca_indexer_topk(const void *qi, const void *ki, const float *w, const int32_t *seg, int32_t *sel, float *scores,
                     int B, int S, int Hi, int Di, int m, int k, void *workspace, size_t workspace_bytes,
                     void *stream) {
  if (B < 0 || S < 0 || Hi < 1 || S > (1 << 30) || (double)B * S * Hi * Di > 9.0e18) return HCA_ERR_SHAPE;
  if (m < 1 || k < 1) return HCA_ERR_ARG;
  if (Di != 128) return HCA_ERR_UNSUPPORTED;
  const long long Sc = ((long long)S + m - 1) / m;
  if (Sc > (long long)indexer_max_entries()) return HCA_ERR_UNSUPPORTED;
  if (B * (long long)S == 0) return HCA_OK;
  if (!qi || !ki || !w || !sel) return HCA_ERR_NULL;
  if (!aligned16(qi) || !aligned16(ki) || (seg && !aligned16(seg))) return HCA_ERR_ALIGN;
  int rc = check_ws(workspace, workspace_bytes, indexer_workspace_bytes(B, S, m));
  if (rc != HCA_OK) return rc;
  if (take_launch_failure()) return HCA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c = carve_fwd(workspace, B, S);
  rc = cuda_status(launch_prep(seg, B, S, c.sstart, c.status, st));
  if (rc != HCA_OK) return rc;
  char *p = c.p + fwd_ws_bytes(B, S);
  IndexerArgs a;
  a.qi = qi; a.ki = ki; a.w = w; a.sstart = seg ? c.sstart : nullptr; a.sel = sel; a.scores = scores;
  a.qc = p;
  a.buf = reinterpret_cast<float *>(p + align_up((size_t)B * S * 128 * 2));
  a.status = c.status; a.wait_ns = wait_limit_ns();
  a.B = B; a.S = S; a.Hi = Hi; a.m = m; a.k = k;
  return cuda_status(indexer_topk(a, st));
}

int hca_query_tile_positions(int H, int D, int dtype) {
  if (H < 1) return 0;
  if (tc_fwd_supported(H, D, dtype)) return tc_query_tile_positions(H);
  return 1;
}

int hca_attn_fwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, void *out, float *lse, int B,
                 int H, int S, int D, int W, int m, float scale, int dtype, void *workspace, size_t workspace_bytes,
                 void *stream) {
  int rc = check_dims(B, H, S, D, W, m, dtype);
  if (rc != HCA_OK) return rc;
  if (!std::isfinite(scale)) return HCA_ERR_ARG;
  if (!supported(H, D, dtype)) return HCA_ERR_UNSUPPORTED;
  if (B * (long long)S == 0) return HCA_OK;
  if (!q || !kv || !ckv || !out || !lse) return HCA_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(ckv) || !aligned16(out) || !aligned16(lse) ||
      (seg && !aligned16(seg)))
    return HCA_ERR_ALIGN;
  rc = check_ws(workspace, workspace_bytes, fwd_ws_bytes(B, S));
  if (rc != HCA_OK) return rc;
  if (take_launch_failure()) return HCA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c = carve_fwd(workspace, B, S);
  rc = cuda_status(launch_prep(seg, B, S, c.sstart, c.status, st));
  if (rc != HCA_OK) return rc;
  FwdArgs a;
  a.q = q; a.kv = kv; a.ckv = ckv;
  a.sstart = seg ? c.sstart : nullptr;
  a.status = c.status; a.status_rw = c.status;
  a.out = out; a.lse = lse;
  a.B = B; a.H = H; a.S = S; a.D = D; a.W = W; a.m = m; a.scale = scale; a.dtype = dtype;
  a.wait_ns = wait_limit_ns();
  a.stall = 0;
  if (dtype == HCA_BF16) {
    a.stall = take_stall_mask() & HCA_STALL_FWD;
    return cuda_status(tc_fwd(a, st));
  }
  return cuda_status(simt_fwd(a, st));
}

int hca_attn_bwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const void *out,
                 const float *lse, const void *dout, void *dq, void *dkv, void *dckv, int B, int H, int S, int D,
                 int W, int m, float scale, int dtype, void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_dims(B, H, S, D, W, m, dtype);
  if (rc != HCA_OK) return rc;
  if (!std::isfinite(scale)) return HCA_ERR_ARG;
  if (!supported(H, D, dtype)) return HCA_ERR_UNSUPPORTED;
  if (B * (long long)S == 0) return HCA_OK;
  if (!q || !kv || !ckv || !out || !lse || !dout || !dq || !dkv || !dckv) return HCA_ERR_NULL;
  const void *ptrs[] = {q, kv, ckv, out, lse, dout, dq, dkv, dckv};
  for (const void *p : ptrs)
    if (!aligned16(p)) return HCA_ERR_ALIGN;
  if (seg && !aligned16(seg)) return HCA_ERR_ALIGN;
  rc = check_ws(workspace, workspace_bytes, bwd_ws_bytes(B, H, S, D, W, m, dtype));
  if (rc != HCA_OK) return rc;
  if (take_launch_failure()) return HCA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c = carve_fwd(workspace, B, S);
  rc = cuda_status(launch_prep(seg, B, S, c.sstart, c.status, st));
  if (rc != HCA_OK) return rc;
  char *p = c.p + fwd_ws_bytes(B, S);
  BwdArgs a;
  a.q = q; a.kv = kv; a.ckv = ckv; a.out = out; a.dout = dout; a.lse = lse;
  a.sstart = seg ? c.sstart : nullptr;
  a.status = c.status; a.status_rw = c.status;
  a.dq = dq; a.dkv = dkv; a.dckv = dckv;
  a.delta = reinterpret_cast<float *>(p);
  p += align_up((size_t)B * H * S * sizeof(float));
  a.scratch = p;
  a.scratch_bytes = tc_bwd_scratch_bytes(B, H, S, D, W, m, dtype);
  a.B = B; a.H = H; a.S = S; a.D = D; a.W = W; a.m = m; a.scale = scale; a.dtype = dtype;
  a.wait_ns = wait_limit_ns();
  a.stall = 0;
  if (dtype == HCA_BF16) {
    a.stall = take_stall_mask() & (HCA_STALL_DQ | HCA_STALL_DKV);
    return cuda_status(tc_bwd(a, st));
  }
  return cuda_status(simt_bwd(a, st));
}

size_t hca_csa_workspace_size(int B, int H, int S, int D, int W, int m, int k, int dtype, int for_backward) {
  if (check_dims(B, H, S, D, W, m, dtype) != HCA_OK || k < 1) return 0;
  if (dtype != HCA_BF16 || D != 128 || !tc_fwd_supported(H, D, dtype) || !csa_shape_ok(H, k)) return 0;
  return for_backward ? csa_bwd_ws_bytes(B, H, S, D, W, m, k) : csa_fwd_ws_bytes(B, H, S, k);
}

static int csa_checks(int B, int H, int S, int D, int W, int m, int k, float scale, int dtype) {
  int rc = check_dims(B, H, S, D, W, m, dtype);
  if (rc != HCA_OK) return rc;
  if (!std::isfinite(scale) || k < 1) return HCA_ERR_ARG;
  // CSA runs on the tensor-core kernels only (bf16, D = 128, H a multiple of 32)
  if (dtype != HCA_BF16 || D != 128 || !tc_fwd_supported(H, D, dtype) || !csa_shape_ok(H, k)) return HCA_ERR_UNSUPPORTED;
  return HCA_OK;
}

int hca_csa_attn_fwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const int32_t *sel,
                     void *out, float *lse, int B, int H, int S, int D, int W, int m, int k, float scale, int dtype,
                     void *workspace, size_t workspace_bytes, void *stream) {
  int rc = csa_checks(B, H, S, D, W, m, k, scale, dtype);
  if (rc != HCA_OK) return rc;
  if (B * (long long)S == 0) return HCA_OK;
  if (!q || !kv || !ckv || !sel || !out || !lse) return HCA_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(ckv) || !aligned16(out) || !aligned16(lse) ||
      (seg && !aligned16(seg)) || !aligned16(sel))
    return HCA_ERR_ALIGN;
  rc = check_ws(workspace, workspace_bytes, csa_fwd_ws_bytes(B, H, S, k));
  if (rc != HCA_OK) return rc;
  if (take_launch_failure()) return HCA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c = carve_fwd(workspace, B, S);
  rc = cuda_status(launch_prep(seg, B, S, c.sstart, c.status, st));
  if (rc != HCA_OK) return rc;
  CsaUnion u;
  rc = cuda_status(csa_build_union(sel, seg ? c.sstart : nullptr, B, S, m, k, 2 * csa_pq(H), u,
                                   c.p + fwd_ws_bytes(B, S), st));
  if (rc != HCA_OK) return rc;
  FwdArgs a;
  a.q = q; a.kv = kv; a.ckv = ckv;
  a.sstart = seg ? c.sstart : nullptr;
  a.status = c.status; a.status_rw = c.status;
  a.out = out; a.lse = lse;
  a.B = B; a.H = H; a.S = S; a.D = D; a.W = W; a.m = m; a.scale = scale; a.dtype = dtype;
  a.wait_ns = wait_limit_ns();
  a.stall = take_stall_mask() & HCA_STALL_FWD;
  return cuda_status(tc_fwd(a, st, &u));
}

int hca_csa_attn_bwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const int32_t *sel,
                     const void *out, const float *lse, const void *dout, void *dq, void *dkv, void *dckv, int B,
                     int H, int S, int D, int W, int m, int k, float scale, int dtype, void *workspace,
                     size_t workspace_bytes, void *stream) {
  int rc = csa_checks(B, H, S, D, W, m, k, scale, dtype);
  if (rc != HCA_OK) return rc;
  if (B * (long long)S == 0) return HCA_OK;
  if (!q || !kv || !ckv || !sel || !out || !lse || !dout || !dq || !dkv || !dckv) return HCA_ERR_NULL;
  const void *ptrs[] = {q, kv, ckv, sel, out, lse, dout, dq, dkv, dckv};
  for (const void *p : ptrs)
    if (!aligned16(p)) return HCA_ERR_ALIGN;
  if (seg && !aligned16(seg)) return HCA_ERR_ALIGN;
  rc = check_ws(workspace, workspace_bytes, csa_bwd_ws_bytes(B, H, S, D, W, m, k));
  if (rc != HCA_OK) return rc;
  if (take_launch_failure()) return HCA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c = carve_fwd(workspace, B, S);
  rc = cuda_status(launch_prep(seg, B, S, c.sstart, c.status, st));
  if (rc != HCA_OK) return rc;
  char *p = c.p + fwd_ws_bytes(B, S);
  BwdArgs a;
  a.q = q; a.kv = kv; a.ckv = ckv; a.out = out; a.dout = dout; a.lse = lse;
  a.sstart = seg ? c.sstart : nullptr;
  a.status = c.status; a.status_rw = c.status;
  a.dq = dq; a.dkv = dkv; a.dckv = dckv;
  a.delta = reinterpret_cast<float *>(p);
  p += align_up((size_t)B * H * S * sizeof(float));
  a.scratch = p;
  a.scratch_bytes = tc_bwd_scratch_bytes(B, H, S, D, W, m, dtype, true);
  p += a.scratch_bytes;
  a.B = B; a.H = H; a.S = S; a.D = D; a.W = W; a.m = m; a.scale = scale; a.dtype = dtype;
  a.wait_ns = wait_limit_ns();
  a.stall = take_stall_mask() & (HCA_STALL_DQ | HCA_STALL_DKV);
  CsaBwd cb;
  rc = cuda_status(csa_build_union(sel, a.sstart, B, S, m, k, csa_pq(H), cb.u, p, st));
  if (rc != HCA_OK) return rc;
  p += csa_union_bytes(B, S, csa_pq(H), k);
  cb.acc = reinterpret_cast<float *>(p);
  return cuda_status(tc_bwd(a, st, &cb));
}

// Local sliding attention: the HCA calls with a compression ratio larger
// than the sequence (no window of length m completes, so the compressed set
// is empty).  The one ckv row that this ratio implies is never visible; kv
// stands in for it, and its gradient row lands in scratch at the end of the
// backward workspace.
size_t hca_local_workspace_size(int B, int H, int S, int D, int W, int dtype, int for_backward) {
  const int m = S + 1;
  if (check_dims(B, H, S, D, W, m, dtype) != HCA_OK) return 0;
  if (!for_backward) return fwd_ws_bytes(B, S);
  return bwd_ws_bytes(B, H, S, D, W, m, dtype) + align_up((size_t)B * D * elt_bytes(dtype));
}

int hca_local_attn_fwd(const void *q, const void *kv, const int32_t *seg, void *out, float *lse, int B, int H, int S,
                       int D, int W, float scale, int dtype, void *workspace, size_t workspace_bytes, void *stream) {
  return hca_attn_fwd(q, kv, kv, seg, out, lse, B, H, S, D, W, S + 1, scale, dtype, workspace, workspace_bytes,
                      stream);
}

int hca_local_attn_bwd(const void *q, const void *kv, const int32_t *seg, const void *out, const float *lse,
                       const void *dout, void *dq, void *dkv, int B, int H, int S, int D, int W, float scale, int dtype,
                       void *workspace, size_t workspace_bytes, void *stream) {
  const int m = S + 1;
  int rc = check_dims(B, H, S, D, W, m, dtype);
  if (rc != HCA_OK) return rc;
  const size_t need = bwd_ws_bytes(B, H, S, D, W, m, dtype);
  rc = check_ws(workspace, workspace_bytes, need + align_up((size_t)B * D * elt_bytes(dtype)));
  if (rc != HCA_OK) return rc;
  void *dckv = static_cast<char *>(workspace) + need;  // [B, 1, D], discarded
  return hca_attn_bwd(q, kv, kv, seg, out, lse, dout, dq, dkv, dckv, B, H, S, D, W, m, scale, dtype, workspace,
                      need, stream);
}

int hca_visible_pairs(const int32_t *seg, int B, int S, int W, int m, int64_t *raw_pairs, int64_t *comp_pairs,
                      void *workspace, size_t workspace_bytes, void *stream) {
  if (B < 0 || S < 0 || S > (1 << 30)) return HCA_ERR_SHAPE;
  if (W < 1 || m < 1) return HCA_ERR_ARG;
  if (B == 0) return HCA_OK;
  if (!raw_pairs || !comp_pairs) return HCA_ERR_NULL;
  if (seg && !aligned16(seg)) return HCA_ERR_ALIGN;
  int rc = check_ws(workspace, workspace_bytes, fwd_ws_bytes(B, S));
  if (rc != HCA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c = carve_fwd(workspace, B, S);
  rc = cuda_status(launch_prep(seg, B, S, c.sstart, c.status, st));
  if (rc != HCA_OK) return rc;
  return cuda_status(launch_visible_pairs(seg ? c.sstart : nullptr, B, S, W, m, raw_pairs, comp_pairs, st));
}

int hca_tile_map(const int32_t *seg, int B, int S, int W, int m, int Pq, int32_t *map, void *workspace,
                 size_t workspace_bytes, void *stream) {
  if (B < 0 || S < 0 || S > (1 << 30)) return HCA_ERR_SHAPE;
  if (W < 1 || m < 1 || Pq < 1) return HCA_ERR_ARG;
  if (B * (long long)S == 0) return HCA_OK;
  if (!map) return HCA_ERR_NULL;
  if (!aligned16(map) || (seg && !aligned16(seg))) return HCA_ERR_ALIGN;
  int rc = check_ws(workspace, workspace_bytes, fwd_ws_bytes(B, S));
  if (rc != HCA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c = carve_fwd(workspace, B, S);
  rc = cuda_status(launch_prep(seg, B, S, c.sstart, c.status, st));
  if (rc != HCA_OK) return rc;
  return cuda_status(launch_tile_map(seg ? c.sstart : nullptr, B, S, W, m, Pq, map, st));
}

int hca_workspace_status(const void *workspace, void *stream) {
  if (!workspace) return HCA_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return HCA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return HCA_ERR_CUDA;
  return v;
}

}  // extern "C"
