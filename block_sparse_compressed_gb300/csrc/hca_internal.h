// hca_internal.h -- launch interfaces shared by the translation units of
// libhca (not part of the public C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace hca {

// kernels the optional profiler distinguishes (hca_profile_read ids)
enum KernelId {
  kKPrep = 0, kKFwdTc, kKBwdDq, kKBwdDkv, kKBwdReduce, kKSimtFwd, kKSimtBwd, kKVisibility, kKCompress,
  kKIndexScore, kKIndexTopk, kKCsaUnion, kKCsaDckv, kNumKernels
};

// Brackets the launches issued during its lifetime with CUDA events on `st`
// when profiling is enabled (hca_profile_enable); otherwise does nothing.
class ProfScope {
 public:
  ProfScope(int kernel, cudaStream_t st);
  ~ProfScope();
  ProfScope(const ProfScope &) = delete;
  ProfScope &operator=(const ProfScope &) = delete;

 private:
  int kernel_;
  cudaStream_t st_;
  cudaEvent_t start_;
};

struct FwdArgs {
  const void *q, *kv, *ckv;
  const int32_t *sstart;  // NULL = one segment per row
  const int32_t *status;  // device status word (non-zero: poison outputs)
  int32_t *status_rw;     // same word, writable (bounded waits report here)
  void *out;
  float *lse;
  int B, H, S, D, W, m;
  float scale;
  int dtype;
  uint64_t wait_ns;  // limit of the kernels' bounded waits
  int stall;         // failure-path test (hca_test_inject): HCA_STALL_* mask of kernels whose MMA warp stalls
};

struct BwdArgs {
  const void *q, *kv, *ckv, *out, *dout;
  const float *lse;
  const int32_t *sstart;
  const int32_t *status;
  int32_t *status_rw;
  void *dq, *dkv, *dckv;
  float *delta;  // [B,H,S] workspace
  void *scratch; // further backward workspace (tensor-core path)
  size_t scratch_bytes;
  int B, H, S, D, W, m;
  float scale;
  int dtype;
  uint64_t wait_ns;
  int stall;
};

// Failure-path test hooks (hca_test_inject).  take_launch_failure() is true
// when an injected launch failure is pending (and consumes it);
// take_stall_mask() returns (and clears) the HCA_STALL_* mask of kernels
// whose MMA warp stalls in the next call; wait_limit_ns() is the bounded wait
// limit for the next launch (2 s unless a test shortened it).
bool take_launch_failure();
int take_stall_mask();
uint64_t wait_limit_ns();
// How the CSA union is built (HCA_INJECT_CSA_UNION): 0 automatic, 1 the
// sorting kernel, c >= 64 the byte-mask kernel with chunks of c entries.
int csa_union_setting();

cudaError_t launch_prep(const int32_t *seg, int B, int S, int32_t *sstart, int32_t *status, cudaStream_t st);
cudaError_t launch_visible_pairs(const int32_t *sstart, int B, int S, int W, int m, int64_t *raw, int64_t *comp,
                                 cudaStream_t st);
cudaError_t launch_tile_map(const int32_t *sstart, int B, int S, int W, int m, int Pq, int32_t *map, cudaStream_t st);

cudaError_t simt_fwd(const FwdArgs &a, cudaStream_t st);
cudaError_t simt_bwd(const BwdArgs &a, cudaStream_t st);

// HCA compressor (hca_compress.cu)
size_t compress_workspace_bytes(int B, int S, int m);
cudaError_t compress_fwd(const void *x, const float *g, const float *bias, const int32_t *seg, void *ckv, int B, int S,
                         int D, int m, int dtype, cudaStream_t st);
cudaError_t compress_bwd(const void *x, const float *g, const float *bias, const int32_t *seg, const void *dckv,
                         void *dx, float *dg, float *dbias, float *dz, int B, int S, int D, int m, int dtype,
                         cudaStream_t st);

// Lightning Indexer (hca_indexer.cu)
struct IndexerArgs {
  const void *qi, *ki;       // [B,S,Hi,128], [B,Sc,128] bf16
  const float *w;            // [B,S,Hi]
  const int32_t *sstart;     // document starts (NULL = one document)
  int32_t *sel;              // [B,S,k]
  float *scores;             // optional [B,S,Sc]
  void *qc;                  // workspace: collapsed queries [B,S,128] bf16
  float *buf;                // workspace: chunk score buffer
  int32_t *status;
  uint64_t wait_ns;
  int B, S, Hi, m, k;
};
size_t indexer_workspace_bytes(int B, int S, int m);
size_t indexer_max_entries();
cudaError_t indexer_topk(const IndexerArgs &a, cudaStream_t st);

// CSA (hca_csa.cu): per group of P positions, the union of their valid
// selections with one position bit per entry
struct CsaUnion {
  int32_t *cnt;    // [B*ngroups] entries in the union
  int32_t *ent;    // [B*ngroups][cap] entry ids, ascending, padded to 16 with 0
  uint32_t *mask;  // [B*ngroups][cap] bit p: position p of the group selected it
  int P, cap, ngroups;
};
bool csa_shape_ok(int H, int k);
size_t csa_union_bytes(int B, int S, int P, int k);
cudaError_t csa_build_union(const int32_t *sel, const int32_t *sstart, int B, int S, int m, int k, int P,
                            CsaUnion &u, void *mem, cudaStream_t st);
size_t csa_dckv_acc_bytes(int B, int Sc);
struct BwdArgs;
cudaError_t csa_dckv(const BwdArgs &a, const CsaUnion &u, const float *rowstat, float *acc, cudaStream_t st);

// tensor-core (tcgen05) path
bool tc_fwd_supported(int H, int D, int dtype);
int tc_query_tile_positions(int H);
cudaError_t tc_fwd(const FwdArgs &a, cudaStream_t st, const CsaUnion *csa = nullptr);
bool tc_bwd_supported(int H, int D, int dtype);
struct CsaBwd {
  CsaUnion u;  // per dq tile (Pq positions)
  float *acc;  // [B][Sc][D] fp32 dckv accumulator
};
size_t tc_bwd_scratch_bytes(int B, int H, int S, int D, int W, int m, int dtype, bool csa = false);
cudaError_t tc_bwd(const BwdArgs &a, cudaStream_t st, const CsaBwd *csa = nullptr);

}  // namespace hca
