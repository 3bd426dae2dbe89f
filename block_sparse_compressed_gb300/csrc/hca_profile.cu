// hca_profile.cu -- optional per-kernel timing of libhca launches.
//
// While enabled, every kernel the library launches is bracketed by a pair of
// CUDA events recorded on the launch stream; hca_profile_read synchronises
// on the recorded events and returns launches and total device time per
// kernel.  Disabled (the default), a launch only tests one flag.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "hca_common.cuh"
#include "hca_internal.h"

namespace hca {
namespace {

struct Rec {
  int kernel;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_pending;
std::vector<cudaEvent_t> g_pool;
long long g_launches[kNumKernels] = {};
double g_ms[kNumKernels] = {};

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

const char *kNames[kNumKernels] = {"hca_prep",       "hca_fwd_tc",   "hca_bwd_dq",       "hca_bwd_dkv",
                                   "hca_bwd_reduce", "hca_simt_fwd", "hca_simt_bwd",     "hca_visibility",
                                   "hca_compress",   "hca_index_score", "hca_index_topk",   "hca_csa_union",
                                   "hca_csa_dckv"};

}  // namespace

ProfScope::ProfScope(int kernel, cudaStream_t st) : kernel_(kernel), st_(st), start_(nullptr) {
  if (!g_on) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  start_ = take_event();
  if (start_ && cudaEventRecord(start_, st_) != cudaSuccess) {
    g_pool.push_back(start_);
    start_ = nullptr;
  }
}

ProfScope::~ProfScope() {
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t stop = take_event();
  if (stop && cudaEventRecord(stop, st_) == cudaSuccess) {
    g_pending.push_back(Rec{kernel_, start_, stop});
  } else {
    g_pool.push_back(start_);
    if (stop) g_pool.push_back(stop);
  }
}

}  // namespace hca

using namespace hca;

extern "C" {

HCA_API int hca_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = on != 0;
  for (int k = 0; k < kNumKernels; ++k) {
    g_launches[k] = 0;
    g_ms[k] = 0.0;
  }
  for (Rec &r : g_pending) {
    cudaEventSynchronize(r.stop);
    g_pool.push_back(r.start);
    g_pool.push_back(r.stop);
  }
  g_pending.clear();
  return HCA_OK;
}

HCA_API int hca_profile_read(int kernel, long long *launches, double *total_ms) {
  if (kernel < 0 || kernel >= kNumKernels) return HCA_ERR_ARG;
  if (!launches || !total_ms) return HCA_ERR_NULL;
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = HCA_OK;
  for (Rec &r : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      rc = HCA_ERR_CUDA;
    g_launches[r.kernel] += 1;
    g_ms[r.kernel] += ms;
    g_pool.push_back(r.start);
    g_pool.push_back(r.stop);
  }
  g_pending.clear();
  *launches = g_launches[kernel];
  *total_ms = g_ms[kernel];
  return rc;
}

HCA_API const char *hca_kernel_name(int kernel) {
  if (kernel < 0 || kernel >= kNumKernels) return "";
  return kNames[kernel];
}

HCA_API int hca_num_kernels(void) { return kNumKernels; }

}  // extern "C"
