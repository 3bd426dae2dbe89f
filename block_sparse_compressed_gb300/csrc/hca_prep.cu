// hca_prep.cu -- segment preparation and the visibility enumerations.
//
//  * hca_prep_kernel: from seg[B,S] computes sstart[B,S] (first position of
//    each position's document, -1 for padding) with a block-wide max-scan,
//    and checks the ordering the interval form relies on (non-negative ids
//    non-decreasing, padding a suffix).  A violation is written to the
//    status word of the workspace.  ("Add HCA Static Compilation for Splash
//    Attention [Deepseek v4]", Description, packing/segment-id bullet.)
//  * visible_pairs_kernel / tile_map_kernel: the pair counts and per-tile key
//    ranges implied by the same interval arithmetic the attention kernels use
//    (hca_common.cuh), so they can be compared exactly with an enumeration.
#include "hca_common.cuh"
#include "hca_internal.h"

namespace hca {

constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads) hca_prep_kernel(const int32_t *__restrict__ seg, int S,
                                                                 int32_t *__restrict__ sstart,
                                                                 int32_t *__restrict__ status) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ int wmax[32];
  __shared__ int carry_s;
  __shared__ int bad_s;
  if (tid == 0) { carry_s = -1; bad_s = 0; }
  __syncthreads();
  const int32_t *sg = seg + (size_t)b * S;
  int32_t *ss = sstart + (size_t)b * S;
  for (int base = 0; base < S; base += kPrepThreads) {
    const int i = base + tid;
    int mark = -1;
    int id = -1;
    if (i < S) {
      id = sg[i];
      const int prev = i > 0 ? sg[i - 1] : -1;
      if (id >= 0 && (i == 0 || id != prev)) mark = i;
      // ordering: a valid id must follow a valid id that is not larger
      if (i > 0 && id >= 0 && (prev < 0 || prev > id)) bad_s = 1;
    }
    // inclusive max-scan of start marks
    int v = mark;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v = max(v, u);
    }
    if (lane == 31) wmax[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = wmax[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w = max(w, u);
      }
      wmax[lane] = w;
    }
    __syncthreads();
    const int carry = carry_s;
    if (warp > 0) v = max(v, wmax[warp - 1]);
    v = max(v, carry);
    if (i < S) ss[i] = id >= 0 ? v : -1;
    __syncthreads();
    if (tid == kPrepThreads - 1) carry_s = v;
    __syncthreads();
  }
  if (tid == 0 && bad_s) atomicExch(status, (int)HCA_ERR_SEG);
}

__global__ void hca_visible_pairs_kernel(const int32_t *__restrict__ sstart, int S, int W, int m,
                                         unsigned long long *__restrict__ raw_pairs,
                                         unsigned long long *__restrict__ comp_pairs) {
  const int b = blockIdx.y;
  unsigned long long r = 0, c = 0;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < S; i += gridDim.x * blockDim.x) {
    RowIv iv = row_interval(sstart, b, S, i, W, m);
    if (!iv.valid) continue;
    r += (unsigned long long)(iv.rhi - iv.rlo + 1);
    if (iv.chi >= iv.clo) c += (unsigned long long)(iv.chi - iv.clo + 1);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    r += __shfl_down_sync(0xffffffffu, r, off);
    c += __shfl_down_sync(0xffffffffu, c, off);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(raw_pairs + b, r);
    atomicAdd(comp_pairs + b, c);
  }
}

__global__ void hca_tile_map_kernel(const int32_t *__restrict__ sstart, int S, int W, int m, int Pq, int ntiles,
                                    int32_t *__restrict__ map) {
  const int b = blockIdx.y;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < ntiles; t += gridDim.x * blockDim.x) {
    TileRange r = tile_range_serial(sstart, b, S, t * Pq, t * Pq + Pq, W, m);
    int4 e = make_int4(r.rlo, r.rhi, r.clo, r.chi);
    reinterpret_cast<int4 *>(map)[(size_t)b * ntiles + t] = e;
  }
}

cudaError_t launch_prep(const int32_t *seg, int B, int S, int32_t *sstart, int32_t *status, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  if (seg == nullptr || B == 0 || S == 0) return cudaSuccess;
  ProfScope prof(kKPrep, st);
  hca_prep_kernel<<<B, kPrepThreads, 0, st>>>(seg, S, sstart, status);
  return cudaGetLastError();
}

cudaError_t launch_visible_pairs(const int32_t *sstart, int B, int S, int W, int m, int64_t *raw, int64_t *comp,
                                 cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(raw, 0, sizeof(int64_t) * B, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(comp, 0, sizeof(int64_t) * B, st);
  if (e != cudaSuccess || B == 0 || S == 0) return e;
  int blocks = (S + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  ProfScope prof(kKVisibility, st);
  hca_visible_pairs_kernel<<<dim3(blocks, B), 256, 0, st>>>(sstart, S, W, m,
                                                            reinterpret_cast<unsigned long long *>(raw),
                                                            reinterpret_cast<unsigned long long *>(comp));
  return cudaGetLastError();
}

cudaError_t launch_tile_map(const int32_t *sstart, int B, int S, int W, int m, int Pq, int32_t *map, cudaStream_t st) {
  if (B == 0 || S == 0) return cudaSuccess;
  const int nt = (S + Pq - 1) / Pq;
  int blocks = (nt + 127) / 128;
  if (blocks > 1024) blocks = 1024;
  ProfScope prof(kKVisibility, st);
  hca_tile_map_kernel<<<dim3(blocks, B), 128, 0, st>>>(sstart, S, W, m, Pq, nt, map);
  return cudaGetLastError();
}

}  // namespace hca
