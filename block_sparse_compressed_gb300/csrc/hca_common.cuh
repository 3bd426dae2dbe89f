// hca_common.cuh -- shared device helpers of libhca: the analytic
// visibility intervals, workspace layout and status word.
//
// Visibility ("Add HCA Static Compilation for Splash Attention [Deepseek
// v4]", Description: sliding window + completed compression windows, segment
// ids).  With segments stored as contiguous runs (non-decreasing ids,
// padding as a suffix) the per-element rule collapses to two intervals per
// query i, given sstart = first position of i's segment:
//   raw rows          t in [max(i-W+1, sstart), i]
//   compressed        j in [ceil(sstart/m), floor((i+1)/m) - 1]
// A compressed window [j*m, (j+1)*m-1] lies inside the query's document
// exactly when j*m >= sstart and (j+1)*m-1 <= i.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/hca.h"

namespace hca {

// ---------------------------------------------------------------------------
// workspace layout (all offsets 256-byte aligned)
// ---------------------------------------------------------------------------
constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;  // int32 status at offset 0

__host__ __device__ inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

struct FwdWs {
  int32_t *status;
  int32_t *sstart;  // [B,S] segment start per position, -1 = padding
};

// ---------------------------------------------------------------------------
// per-row intervals
// ---------------------------------------------------------------------------
struct RowIv {
  int valid;
  int rlo, rhi;  // inclusive raw range (rlo <= rhi when valid)
  int clo, chi;  // inclusive compressed range (empty when clo > chi)
};

__device__ __forceinline__ int seg_start(const int32_t *sstart, int b, int S, int i) {
  return sstart ? sstart[(size_t)b * S + i] : 0;
}

__device__ __forceinline__ RowIv row_interval(const int32_t *sstart, int b, int S, int i, int W, int m) {
  RowIv r;
  r.valid = 0;
  r.rlo = 0; r.rhi = -1; r.clo = 0; r.chi = -1;
  if (i < 0 || i >= S) return r;
  int ss = seg_start(sstart, b, S, i);
  if (ss < 0) return r;
  r.valid = 1;
  r.rlo = max(i - W + 1, ss);
  r.rhi = i;
  r.clo = (ss + m - 1) / m;
  r.chi = (i + 1) / m - 1;
  return r;
}

// Union of the intervals of query positions [p0, p1): the key ranges a tile
// of those positions has to visit, as half-open ranges (lo == hi: none).
struct TileRange {
  int rlo, rhi, clo, chi;
};

__device__ __forceinline__ TileRange tile_range_serial(const int32_t *sstart, int b, int S, int p0, int p1, int W, int m) {
  TileRange t;
  int rlo = 0x7fffffff, rhi = -1, clo = 0x7fffffff, chi = -1;
  for (int i = p0; i < p1 && i < S; ++i) {
    RowIv r = row_interval(sstart, b, S, i, W, m);
    if (!r.valid) continue;
    rlo = min(rlo, r.rlo);
    rhi = max(rhi, r.rhi);
    if (r.chi >= r.clo) {
      clo = min(clo, r.clo);
      chi = max(chi, r.chi);
    }
  }
  t.rlo = rhi < 0 ? 0 : rlo;
  t.rhi = rhi < 0 ? 0 : rhi + 1;
  t.clo = chi < 0 ? 0 : clo;
  t.chi = chi < 0 ? 0 : chi + 1;
  return t;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

}  // namespace hca
