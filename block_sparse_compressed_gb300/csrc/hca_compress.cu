// hca_compress.cu -- the HCA compressor: pooling of length-m windows of kv
// rows into compressed entries, forward and backward.
//
// "[DeepSeek-V4] Implement Compressed Attention Layers", Description: the
// CSA/HCA compressors pool with a causal block bias; "Add HCA Static
// Compilation for Splash Attention [Deepseek v4]": the compressed entries
// are the length-m windows whose boundaries the static mask reproduces.
// Per window j of batch row b, over its positions t = j*m + r that exist and
// are not padding:
//   z_r = g[b,t] + bias[r],  a = softmax(z),  ckv[b,j,:] = sum_r a_r x[b,t,:]
// (a window with no such position gives a zero row).  Backward, for dckv:
//   dx[b,t] = a_r dckv[b,j],  da_r = <dckv[b,j], x[b,t]>,
//   dz_r = a_r (da_r - sum_s a_s da_s),  dg[b,t] = dz_r,
//   dbias[r] = sum over (b, j) of dz_r   (fixed-order reduction: deterministic)
//
// One warp per window.  Lanes first hold the window's logits (32 positions at
// a time), then D/32 consecutive columns each (one vector load per row) for
// the weighted row sum, several rows in flight per lane.  HBM-bound: x is
// read once per pass, ckv / dx written once.
#include <cuda_bf16.h>

#include "hca_common.cuh"
#include "hca_internal.h"

namespace hca {
namespace {

constexpr int kWarpsPerBlock = 8;

template <typename T>
__device__ __forceinline__ float ldf(const T *p);
template <>
__device__ __forceinline__ float ldf<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
template <typename T>
__device__ __forceinline__ void stf(T *p, float v);
template <>
__device__ __forceinline__ void stf<float>(float *p, float v) { *p = v; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// NC consecutive columns of a row per lane: one vector load / store.
template <typename T, int NC>
__device__ __forceinline__ void load_cols(const T *row, int lane, float (&v)[NC]) {
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int c = 0; c < NC; ++c) v[c] = row[NC * lane + c];
  } else {
    const uint16_t *h = reinterpret_cast<const uint16_t *>(row) + NC * lane;
    if constexpr (NC == 1) {
      v[0] = __uint_as_float((uint32_t)h[0] << 16);
    } else if constexpr (NC == 2) {
      const uint32_t u = *reinterpret_cast<const uint32_t *>(h);
      v[0] = __uint_as_float(u << 16);
      v[1] = __uint_as_float(u & 0xffff0000u);
    } else if constexpr (NC == 4) {
      const uint2 u = *reinterpret_cast<const uint2 *>(h);
      v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
      v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
      const uint4 u = *reinterpret_cast<const uint4 *>(h);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[2 * q] = __uint_as_float(w4[q] << 16);
        v[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
      }
    }
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// NC consecutive columns of a row per lane: one vector store.
template <typename T, int NC>
__device__ __forceinline__ void store_cols(T *row, int lane, const float (&v)[NC]) {
  if constexpr (sizeof(T) == 4 && NC == 4) {
    *reinterpret_cast<float4 *>(row + NC * lane) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (sizeof(T) == 4 && NC == 8) {
    float4 *q = reinterpret_cast<float4 *>(row + NC * lane);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else if constexpr (sizeof(T) == 2 && NC == 2) {
    *reinterpret_cast<uint32_t *>(row + NC * lane) = bf16x2_bits(v[0], v[1]);
  } else if constexpr (sizeof(T) == 2 && NC == 4) {
    *reinterpret_cast<uint2 *>(row + NC * lane) = make_uint2(bf16x2_bits(v[0], v[1]), bf16x2_bits(v[2], v[3]));
  } else if constexpr (sizeof(T) == 2 && NC == 8) {
    *reinterpret_cast<uint4 *>(row + NC * lane) = make_uint4(bf16x2_bits(v[0], v[1]), bf16x2_bits(v[2], v[3]),
                                                             bf16x2_bits(v[4], v[5]), bf16x2_bits(v[6], v[7]));
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c) stf(row + NC * lane + c, v[c]);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct CompressArgs {
  const void *x, *dckv;
  const float *g, *bias;
  const int32_t *seg;
  void *ckv, *dx;
  float *dg, *dz;  // dz: [B*Sc][m] per-window logit gradients (backward)
  int B, S, D, m, Sc;
};

// Max and normaliser of the window's logits; lane-strided over its positions.
__device__ __forceinline__ void window_stats(const CompressArgs &a, int b, int j, int lane, float &mx, float &sum) {
  mx = -INFINITY;
  for (int r = lane; r < a.m; r += 32) {
    const int t = j * a.m + r;
    if (t < a.S && (a.seg == nullptr || a.seg[(size_t)b * a.S + t] >= 0))
      mx = fmaxf(mx, a.g[(size_t)b * a.S + t] + a.bias[r]);
  }
  mx = warp_max(mx);
  sum = 0.f;
  if (mx > -INFINITY) {
    for (int r = lane; r < a.m; r += 32) {
      const int t = j * a.m + r;
      if (t < a.S && (a.seg == nullptr || a.seg[(size_t)b * a.S + t] >= 0))
        sum += expf(a.g[(size_t)b * a.S + t] + a.bias[r] - mx);
    }
    sum = warp_sum(sum);
  }
}

// Weight of position r of the window (0 if it does not exist or is padding).
__device__ __forceinline__ float window_weight(const CompressArgs &a, int b, int j, int r, float mx, float inv) {
  const int t = j * a.m + r;
  if (t >= a.S || (a.seg != nullptr && a.seg[(size_t)b * a.S + t] < 0)) return 0.f;
  return expf(a.g[(size_t)b * a.S + t] + a.bias[r] - mx) * inv;
}

template <typename T, int NC>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) hca_compress_fwd_kernel(const CompressArgs a) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (w >= (long long)a.B * a.Sc) return;
  const int b = (int)(w / a.Sc), j = (int)(w % a.Sc);
  float mx, sum;
  window_stats(a, b, j, lane, mx, sum);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  const T *x = static_cast<const T *>(a.x);
  if (sum > 0.f) {
    for (int r0 = 0; r0 < a.m; r0 += 32) {
      const float my = r0 + lane < a.m ? window_weight(a, b, j, r0 + lane, mx, inv) : 0.f;
      const int rn = min(32, min(a.m - r0, a.S - (j * a.m + r0)));
      const T *rows = x + ((size_t)b * a.S + j * a.m + r0) * a.D;
      // eight rows in flight per lane
      int rr = 0;
      for (; rr + 8 <= rn; rr += 8) {
        float v[8][NC];
#pragma unroll
        for (int u = 0; u < 8; ++u) load_cols<T, NC>(rows + (size_t)(rr + u) * a.D, lane, v[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          // padding rows (weight 0) are skipped, not multiplied: their values are arbitrary
          const float wr = __shfl_sync(0xffffffffu, my, rr + u);
          if (wr != 0.f) {
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[c] = fmaf(wr, v[u][c], acc[c]);
          }
        }
      }
      for (; rr < rn; ++rr) {
        float v[NC];
        load_cols<T, NC>(rows + (size_t)rr * a.D, lane, v);
        const float wr = __shfl_sync(0xffffffffu, my, rr);
        if (wr != 0.f) {
#pragma unroll
          for (int c = 0; c < NC; ++c) acc[c] = fmaf(wr, v[c], acc[c]);
        }
      }
    }
  }
  store_cols<T, NC>(static_cast<T *>(a.ckv) + ((size_t)b * a.Sc + j) * a.D, lane, acc);
}

template <typename T, int NC>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) hca_compress_bwd_kernel(const CompressArgs a) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (w >= (long long)a.B * a.Sc) return;
  const int b = (int)(w / a.Sc), j = (int)(w % a.Sc);
  float mx, sum;
  window_stats(a, b, j, lane, mx, sum);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  const T *x = static_cast<const T *>(a.x);
  T *dx = static_cast<T *>(a.dx);
  float gv[NC];
  load_cols<T, NC>(static_cast<const T *>(a.dckv) + ((size_t)b * a.Sc + j) * a.D, lane, gv);
  // pass 1: da_r = <dckv, x_r>, s = sum_r a_r da_r, dx_r = a_r dckv
  float s = 0.f;
  for (int r0 = 0; r0 < a.m; r0 += 32) {
    const float my = r0 + lane < a.m && sum > 0.f ? window_weight(a, b, j, r0 + lane, mx, inv) : 0.f;
    float my_da = 0.f;
    const int rn = max(0, min(32, min(a.m - r0, a.S - (j * a.m + r0))));
    const size_t base = (size_t)b * a.S + j * a.m + r0;
    int rr = 0;
    for (; rr + 4 <= rn; rr += 4) {
      float v[4][NC], d[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) load_cols<T, NC>(x + (base + rr + u) * a.D, lane, v[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float wr = __shfl_sync(0xffffffffu, my, rr + u);
        float o[NC];
        d[u] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          d[u] = fmaf(gv[c], v[u][c], d[u]);
          o[c] = wr * gv[c];
        }
        store_cols<T, NC>(dx + (base + rr + u) * a.D, lane, o);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float t = warp_sum(d[u]);
        if (lane == rr + u) my_da = t;
      }
    }
    for (; rr < rn; ++rr) {
      float v[NC], o[NC];
      load_cols<T, NC>(x + (base + rr) * a.D, lane, v);
      const float wr = __shfl_sync(0xffffffffu, my, rr);
      float d = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        d = fmaf(gv[c], v[c], d);
        o[c] = wr * gv[c];
      }
      store_cols<T, NC>(dx + (base + rr) * a.D, lane, o);
      d = warp_sum(d);
      if (lane == rr) my_da = d;
    }
    // positions without weight (padding) hold arbitrary values: their da is dropped
    if (my == 0.f) my_da = 0.f;
    s += warp_sum(my * my_da);
    // this chunk's da_r, kept for pass 2 in the logit-gradient buffer
    if (r0 + lane < a.m) a.dz[w * a.m + r0 + lane] = my_da;
  }
  // pass 2: dz_r = a_r (da_r - s)
  for (int r = lane; r < a.m; r += 32) {
    const int t = j * a.m + r;
    const float ar = sum > 0.f ? window_weight(a, b, j, r, mx, inv) : 0.f;
    const float dz = ar * (a.dz[w * a.m + r] - s);
    a.dz[w * a.m + r] = dz;
    if (t < a.S) a.dg[(size_t)b * a.S + t] = dz;
  }
}

// dbias[r] = sum over windows of dz[., r]: one block per r, a fixed
// per-thread stride then a fixed tree, so the result is run-to-run identical.
__global__ void __launch_bounds__(256) hca_compress_dbias_kernel(const float *dz, long long nwin, int m, float *dbias) {
  __shared__ float part[256];
  const int r = blockIdx.x;
  float acc = 0.f;
  for (long long wv = threadIdx.x; wv < nwin; wv += 256) acc += dz[wv * m + r];
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) dbias[r] = part[0];
}

template <typename T, int NC>
cudaError_t launch_fwd_nc(const CompressArgs &a, cudaStream_t st) {
  const long long nwin = (long long)a.B * a.Sc;
  if (nwin == 0) return cudaSuccess;
  ProfScope prof(kKCompress, st);
  hca_compress_fwd_kernel<T, NC><<<(unsigned)((nwin + kWarpsPerBlock - 1) / kWarpsPerBlock), 32 * kWarpsPerBlock, 0,
                                   st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fwd(const CompressArgs &a, cudaStream_t st) {
  switch (a.D / 32) {
    case 1: return launch_fwd_nc<T, 1>(a, st);
    case 2: return launch_fwd_nc<T, 2>(a, st);
    case 4: return launch_fwd_nc<T, 4>(a, st);
    case 8: return launch_fwd_nc<T, 8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int NC>
cudaError_t launch_bwd_nc(const CompressArgs &a, cudaStream_t st) {
  const long long nwin = (long long)a.B * a.Sc;
  hca_compress_bwd_kernel<T, NC><<<(unsigned)((nwin + kWarpsPerBlock - 1) / kWarpsPerBlock), 32 * kWarpsPerBlock, 0,
                                   st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd(const CompressArgs &a, float *dbias, cudaStream_t st) {
  const long long nwin = (long long)a.B * a.Sc;
  if (nwin == 0) return cudaMemsetAsync(dbias, 0, sizeof(float) * a.m, st);
  ProfScope prof(kKCompress, st);
  cudaError_t e0 = cudaErrorInvalidValue;
  switch (a.D / 32) {
    case 1: e0 = launch_bwd_nc<T, 1>(a, st); break;
    case 2: e0 = launch_bwd_nc<T, 2>(a, st); break;
    case 4: e0 = launch_bwd_nc<T, 4>(a, st); break;
    case 8: e0 = launch_bwd_nc<T, 8>(a, st); break;
    default: break;
  }
  if (e0 != cudaSuccess) return e0;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  hca_compress_dbias_kernel<<<a.m, 256, 0, st>>>(a.dz, nwin, a.m, dbias);
  return cudaGetLastError();
}

}  // namespace

size_t compress_workspace_bytes(int B, int S, int m) {
  const long long Sc = (S + m - 1) / m;
  return align_up((size_t)B * Sc * m * sizeof(float));
}

cudaError_t compress_fwd(const void *x, const float *g, const float *bias, const int32_t *seg, void *ckv, int B, int S,
                         int D, int m, int dtype, cudaStream_t st) {
  CompressArgs a = {};
  a.x = x; a.g = g; a.bias = bias; a.seg = seg; a.ckv = ckv;
  a.B = B; a.S = S; a.D = D; a.m = m; a.Sc = (S + m - 1) / m;
  return dtype == HCA_F32 ? launch_fwd<float>(a, st) : launch_fwd<__nv_bfloat16>(a, st);
}

cudaError_t compress_bwd(const void *x, const float *g, const float *bias, const int32_t *seg, const void *dckv,
                         void *dx, float *dg, float *dbias, float *dz, int B, int S, int D, int m, int dtype,
                         cudaStream_t st) {
  CompressArgs a = {};
  a.x = x; a.g = g; a.bias = bias; a.seg = seg; a.dckv = dckv; a.dx = dx; a.dg = dg; a.dz = dz;
  a.B = B; a.S = S; a.D = D; a.m = m; a.Sc = (S + m - 1) / m;
  return dtype == HCA_F32 ? launch_bwd<float>(a, dbias, st) : launch_bwd<__nv_bfloat16>(a, dbias, st);
}

}  // namespace hca
