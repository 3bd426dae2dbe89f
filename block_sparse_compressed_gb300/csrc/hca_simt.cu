// hca_simt.cu -- CUDA-core (SIMT) HCA forward and backward.
//
// These kernels carry the fp32 mode (fp32 inputs, fp32 arithmetic; a 1e-5
// accuracy target rules out TF32 tensor cores).  One warp owns one (b, h, i) query
// row for the forward and dq, or one key row for dkv / dckv; each lane holds
// D/32 coordinates.  The key ranges come from the analytic intervals in
// hca_common.cuh, so no mask is read or written.
//
// Math ("[DeepSeek-V4] Implement Compressed Attention Layers", review
// suggestions on the einsums: k = v = kv; "Add HCA Static Compilation for
// Splash Attention [Deepseek v4]", Description: sliding window + completed
// compression windows):
//   s = scale <q, r>;  online softmax over the visible keys;  lse = m + log l
//   backward:  P = exp(s - lse),  dP = <dO, r>,  Delta = <dO, out>,
//              dS = P (dP - Delta),  dq = scale sum dS r,
//              d r = sum over heads/queries (scale dS q + P dO).
#include <cuda_bf16.h>

#include "hca_common.cuh"
#include "hca_internal.h"

namespace hca {

template <typename T>
__device__ __forceinline__ float ld(const T *p) { return (float)*p; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
template <typename T>
__device__ __forceinline__ void stv(T *p, float v) { *p = (T)v; }
template <>
__device__ __forceinline__ void stv<__nv_bfloat16>(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <typename T, int DPL>
__device__ __forceinline__ void load_row(const T *row, int D, int lane, float (&x)[DPL]) {
#pragma unroll
  for (int k = 0; k < DPL; ++k) {
    int d = lane + 32 * k;
    x[k] = d < D ? ld(row + d) : 0.f;
  }
}

template <int DPL>
__device__ __forceinline__ float dot(const float (&a)[DPL], const float (&b)[DPL]) {
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < DPL; ++k) s = fmaf(a[k], b[k], s);
  return warp_sum(s);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <typename T, int DPL>
__global__ void __launch_bounds__(128) simt_fwd_kernel(const T *__restrict__ q, const T *__restrict__ kv,
                                                       const T *__restrict__ ckv, const int32_t *__restrict__ sstart,
                                                       const int32_t *__restrict__ status, T *__restrict__ out,
                                                       float *__restrict__ lse, int B, int H, int S, int D, int W,
                                                       int m, float scale) {
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * H * S) return;
  const int i = (int)(row % S);
  const int b = (int)(row / ((long long)S * H));
  const int Sc = (S + m - 1) / m;
  T *orow = out + row * D;
  if (*status != 0) {
    for (int d = lane; d < D; d += 32) stv(orow + d, __int_as_float(0x7fc00000));
    if (lane == 0) lse[row] = __int_as_float(0x7fc00000);
    return;
  }
  RowIv iv = row_interval(sstart, b, S, i, W, m);
  if (!iv.valid) {
    for (int d = lane; d < D; d += 32) stv(orow + d, 0.f);
    if (lane == 0) lse[row] = -INFINITY;
    return;
  }
  float qv[DPL], o[DPL], k[DPL];
  load_row<T, DPL>(q + row * D, D, lane, qv);
#pragma unroll
  for (int x = 0; x < DPL; ++x) o[x] = 0.f;
  float mx = -INFINITY, l = 0.f;
  const int nraw = iv.rhi - iv.rlo + 1;
  const int ncomp = iv.chi >= iv.clo ? iv.chi - iv.clo + 1 : 0;
  for (int n = 0; n < nraw + ncomp; ++n) {
    const T *kr = n < nraw ? kv + ((size_t)b * S + iv.rlo + n) * D : ckv + ((size_t)b * Sc + iv.clo + n - nraw) * D;
    load_row<T, DPL>(kr, D, lane, k);
    const float s = scale * dot(qv, k);
    const float mn = fmaxf(mx, s);
    const float corr = expf(mx - mn);
    const float p = expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int x = 0; x < DPL; ++x) o[x] = fmaf(p, k[x], o[x] * corr);
    mx = mn;
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int x = 0; x < DPL; ++x) {
    int d = lane + 32 * x;
    if (d < D) stv(orow + d, o[x] * inv);
  }
  if (lane == 0) lse[row] = mx + logf(l);
}

// ---------------------------------------------------------------------------
// backward: Delta = <dO, out>
// ---------------------------------------------------------------------------
template <typename T, int DPL>
__global__ void __launch_bounds__(128) simt_delta_kernel(const T *__restrict__ out, const T *__restrict__ dout,
                                                         float *__restrict__ delta, long long rows, int D) {
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float a[DPL], g[DPL];
  load_row<T, DPL>(out + row * D, D, lane, a);
  load_row<T, DPL>(dout + row * D, D, lane, g);
  float s = dot(a, g);
  if (lane == 0) delta[row] = s;
}

// dq for one (b,h,i) row per warp
template <typename T, int DPL>
__global__ void __launch_bounds__(128) simt_dq_kernel(const T *__restrict__ q, const T *__restrict__ kv,
                                                      const T *__restrict__ ckv, const int32_t *__restrict__ sstart,
                                                      const int32_t *__restrict__ status, const float *__restrict__ lse,
                                                      const float *__restrict__ delta, const T *__restrict__ dout,
                                                      T *__restrict__ dq, int B, int H, int S, int D, int W, int m,
                                                      float scale) {
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * H * S) return;
  const int i = (int)(row % S);
  const int b = (int)(row / ((long long)S * H));
  const int Sc = (S + m - 1) / m;
  T *grow = dq + row * D;
  if (*status != 0) {
    for (int d = lane; d < D; d += 32) stv(grow + d, __int_as_float(0x7fc00000));
    return;
  }
  RowIv iv = row_interval(sstart, b, S, i, W, m);
  if (!iv.valid) {
    for (int d = lane; d < D; d += 32) stv(grow + d, 0.f);
    return;
  }
  float qv[DPL], g[DPL], k[DPL], acc[DPL];
  load_row<T, DPL>(q + row * D, D, lane, qv);
  load_row<T, DPL>(dout + row * D, D, lane, g);
#pragma unroll
  for (int x = 0; x < DPL; ++x) acc[x] = 0.f;
  const float L = lse[row], Dl = delta[row];
  const int nraw = iv.rhi - iv.rlo + 1;
  const int ncomp = iv.chi >= iv.clo ? iv.chi - iv.clo + 1 : 0;
  for (int n = 0; n < nraw + ncomp; ++n) {
    const T *kr = n < nraw ? kv + ((size_t)b * S + iv.rlo + n) * D : ckv + ((size_t)b * Sc + iv.clo + n - nraw) * D;
    load_row<T, DPL>(kr, D, lane, k);
    float s = 0.f, dp = 0.f;
#pragma unroll
    for (int x = 0; x < DPL; ++x) {
      s = fmaf(qv[x], k[x], s);
      dp = fmaf(g[x], k[x], dp);
    }
    s = warp_sum(s);
    dp = warp_sum(dp);
    const float p = expf(scale * s - L);
    const float ds = p * (dp - Dl);
#pragma unroll
    for (int x = 0; x < DPL; ++x) acc[x] = fmaf(ds, k[x], acc[x]);
  }
#pragma unroll
  for (int x = 0; x < DPL; ++x) {
    int d = lane + 32 * x;
    if (d < D) stv(grow + d, scale * acc[x]);
  }
}

// gradient of one key row per warp: raw row t (comp = 0) or compressed entry j
template <typename T, int DPL>
__global__ void __launch_bounds__(128) simt_dkey_kernel(const T *__restrict__ q, const T *__restrict__ kv,
                                                        const T *__restrict__ ckv, const int32_t *__restrict__ sstart,
                                                        const int32_t *__restrict__ status,
                                                        const float *__restrict__ lse, const float *__restrict__ delta,
                                                        const T *__restrict__ dout, T *__restrict__ dkv,
                                                        T *__restrict__ dckv, int B, int H, int S, int D, int W, int m,
                                                        float scale) {
  const int Sc = (S + m - 1) / m;
  const long long kid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long nraw = (long long)B * S;
  if (kid >= nraw + (long long)B * Sc) return;
  const bool comp = kid >= nraw;
  const int b = comp ? (int)((kid - nraw) / Sc) : (int)(kid / S);
  const int key = comp ? (int)((kid - nraw) % Sc) : (int)(kid % S);
  T *grow = comp ? dckv + ((size_t)b * Sc + key) * D : dkv + ((size_t)b * S + key) * D;
  if (*status != 0) {
    for (int d = lane; d < D; d += 32) stv(grow + d, __int_as_float(0x7fc00000));
    return;
  }
  float r[DPL], qv[DPL], g[DPL], acc[DPL];
  load_row<T, DPL>(comp ? ckv + ((size_t)b * Sc + key) * D : kv + ((size_t)b * S + key) * D, D, lane, r);
#pragma unroll
  for (int x = 0; x < DPL; ++x) acc[x] = 0.f;
  // candidate queries: raw row t is seen by i in [t, t+W-1]; entry j by
  // i >= (j+1)m - 1 up to the end of the document holding j's window.
  const int i0 = comp ? (key + 1) * m - 1 : key;
  const int i1 = comp ? S : (int)min((long long)S, (long long)key + W);
  for (int i = i0; i < i1; ++i) {
    RowIv iv = row_interval(sstart, b, S, i, W, m);
    if (!iv.valid) break;  // padding is a suffix
    bool vis = comp ? (iv.clo <= key && key <= iv.chi) : (iv.rlo <= key);
    if (!vis) {
      if (comp) break;  // later documents start after this window
      continue;
    }
    for (int h = 0; h < H; ++h) {
      const long long row = ((long long)b * H + h) * S + i;
      load_row<T, DPL>(q + row * D, D, lane, qv);
      load_row<T, DPL>(dout + row * D, D, lane, g);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int x = 0; x < DPL; ++x) {
        s = fmaf(qv[x], r[x], s);
        dp = fmaf(g[x], r[x], dp);
      }
      s = warp_sum(s);
      dp = warp_sum(dp);
      const float p = expf(scale * s - lse[row]);
      const float ds = scale * p * (dp - delta[row]);
#pragma unroll
      for (int x = 0; x < DPL; ++x) acc[x] = fmaf(ds, qv[x], fmaf(p, g[x], acc[x]));
    }
  }
#pragma unroll
  for (int x = 0; x < DPL; ++x) {
    int d = lane + 32 * x;
    if (d < D) stv(grow + d, acc[x]);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <typename T, int DPL>
static cudaError_t fwd_t(const FwdArgs &a, cudaStream_t st) {
  const long long rows = (long long)a.B * a.H * a.S;
  if (rows == 0) return cudaSuccess;
  ProfScope prof(kKSimtFwd, st);
  simt_fwd_kernel<T, DPL><<<(unsigned)((rows + 3) / 4), 128, 0, st>>>(
      (const T *)a.q, (const T *)a.kv, (const T *)a.ckv, a.sstart, a.status, (T *)a.out, a.lse, a.B, a.H, a.S, a.D,
      a.W, a.m, a.scale);
  return cudaGetLastError();
}

template <typename T, int DPL>
static cudaError_t bwd_t(const BwdArgs &a, cudaStream_t st) {
  const long long rows = (long long)a.B * a.H * a.S;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  ProfScope prof(kKSimtBwd, st);
  simt_delta_kernel<T, DPL><<<grid, 128, 0, st>>>((const T *)a.out, (const T *)a.dout, a.delta, rows, a.D);
  simt_dq_kernel<T, DPL><<<grid, 128, 0, st>>>((const T *)a.q, (const T *)a.kv, (const T *)a.ckv, a.sstart, a.status,
                                               a.lse, a.delta, (const T *)a.dout, (T *)a.dq, a.B, a.H, a.S, a.D, a.W,
                                               a.m, a.scale);
  const int Sc = (a.S + a.m - 1) / a.m;
  const long long keys = (long long)a.B * a.S + (long long)a.B * Sc;
  simt_dkey_kernel<T, DPL><<<(unsigned)((keys + 3) / 4), 128, 0, st>>>(
      (const T *)a.q, (const T *)a.kv, (const T *)a.ckv, a.sstart, a.status, a.lse, a.delta, (const T *)a.dout,
      (T *)a.dkv, (T *)a.dckv, a.B, a.H, a.S, a.D, a.W, a.m, a.scale);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t fwd_dispatch(const FwdArgs &a, cudaStream_t st) {
  if (a.D <= 32) return fwd_t<T, 1>(a, st);
  if (a.D <= 64) return fwd_t<T, 2>(a, st);
  if (a.D <= 128) return fwd_t<T, 4>(a, st);
  return fwd_t<T, 8>(a, st);
}

template <typename T>
static cudaError_t bwd_dispatch(const BwdArgs &a, cudaStream_t st) {
  if (a.D <= 32) return bwd_t<T, 1>(a, st);
  if (a.D <= 64) return bwd_t<T, 2>(a, st);
  if (a.D <= 128) return bwd_t<T, 4>(a, st);
  return bwd_t<T, 8>(a, st);
}

// fp32 mode only: bf16 runs on the tensor-core kernels (hca_api.cu rejects
// the bf16 shapes they do not take with HCA_ERR_UNSUPPORTED)
cudaError_t simt_fwd(const FwdArgs &a, cudaStream_t st) {
  return a.dtype == HCA_F32 ? fwd_dispatch<float>(a, st) : cudaErrorInvalidValue;
}

cudaError_t simt_bwd(const BwdArgs &a, cudaStream_t st) {
  return a.dtype == HCA_F32 ? bwd_dispatch<float>(a, st) : cudaErrorInvalidValue;
}

}  // namespace hca
