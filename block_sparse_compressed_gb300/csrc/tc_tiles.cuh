// tc_tiles.cuh -- query-tile geometry shared by the tensor-core kernels:
// head-packed query tiles, their key ranges cut into blocks, the 128-byte
// swizzled tile layout, and host helpers for TMA tensor maps.
//
// A query tile packs Pq consecutive positions x HG heads of one batch row
// into the 128 MMA rows (row r = head_in_group * Pq + p).  Every head of a
// position sees the same keys (one shared kv head: "[DeepSeek-V4] Implement
// Compressed Attention Layers", einsum review suggestions), so the tile's
// key set is the union of its Pq positions' intervals (hca_common.cuh).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "hca_common.cuh"
#include "tc_ptx.cuh"

namespace hca {
namespace tc {

constexpr int kRows = 128;        // MMA M: rows of a query tile / keys of a key block
constexpr int kHeadDim = 128;     // D of the tensor-core kernels
constexpr int kBlockKeys = 128;   // keys per block
constexpr int kTile = 32768;      // bytes of a 128 x 128 bf16 tile
constexpr int kHalfTile = 16384;  // one 64-column (128-byte) swizzled half

struct QTiling {
  const int32_t *sstart;  // [B,S] document starts, NULL = one document
  int B, H, S, W, m, Sc;
  int HG, Pq, groups, ntq;  // heads per tile, positions per tile, head groups, tiles per (b, group)
  long long ntiles;
};

struct Tile {
  int b, g, i0;
  int rlo, rhi, clo, chi;  // half-open key ranges (union over the tile's rows)
  int nraw, ncomp;         // blocks of <= kBlockKeys keys
};

// Tile u of the schedule: positions descending, so the tiles with the most
// compressed keys come first (the compressed range grows with the position).
__device__ __forceinline__ void tile_coords(const QTiling &p, long long u, Tile &t) {
  const long long per = (long long)p.B * p.groups;
  const int tq = p.ntq - 1 - (int)(u / per);
  const int rem = (int)(u % per);
  t.b = rem / p.groups;
  t.g = rem % p.groups;
  t.i0 = tq * p.Pq;
}

// Warp-cooperative union of the row intervals of positions [i0, i0+Pq).
__device__ __forceinline__ void tile_ranges_warp(const QTiling &p, Tile &t, int lane) {
  int rlo = 0x7fffffff, rhi = -1, clo = 0x7fffffff, chi = -1;
  for (int q = lane; q < p.Pq; q += 32) {
    RowIv iv = row_interval(p.sstart, t.b, p.S, t.i0 + q, p.W, p.m);
    if (!iv.valid) continue;
    rlo = min(rlo, iv.rlo);
    rhi = max(rhi, iv.rhi);
    if (iv.chi >= iv.clo) {
      clo = min(clo, iv.clo);
      chi = max(chi, iv.chi);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    rlo = min(rlo, __shfl_xor_sync(0xffffffffu, rlo, off));
    rhi = max(rhi, __shfl_xor_sync(0xffffffffu, rhi, off));
    clo = min(clo, __shfl_xor_sync(0xffffffffu, clo, off));
    chi = max(chi, __shfl_xor_sync(0xffffffffu, chi, off));
  }
  t.rlo = rhi < 0 ? 0 : rlo;
  t.rhi = rhi < 0 ? 0 : rhi + 1;
  t.clo = chi < 0 ? 0 : clo;
  t.chi = chi < 0 ? 0 : chi + 1;
  t.nraw = (t.rhi - t.rlo + kBlockKeys - 1) / kBlockKeys;
  t.ncomp = (t.chi - t.clo + kBlockKeys - 1) / kBlockKeys;
}

// Broadcast a tile's ranges from lane 0: the compiler then treats them and
// everything derived from them as warp-uniform (uniform registers).
__device__ __forceinline__ void uniform_tile(Tile &t) {
  t.rlo = __shfl_sync(0xffffffffu, t.rlo, 0);
  t.rhi = __shfl_sync(0xffffffffu, t.rhi, 0);
  t.clo = __shfl_sync(0xffffffffu, t.clo, 0);
  t.chi = __shfl_sync(0xffffffffu, t.chi, 0);
  t.nraw = __shfl_sync(0xffffffffu, t.nraw, 0);
  t.ncomp = __shfl_sync(0xffffffffu, t.ncomp, 0);
}

// Block j of a tile: raw kv blocks first, then compressed ckv blocks.
__device__ __forceinline__ void block_of(const Tile &t, int j, bool &comp, int &start, int &n) {
  if (j < t.nraw) {
    comp = false;
    start = t.rlo + j * kBlockKeys;
    n = min(kBlockKeys, t.rhi - start);
  } else {
    comp = true;
    start = t.clo + (j - t.nraw) * kBlockKeys;
    n = min(kBlockKeys, t.chi - start);
  }
}

// Bits c of a 64-bit mask for which lo <= base + c <= hi.
__device__ __forceinline__ uint64_t range_mask64(int lo, int hi, int base) {
  const int l = max(lo - base, 0), h = min(hi - base, 63);
  if (h < l) return 0ull;
  const int w = h - l + 1;
  return (w >= 64 ? ~0ull : ((1ull << w) - 1ull)) << l;
}

// Byte offset of 16-byte chunk `chunk16` (0..15 over both halves) of row
// `row` in a 128-row x 256-byte tile stored as two 128B-swizzled halves --
// the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B and the UMMA
// descriptors read (chunk index XOR row mod 8 inside each 1 KB atom).
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk16) {
  const int half = chunk16 >> 3, c = chunk16 & 7;
  return (uint32_t)(half * kHalfTile + row * 128 + ((c ^ (row & 7)) << 4));
}

// UMMA descriptor offsets (in the descriptor's 16-byte units) of k-step k
// (16 bf16 of K) inside a 128-row tile stored as two 128B-swizzled halves:
// K-major operands advance 32 bytes inside a half, then jump to the next half;
// MN-major operands (K along the rows) advance 16 rows = 2048 bytes.
__host__ __device__ constexpr uint64_t kmaj_step(int k) {
  return (uint64_t)(((k >> 2) * kHalfTile + (k & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t mnmaj_step(int k) { return (uint64_t)((k * 2048) >> 4); }
__host__ __device__ constexpr uint64_t desc_bytes(uint32_t bytes) { return (uint64_t)(bytes >> 4); }

// Bounded wait whose outcome is the same for the whole warp, so that a warp
// never splits around warp-collective tcgen05.ld / tcgen05.st.
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort, int32_t *status,
                                          uint32_t spin = 0) {
  const bool ok = mbar_wait(bar, parity, abort, status, kWaitLimitNs, spin);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 3-D bf16 map {inner, mid, outer} (contiguous) with a {64, box1, box2} box
// and 128-byte swizzle; out-of-range elements read as zero.
inline bool make_map_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t mid, uint64_t outer,
                          uint32_t box1, uint32_t box2) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

inline int heads_per_tile(int H) { return H >= kRows ? kRows : H; }

inline bool tc_shape_ok(int H, int D, int dtype) {
  if (dtype != HCA_BF16 || D != kHeadDim || H < 1) return false;
  if (H <= kRows) return (kRows % H) == 0;
  return (H % kRows) == 0;
}

inline QTiling make_qtiling(const int32_t *sstart, int B, int H, int S, int W, int m) {
  QTiling q;
  q.sstart = sstart;
  q.B = B; q.H = H; q.S = S; q.W = W; q.m = m;
  q.Sc = (S + m - 1) / m;
  q.HG = heads_per_tile(H);
  q.Pq = kRows / q.HG;
  q.groups = H / q.HG;
  q.ntq = (S + q.Pq - 1) / q.Pq;
  q.ntiles = (long long)B * q.groups * q.ntq;
  return q;
}

}  // namespace tc
}  // namespace hca
