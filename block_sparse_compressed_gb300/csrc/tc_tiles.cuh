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

// A tile's keys form one list of columns: the compressed entries
// [clo, clo + cpad) (cpad = chi - clo rounded up to 16; the extra entries are
// masked) followed by the raw keys [rlo, rhi).  Blocks are consecutive
// 128-column slices of that list, so the few raw keys past a 128-key window
// share a block with the last compressed entries instead of taking a block
// of their own.
struct Tile {
  int b, g, i0;
  int rlo, rhi, clo, chi;  // half-open key ranges (union over the tile's rows)
  int cpad;                // column where the raw keys start (multiple of 16)
  int ncols, nb;           // columns of the key list, blocks of <= kBlockKeys columns
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
  t.cpad = (t.chi - t.clo + 15) & ~15;
  t.ncols = t.cpad + (t.rhi - t.rlo);
  t.nb = (t.ncols + kBlockKeys - 1) / kBlockKeys;
}

// Broadcast a tile's ranges from lane 0: the compiler then treats them and
// everything derived from them as warp-uniform (uniform registers).
__device__ __forceinline__ void uniform_tile(Tile &t) {
  t.rlo = __shfl_sync(0xffffffffu, t.rlo, 0);
  t.rhi = __shfl_sync(0xffffffffu, t.rhi, 0);
  t.clo = __shfl_sync(0xffffffffu, t.clo, 0);
  t.chi = __shfl_sync(0xffffffffu, t.chi, 0);
  t.cpad = __shfl_sync(0xffffffffu, t.cpad, 0);
  t.ncols = __shfl_sync(0xffffffffu, t.ncols, 0);
  t.nb = __shfl_sync(0xffffffffu, t.nb, 0);
}

// Block j of a tile: columns [128 j, 128 j + n) of the key list, of which
// the first nc (a multiple of 16) are compressed entries and the rest raw keys.
__device__ __forceinline__ void block_cols(const Tile &t, int j, int &n, int &nc) {
  const int c0 = j * kBlockKeys;
  n = min(kBlockKeys, t.ncols - c0);
  nc = min(max(t.cpad - c0, 0), n);
}

// Columns of block j that a row sees, as two inclusive ranges: [a1, b1] of
// compressed entries and [a2, b2] of raw keys (either may be empty; b1 < a2).
__device__ __forceinline__ void row_cols(const Tile &t, const RowIv &iv, int j, int n, int nc, int &a1, int &b1,
                                         int &a2, int &b2) {
  if (!iv.valid) {
    a1 = a2 = 0;
    b1 = b2 = -1;
    return;
  }
  const int c0 = j * kBlockKeys;
  a1 = max(iv.clo - t.clo - c0, 0);
  b1 = min(iv.chi - t.clo - c0, nc - 1);
  const int off = t.rlo + c0 - t.cpad;  // raw key of column c: off + c
  a2 = max(iv.rlo - off, nc);
  b2 = min(iv.rhi - off, n - 1);
}

// Bytes that load_block delivers for a block of n columns, nc compressed,
// of rows with kHalves 64-column halves (head dim 64 * kHalves).
template <int kHalves = 2>
__device__ __forceinline__ uint32_t block_load_bytes(int n, int nc) {
  if (nc == n || nc == 0) return (uint32_t)(kHalves * kHalfTile);
  return (uint32_t)(nc / 16 + (n - nc + 15) / 16) * 16u * 128u * kHalves;
}

// TMA loads of block j's key rows into a 128-row tile at dst (two 64-column
// swizzled halves).  A block of one kind is one 128-row box per half; a block
// that holds both kinds is loaded in 16-row boxes (2 KB, so every box starts
// on a 1 KB swizzle atom), compressed rows first.
template <int kHalves = 2>
__device__ __forceinline__ void load_block(const Tile &t, int j, int n, int nc, const CUtensorMap *kv,
                                           const CUtensorMap *ckv, const CUtensorMap *kv16, const CUtensorMap *ckv16,
                                           uint64_t *bar, uint8_t *dst) {
  const int c0 = j * kBlockKeys;
  const int off = t.rlo + c0 - t.cpad;
  if (nc == n) {
#pragma unroll
    for (int hh = 0; hh < kHalves; ++hh) tma_load_3d(ckv, bar, dst + hh * kHalfTile, 64 * hh, t.clo + c0, t.b);
  } else if (nc == 0) {
#pragma unroll
    for (int hh = 0; hh < kHalves; ++hh) tma_load_3d(kv, bar, dst + hh * kHalfTile, 64 * hh, off, t.b);
  } else {
    for (int r = 0; r < nc; r += 16) {
#pragma unroll
      for (int hh = 0; hh < kHalves; ++hh)
        tma_load_3d(ckv16, bar, dst + hh * kHalfTile + r * 128, 64 * hh, t.clo + c0 + r, t.b);
    }
    for (int r = nc; r < n; r += 16) {
#pragma unroll
      for (int hh = 0; hh < kHalves; ++hh)
        tma_load_3d(kv16, bar, dst + hh * kHalfTile + r * 128, 64 * hh, off + r, t.b);
    }
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

// ---------------------------------------------------------------------------
// CSA key blocks: compressed columns are the tile's union of selected
// entries (gathered), raw columns as in HCA (TMA)
// ---------------------------------------------------------------------------
// Bytes the TMA delivers for the raw rows of block j (n columns, nc of them
// gathered compressed entries).
__device__ __forceinline__ uint32_t raw_load_bytes(int n, int nc) {
  if (nc == 0) return (uint32_t)kTile;
  return (uint32_t)((n - nc + 15) / 16) * 16u * 256u;
}

// TMA loads of the raw rows [nc, n) of block j (16-row boxes after the
// compressed rows, one 128-row box per half when the block is all raw).
__device__ __forceinline__ void load_block_raw(const Tile &t, int j, int n, int nc, const CUtensorMap *kv,
                                               const CUtensorMap *kv16, uint64_t *bar, uint8_t *dst) {
  const int c0 = j * kBlockKeys;
  const int off = t.rlo + c0 - t.cpad;
  if (nc == 0) {
    tma_load_3d(kv, bar, dst, 0, off, t.b);
    tma_load_3d(kv, bar, dst + kHalfTile, 64, off, t.b);
    return;
  }
  for (int r = nc; r < n; r += 16) {
    tma_load_3d(kv16, bar, dst + r * 128, 0, off + r, t.b);
    tma_load_3d(kv16, bar, dst + kHalfTile + r * 128, 64, off + r, t.b);
  }
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
                                          uint64_t limit_ns) {
  const bool ok = mbar_wait(bar, parity, abort, status, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// A wait on a barrier that nothing ever arrives at: it always runs out after
// limit_ns and takes the same abort path as a real wait that gave up.  The
// failure-path tests reach it through hca_test_inject (HCA_INJECT_STALL).
__device__ __forceinline__ void injected_stall(uint64_t *never_bar, volatile int *abort, int32_t *status,
                                               uint64_t limit_ns) {
  (void)wait_warp(never_bar, 0, abort, status, limit_ns);
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

// 2-D row view {inner, rows} of a bf16 tensor with a one-row, 64-column box
// (128 bytes, 128B-swizzled): the map of the TMA gather4 loads.
inline bool make_map_rows_bf16(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Heads packed into one 128-row tile: the largest power of two that divides
// both H and 128, so any head count tiles exactly (H = 48: 16 heads x 8
// positions per tile, three head groups).
inline int heads_per_tile(int H) {
  int hg = 1;
  while (hg < kRows && H % (2 * hg) == 0) hg *= 2;
  return hg;
}

inline bool tc_shape_ok(int H, int D, int dtype) { return dtype == HCA_BF16 && (D == 64 || D == 128) && H >= 1; }

// Dynamic shared-memory limit of a kernel, raised once per device: the
// attribute belongs to the (function, device) pair, so a process that drives
// several GPUs needs it on each of them.  Guarded for concurrent first calls.
class SmemAttrOnce {
 public:
  cudaError_t ensure(const void *kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu_);
    if (done_[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  static constexpr int kMaxDev = 64;
  std::mutex mu_;
  bool done_[kMaxDev] = {};
};

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
