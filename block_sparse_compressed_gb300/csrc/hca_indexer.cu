// hca_indexer.cu -- the Lightning Indexer: index scores of the compressed
// entries per query, sentinel masking and top-k selection, feeding CSA.
//
// "[DeepSeek-V4] Implement Compressed Attention Layers": the LightningIndexer
// implements sentinel masking (Description), and its scores are the matmul
// of the indexer queries with the transposed compressed kv, [B, S, H, W] per
// head (review suggestion on the indexer); "Add HCA Static Compilation for
// Splash Attention [Deepseek v4]", Description: CSA needs a top-k step.
// The per-head scores are combined by a weighted sum over heads:
//   score[b,s,j] = sum_h w[b,s,h] <qi[b,s,h,:], ki[b,j,:]>
//                = < sum_h w[b,s,h] qi[b,s,h,:], ki[b,j,:] >
// (linear in the query, so the heads collapse into one query vector first;
// the pages name no activation between the two steps).  Entry j is visible
// to query i under the HCA compressed rule (window complete at i, inside i's
// document, hca_common.cuh), a contiguous range [clo(i), chi(i)]; every
// other entry carries the sentinel -inf and is never selected.  top-k keeps
// the k largest scores (ties: smaller entry index), written in ascending
// entry order and padded with -1.
//
// Three kernels per chunk of query rows:
//   1. collapse   q~[b,s,:] = sum_h w qi  (fp32 accumulation -> bf16), HBM-bound
//   2. scores     tcgen05 GEMM of 128-position tiles of q~ against 128-entry
//                 blocks of ki (TMA -> smem -> MMA -> TMEM -> fp32 rows in a
//                 chunk buffer); blocks past a tile's last visible entry are
//                 skipped
//   3. top-k      one CTA per query row: 4-pass radix select (8-bit digits)
//                 on order-preserving integer keys in shared memory, then an
//                 ordered compaction of the winners
#include <cuda_bf16.h>

#include "hca_common.cuh"
#include "hca_internal.h"
#include "tc_ptx.cuh"
#include "tc_tiles.cuh"

namespace hca {
using namespace tc;

namespace {

// ---------------------------------------------------------------------------
// 1. head collapse
// ---------------------------------------------------------------------------
constexpr int kCollapseWarps = 8;

__global__ void __launch_bounds__(32 * kCollapseWarps)
    hca_index_collapse_kernel(const __nv_bfloat16 *__restrict__ qi, const float *__restrict__ w,
                              __nv_bfloat16 *__restrict__ qc, long long rows, int Hi) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * kCollapseWarps + (threadIdx.x >> 5);
  if (r >= rows) return;
  // lane holds dims [4 lane, 4 lane + 4) of the 128
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const __nv_bfloat16 *base = qi + (size_t)r * Hi * kHeadDim;
  const float *wr = w + (size_t)r * Hi;
  for (int h = 0; h < Hi; ++h) {
    const float wh = __ldg(wr + h);
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(base + (size_t)h * kHeadDim) + lane);
    acc[0] = fmaf(wh, __uint_as_float(v.x << 16), acc[0]);
    acc[1] = fmaf(wh, __uint_as_float(v.x & 0xffff0000u), acc[1]);
    acc[2] = fmaf(wh, __uint_as_float(v.y << 16), acc[2]);
    acc[3] = fmaf(wh, __uint_as_float(v.y & 0xffff0000u), acc[3]);
  }
  uint2 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  reinterpret_cast<uint2 *>(qc + (size_t)r * kHeadDim)[lane] = o;
}

// ---------------------------------------------------------------------------
// 2. scores: 128 query positions x 128 entries per MMA tile
// ---------------------------------------------------------------------------
namespace isk {
constexpr int kStages = 2;
constexpr int kThreads = 192;  // warps 0-3 epilogue (one TMEM lane quarter each), 4 TMA, 5 MMA
constexpr int kOffA = 0, kOffB = kTile;
// output staging: two buffers (one per accumulator), each four 32-column
// fp32 quarters of 128 rows x 128 bytes, 128B-swizzled for the TMA store
constexpr int kQuarter = kRows * 128;
constexpr int kStageBuf = 4 * kQuarter;
constexpr int kOffStage = kTile + kStages * kTile;
constexpr int kSmemBytes = kOffStage + 2 * kStageBuf + 1024;
constexpr int kTmemCols = 256;  // two 128-column accumulators
}  // namespace isk

// 3-D view {ld, rows, B} of the fp32 score chunk with a 32-column, 128-row
// box (128 bytes per row, 128B-swizzled): the map of the score stores.
static bool make_map_scores(CUtensorMap *m, float *buf, uint64_t ld, uint64_t rows, uint64_t B) {
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {ld, rows, B};
  cuuint64_t strides[2] = {ld * 4, ld * rows * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)kRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, buf, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

struct ScoreParams {
  const int32_t *sstart;  // NULL = one document per row
  float *buf;             // [B][rows][ld] fp32 chunk buffer
  int B, S, m, Sc, row0, rows, ld;
  int groups;             // CTAs per query tile, each taking a share of its entry blocks
  int32_t *status;
  uint64_t wait_ns;
};

struct ScoreBars {
  uint64_t a_full;
  uint64_t b_full[isk::kStages], b_empty[isk::kStages];
  uint64_t acc_full[2], acc_free[2], drain, epi;
  uint32_t tmem_base;
  int abort;
};

// Last entry (exclusive) any position of [p0, p1) can see: entries complete
// at position p1 - 1.
__device__ __forceinline__ int entries_upto(int p1, int m) { return p1 / m; }

__global__ void __launch_bounds__(isk::kThreads, 1)
    hca_index_score_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                           const __grid_constant__ CUtensorMap map_s, const ScoreParams p) {
  using namespace isk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ ScoreBars bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int *abort_flag = &bars.abort;
  // tile: batch row b, positions [p0, p0 + 128) of the chunk; this CTA takes
  // the entry blocks [j0, j0 + nblk) of it (group g of p.groups), so that a
  // chunk of few tiles still fills the GPU
  const int tiles_per_b = (p.rows + kRows - 1) / kRows;
  const int tile = blockIdx.x / p.groups, grp = blockIdx.x % p.groups;
  const int b = tile / tiles_per_b;
  const int p0 = p.row0 + (tile % tiles_per_b) * kRows;
  const int p1 = min(p0 + kRows, min(p.row0 + p.rows, p.S));
  const int nent = min(entries_upto(p1, p.m), p.Sc);
  const int nblk_tile = (nent + kBlockKeys - 1) / kBlockKeys;
  const int per = (nblk_tile + p.groups - 1) / p.groups;
  const int j0 = min(grp * per, nblk_tile);
  const int nblk = min(j0 + per, nblk_tile) - j0;  // local block j is entry block j0 + j

  if (tid == 0) {
    mbar_init(&bars.a_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.b_full[s], 1);
      mbar_init(&bars.b_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.acc_full[x], 1);
      mbar_init(&bars.acc_free[x], 128);
    }
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.epi, 128);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA
    bool ok = true;
    int b_par[kStages] = {-1, -1};
    if (lane == 0 && nblk > 0) {
      mbar_arrive_expect_tx(&bars.a_full, kTile);
      tma_load_3d(&map_q, &bars.a_full, smem + kOffA, 0, p0, b);
      tma_load_3d(&map_q, &bars.a_full, smem + kOffA + kHalfTile, 64, p0, b);
      for (int j = 0; ok && j < nblk; ++j) {
        const int s = j % kStages;
        if (j >= kStages) ok = mbar_wait(&bars.b_empty[s], ((j / kStages) - 1) & 1, abort_flag, p.status, p.wait_ns);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.b_full[s], kTile);
        tma_load_3d(&map_k, &bars.b_full[s], smem + kOffB + s * kTile, 0, (j0 + j) * kBlockKeys, b);
        tma_load_3d(&map_k, &bars.b_full[s], smem + kOffB + s * kTile + kHalfTile, 64, (j0 + j) * kBlockKeys, b);
        b_par[s] = (j / kStages) & 1;
      }
      if (!ok) {
        volatile int never = 0;
        mbar_wait(&bars.a_full, 0, &never, p.status, 100000000ull);
        for (int s = 0; s < kStages; ++s)
          if (b_par[s] >= 0) mbar_wait(&bars.b_full[s], b_par[s], &never, p.status, 100000000ull);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA
    const uint64_t da = smem_desc_sw128(smem_u32(smem + kOffA), 16, 1024);
    const uint64_t db0 = smem_desc_sw128(smem_u32(smem + kOffB), 16, 1024);
    const uint32_t idesc = idesc_bf16_f32(kRows, kBlockKeys, false, false);
    bool ok = nblk > 0, issued = false;
    if (ok) ok = wait_warp(&bars.a_full, 0, abort_flag, p.status, p.wait_ns);
    for (int j = 0; ok && j < nblk; ++j) {
      const int s = j % kStages, x = j & 1;
      ok = wait_warp(&bars.b_full[s], (j / kStages) & 1, abort_flag, p.status, p.wait_ns);
      if (ok && j >= 2) ok = wait_warp(&bars.acc_free[x], ((j / 2) - 1) & 1, abort_flag, p.status, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const uint64_t db = db0 + desc_bytes(s * kTile);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          mma_ss(tmem + x * 128, da + kmaj_step(k), db + kmaj_step(k), idesc, k > 0);
        mma_commit(&bars.acc_full[x]);
        mma_commit(&bars.b_empty[s]);
      }
      __syncwarp();
      issued = true;
    }
    if (!ok && issued) {
      volatile int never = 0;
      if (elect_one()) mma_commit(&bars.drain);
      __syncwarp();
      if (lane == 0) mbar_wait(&bars.drain, 0, &never, p.status, 100000000ull);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // thread r = row r of the tile (TMEM lane r) stages its 128 scores of a
    // block (four 128B-swizzled quarters, conflict-free); thread 0 stores the
    // block with four TMA tensor stores (rows past the chunk are clipped).
    // Staging buffer j & 1 is written again two blocks later: before the
    // rendezvous of block j, thread 0 waits until block j - 1's stores have
    // read their buffer, so every thread may write it in block j + 1.
    const int r = tid;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t epi_phase = 0;
    // bounded rendezvous of the four epilogue warps (an abort ends it too)
    auto rendezvous = [&]() -> bool {
      mbar_arrive(&bars.epi);
      const bool rr = wait_warp(&bars.epi, epi_phase & 1, abort_flag, p.status, p.wait_ns);
      ++epi_phase;
      return rr;
    };
    for (int j = 0; j < nblk; ++j) {
      const int x = j & 1;
      if (!wait_warp(&bars.acc_full[x], (j / 2) & 1, abort_flag, p.status, p.wait_ns)) break;
      tc_fence_after();
      uint8_t *buf = smem + kOffStage + x * kStageBuf;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        tmem_ld32(lane_addr + x * 128 + 32 * q, v);
        tmem_wait_ld();
        uint8_t *rowp = buf + q * kQuarter + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4 *>(rowp + ((c ^ (r & 7)) << 4)) = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      }
      tc_fence_before();
      mbar_arrive(&bars.acc_free[x]);
      fence_async_smem();
      if (tid == 0) bulk_wait_read0();  // block j - 1's stores have read the other buffer
      if (!rendezvous()) break;
      if (tid == 0) {
        const int cx = (j0 + j) * kBlockKeys, cy = p0 - p.row0;
#pragma unroll
        for (int q = 0; q < 4; ++q) tma_store_3d(&map_s, buf + q * kQuarter, cx + 32 * q, cy, b);
        bulk_commit();
      }
    }
    if (tid == 0) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// 3. top-k per query row
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 256;
constexpr int kRadixBins = 2048;  // 11-bit digits
// a query row's visible scores are staged in shared memory (with the 8 KB
// histogram, within the 227 KB a block may use)
constexpr int kMaxEntries = 55296;

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of one int per thread; returns the block total.
__device__ __forceinline__ int block_excl_scan(int v, int &excl, int *wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  int base = 0, total = 0;
#pragma unroll
  for (int k = 0; k < kTopkThreads / 32; ++k) {
    const int s = wsum[k];
    if (k < wid) base += s;
    total += s;
  }
  __syncthreads();
  excl = base + x - v;
  return total;
}

struct TopkParams {
  const float *buf;
  const int32_t *sstart;
  const int32_t *status;  // non-zero (segment ids out of order): nothing is selected
  int32_t *sel;      // [B,S,k]
  float *scores;     // optional [B,S,Sc] with -inf outside the visible range
  int B, S, m, Sc, row0, rows, ld, k;
};

// Digit of a radix pass: scanning the histogram h (nbins = dmask + 1 bins)
// from the top, the bin where the running count reaches rem.  Thread t owns
// the 8 bins [top - 8t - 7, top - 8t]; the thread holding the crossing bin
// writes the digit, the winners still to place inside it and the bin's size.
__device__ __forceinline__ void select_digit(const int *h, int dmask, int rem, int *wsum, int *sh) {
  const int tid = threadIdx.x;
  int c[8], sum = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int d = dmask - (tid * 8 + q);
    c[q] = d >= 0 ? h[d] : 0;
    sum += c[q];
  }
  int before;
  block_excl_scan(sum, before, wsum);
  if (before < rem && before + sum >= rem) {
    int run = before;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (run + c[q] >= rem) {
        sh[0] = dmask - (tid * 8 + q);
        sh[1] = rem - run;
        sh[2] = c[q];
        break;
      }
      run += c[q];
    }
  }
  __syncthreads();
}

// The same for a histogram of at most 256 bins, by warp 0 alone (eight bins
// per lane, one warp scan): the other warps only wait at the barrier.
__device__ __forceinline__ void select_digit_warp(const int *h, int dmask, int rem, int *sh) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    int c[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int d = dmask - (tid * 8 + q);
      c[q] = d >= 0 ? h[d] : 0;
      sum += c[q];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    const int before = incl - sum;
    if (before < rem && incl >= rem) {
      int run = before;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (run + c[q] >= rem) {
          sh[0] = dmask - (tid * 8 + q);
          sh[1] = rem - run;
          sh[2] = c[q];
          break;
        }
        run += c[q];
      }
    }
  }
  __syncthreads();
}

// Candidates: entries whose top digit is the k-th largest key's, when they
// fit beside the small histogram in the top digit's histogram space.
constexpr int kSmallBins = 128;  // 7-bit digits over the candidates
constexpr int kCandCap = kRadixBins - kSmallBins;
// keys at or above a sampled threshold, listed per warp: 8-bit digits over them
constexpr int kByteBins = 256;
constexpr int kListCap = (kRadixBins - kByteBins) / (kTopkThreads / 32);

__global__ void __launch_bounds__(kTopkThreads, 5) hca_index_topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t keys[];
  // the sample's top-digit histogram; then a small histogram and the
  // warps' lists of keys at or above the threshold; on the exact path the
  // top-digit histogram of every key, then a small histogram and the list of
  // its bin's keys, or the wide histogram again
  __shared__ int area[kRadixBins];
  __shared__ int wsum[kTopkThreads / 32];
  __shared__ int sh[3];
  __shared__ int ncand;
  constexpr int kWarps = kTopkThreads / 32;
  __shared__ int wgt[kWarps], weq[kWarps], wlist[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int b = blockIdx.x / p.rows;
  const int i = p.row0 + blockIdx.x % p.rows;
  if (i >= p.S) return;
  const float *row = p.buf + ((size_t)b * p.rows + (i - p.row0)) * p.ld;
  int32_t *out = p.sel + ((size_t)b * p.S + i) * p.k;
  const RowIv iv = row_interval(p.sstart, b, p.S, i, 1, p.m);
  const int lo = iv.valid ? iv.clo : 0;
  const int hi = iv.valid ? min(iv.chi, p.Sc - 1) : -1;
  const int n = hi >= lo ? hi - lo + 1 : 0;
  if (p.scores) {
    float *sr = p.scores + ((size_t)b * p.S + i) * p.Sc;
    for (int j = tid; j < p.Sc; j += kTopkThreads) sr[j] = (j >= lo && j <= hi) ? row[j] : -INFINITY;
  }
  if (*(volatile const int32_t *)p.status != 0) {
    for (int t = tid; t < p.k; t += kTopkThreads) out[t] = -1;
    return;
  }
  if (n <= p.k) {
    for (int t = tid; t < p.k; t += kTopkThreads) out[t] = t < n ? lo + t : -1;
    return;
  }
  // Every eighth key (by entry index) first, into a histogram of the top
  // 11-bit digit: eight strided loads in flight per thread; they touch every
  // 32-byte sector of the row once, so the staging below reads it from L2.
  for (int d = tid; d < kRadixBins; d += kTopkThreads) area[d] = 0;
  if (tid == 0) ncand = 0;
  if (tid < kWarps) {
    wgt[tid] = 0;
    weq[tid] = 0;
  }
  __syncthreads();
  constexpr int kInFlight = 8;
  const float *src = row + lo;
  const int ns = (n + 7) >> 3;
  for (int j0 = 0; j0 < ns; j0 += kInFlight * kTopkThreads) {
    uint32_t kv[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int j = j0 + u * kTopkThreads + tid;
      kv[u] = j < ns ? fkey(src[8 * j]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u)
      if (j0 + u * kTopkThreads + tid < ns) atomicAdd(&area[kv[u] >> 21], 1);
  }
  __syncthreads();
  // Threshold: the lower edge of the top-digit bin where the sample's count
  // from the top reaches its share of k plus a margin (about three standard
  // deviations of that count), so that normally at least k keys lie at or
  // above it; the sample's own digits are exact, only the count is an
  // estimate.
  const int want = min(ns, (int)(((long long)p.k * 115 * ns + 100LL * n - 1) / (100LL * n)) + 16);
  select_digit(area, kRadixBins - 1, want, wsum, sh);
  const uint32_t tau = (uint32_t)sh[0] << 21;
  __syncthreads();  // everyone has read sh and the histogram
  // Warp w owns the keys [w L, (w + 1) L): it stages them (eight loads in
  // flight per lane, 128 bytes per warp load) and lists the ones at or above
  // the threshold, in entry order, in its own part of the area.
  const int L = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int s0 = min(wid * L, n), s1 = min(s0 + L, n);
  const uint32_t lt = (1u << lane) - 1u;
  int *lists = area + kByteBins;
  int *mine = lists + wid * kListCap;
  int wn = 0;
  for (int c0 = s0; c0 < s1; c0 += kInFlight * 32) {
    uint32_t kv[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int t = c0 + u * 32 + lane;
      kv[u] = t < s1 ? fkey(src[t]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int t = c0 + u * 32 + lane;
      const bool c = t < s1 && kv[u] >= tau;
      if (t < s1) keys[t] = kv[u];
      const unsigned bc = __ballot_sync(0xffffffffu, c);
      const int slot = wn + __popc(bc & lt);
      if (c && slot < kListCap) mine[slot] = t;
      wn += __popc(bc);
    }
  }
  if (lane == 0) wlist[wid] = wn;
  __syncthreads();
  int nlisted = 0;
  bool fits = true;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    nlisted += wlist[w];
    fits = fits && wlist[w] <= kListCap;
  }
  uint32_t prefix = 0, mask = 0;
  int rem = p.k;  // winners still to place at or below the current prefix
  if (fits && nlisted >= p.k) {
    // the k-th largest key is among the listed ones (every other key is
    // below the threshold): four 8-bit digits over the lists
    int *hs = area;
    // listed key c of the concatenated lists: warp w = the last with
    // start[w] <= c, slot c - start[w] (all threads share every pass evenly)
    int start[kWarps];
    {
      int run = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        start[w] = run;
        run += wlist[w];
      }
    }
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int d = tid; d < kByteBins; d += kTopkThreads) hs[d] = 0;
      __syncthreads();
      for (int c = tid; c < nlisted; c += kTopkThreads) {
        int w = 0, sw = 0;
#pragma unroll
        for (int x = 1; x < kWarps; ++x)
          if (c >= start[x]) {
            w = x;
            sw = start[x];
          }
        const uint32_t kv = keys[lists[w * kListCap + (c - sw)]];
        if ((kv & mask) == prefix) atomicAdd(&hs[(kv >> shift) & (kByteBins - 1)], 1);
      }
      __syncthreads();
      // the next pass zeroes hs only after two more barriers, and sh is
      // rewritten only after them: no barrier after reading sh
      select_digit_warp(hs, kByteBins - 1, rem, sh);
      prefix |= (uint32_t)sh[0] << shift;
      mask |= (uint32_t)(kByteBins - 1) << shift;
      rem = sh[1];
    }
    // ordered write from the lists: winners are the listed keys above
    // prefix plus the rem keys equal to it with the smallest entry index
    int gt = 0, eqc = 0;
    for (int c0 = 0; c0 < wn; c0 += 32) {
      const int c = c0 + lane;
      const uint32_t kv = c < wn ? keys[mine[c]] : 0u;
      gt += __popc(__ballot_sync(0xffffffffu, c < wn && kv > prefix));
      eqc += __popc(__ballot_sync(0xffffffffu, c < wn && kv == prefix));
    }
    if (lane == 0) {
      wgt[wid] = gt;
      weq[wid] = eqc;
    }
    __syncthreads();
    int gt_run = 0, eq_run = 0;
    for (int w = 0; w < wid; ++w) {
      gt_run += wgt[w];
      eq_run += weq[w];
    }
    int placed = gt_run + min(eq_run, rem);
    for (int c0 = 0; c0 < wn; c0 += 32) {
      const int c = c0 + lane;
      const int t = c < wn ? mine[c] : 0;
      const uint32_t kv = c < wn ? keys[t] : 0u;
      const bool eq = c < wn && kv == prefix;
      const uint32_t beq = __ballot_sync(0xffffffffu, eq);
      const bool take = c < wn && (kv > prefix || (eq && eq_run + __popc(beq & lt) < rem));
      const uint32_t btake = __ballot_sync(0xffffffffu, take);
      if (take) out[placed + __popc(btake & lt)] = lo + t;
      placed += __popc(btake);
      eq_run += __popc(beq);
    }
    return;
  } else {
    // the sample missed: the exact top digit from every key
    for (int d = tid; d < kRadixBins; d += kTopkThreads) area[d] = 0;
    if (tid == 0) ncand = 0;
    __syncthreads();
    for (int t0 = 0; t0 < n; t0 += kTopkThreads) {
      const int t = t0 + tid;
      const uint32_t dg = t < n ? keys[t] >> 21 : 0xffffffffu;
      // lanes whose digit agrees add once per group (match.any): bins that
      // most keys share do not serialise the block on one address
      const unsigned peers = __match_any_sync(0xffffffffu, dg);
      if (t < n && lane == __ffs(peers) - 1) atomicAdd(&area[dg], __popc(peers));
    }
    __syncthreads();
    select_digit(area, kRadixBins - 1, p.k, wsum, sh);
    const uint32_t d0 = (uint32_t)sh[0];
    prefix = d0 << 21;
    mask = 0x7ffu << 21;
    rem = sh[1];
    const bool use_cand = sh[2] <= kCandCap;
    __syncthreads();  // everyone has read sh and the histogram
    if (use_cand) {
      int *hs = area;
      int *cand = area + kSmallBins;
      // one sweep: keys above the top digit per warp, the bin's keys listed
      int above = 0;
      for (int t0 = s0; t0 < s1; t0 += 32) {
        const int t = t0 + lane;
        const uint32_t dg = t < s1 ? keys[t] >> 21 : 0u;
        above += __popc(__ballot_sync(0xffffffffu, t < s1 && dg > d0));
        const bool c = t < s1 && dg == d0;
        const unsigned bc = __ballot_sync(0xffffffffu, c);
        int cb = 0;
        if (lane == 0 && bc) cb = atomicAdd(&ncand, __popc(bc));
        cb = __shfl_sync(0xffffffffu, cb, 0);
        if (c) cand[cb + __popc(bc & lt)] = t;
      }
      if (lane == 0) wgt[wid] = above;
      // the remaining 21 bits in three 7-bit digits, over the bin only
#pragma unroll 1
      for (int pass = 0; pass < 3; ++pass) {
        const int shift = 14 - 7 * pass;
        for (int d = tid; d < kSmallBins; d += kTopkThreads) hs[d] = 0;
        __syncthreads();
        const int nc = ncand;
        for (int c = tid; c < nc; c += kTopkThreads) {
          const uint32_t kv = keys[cand[c]];
          if ((kv & mask) == prefix) atomicAdd(&hs[(kv >> shift) & (kSmallBins - 1)], 1);
        }
        __syncthreads();
        select_digit_warp(hs, kSmallBins - 1, rem, sh);
        prefix |= (uint32_t)sh[0] << shift;
        mask |= (uint32_t)(kSmallBins - 1) << shift;
        rem = sh[1];
      }
      // the bin's keys above and equal to the k-th key, per owning warp
      const int nc = ncand;
      for (int c = tid; c < nc; c += kTopkThreads) {
        const int t = cand[c];
        const uint32_t kv = keys[t];
        if (kv > prefix) atomicAdd(&wgt[t / L], 1);
        else if (kv == prefix) atomicAdd(&weq[t / L], 1);
      }
    } else {
      // too many keys in the bin: digits of 11 and 10 bits over every key
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const uint32_t dmask = pass == 0 ? 0x7ffu : 0x3ffu;
        for (int d = tid; d < kRadixBins; d += kTopkThreads) area[d] = 0;
        __syncthreads();
        for (int t = tid; t < n; t += kTopkThreads) {
          const uint32_t kv = keys[t];
          if ((kv & mask) == prefix) atomicAdd(&area[(kv >> shift) & dmask], 1);
        }
        __syncthreads();
        select_digit(area, (int)dmask, rem, wsum, sh);
        prefix |= (uint32_t)sh[0] << shift;
        mask |= dmask << shift;
        rem = sh[1];
        __syncthreads();
      }
      int gt = 0, eqc = 0;
      for (int t0 = s0; t0 < s1; t0 += 32) {
        const int t = t0 + lane;
        const uint32_t kv = t < s1 ? keys[t] : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, t < s1 && kv > prefix));
        eqc += __popc(__ballot_sync(0xffffffffu, t < s1 && kv == prefix));
      }
      if (lane == 0) {
        wgt[wid] = gt;
        weq[wid] = eqc;
      }
    }
  }
  __syncthreads();
  // ordered write: one scan over the warps' counts gives each warp its
  // output and tie offsets, then a sweep with ballots
  int gt_run = 0, eq_run = 0;
  for (int w = 0; w < wid; ++w) {
    gt_run += wgt[w];
    eq_run += weq[w];
  }
  int placed = gt_run + min(eq_run, rem);  // winners with a smaller entry index
  for (int t0 = s0; t0 < s1; t0 += 32) {
    const int t = t0 + lane;
    const uint32_t kv = t < s1 ? keys[t] : 0u;
    const bool eq = t < s1 && kv == prefix;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const bool take = t < s1 && (kv > prefix || (eq && eq_run + __popc(beq & lt) < rem));
    const uint32_t btake = __ballot_sync(0xffffffffu, take);
    if (take) out[placed + __popc(btake & lt)] = lo + t;
    placed += __popc(btake);
    eq_run += __popc(beq);
  }
}

}  // namespace

size_t indexer_max_entries() { return kMaxEntries; }

size_t indexer_chunk_rows(int B, int S, int Sc) {
  // rows of query positions per pass: the fp32 score buffer stays <= 256 MB
  const size_t ld = (size_t)((Sc + kBlockKeys - 1) / kBlockKeys) * kBlockKeys;
  size_t rows = (size_t)256 << 20;
  rows /= (size_t)(B > 0 ? B : 1) * ld * sizeof(float);
  rows = rows / kRows * kRows;
  if (rows < kRows) rows = kRows;
  if (rows > (size_t)S) rows = ((size_t)S + kRows - 1) / kRows * kRows;
  return rows;
}

size_t indexer_workspace_bytes(int B, int S, int m) {
  const int Sc = (S + m - 1) / m;
  const size_t ld = (size_t)((Sc + kBlockKeys - 1) / kBlockKeys) * kBlockKeys;
  const size_t rows = indexer_chunk_rows(B, S, Sc);
  return kHeaderBytes + align_up((size_t)B * S * sizeof(int32_t)) + align_up((size_t)B * S * kHeadDim * 2) +
         align_up((size_t)B * rows * ld * sizeof(float));
}

cudaError_t indexer_topk(const IndexerArgs &a, cudaStream_t st) {
  const int Sc = (a.S + a.m - 1) / a.m;
  const int ld = (Sc + kBlockKeys - 1) / kBlockKeys * kBlockKeys;
  const int rows_chunk = (int)indexer_chunk_rows(a.B, a.S, Sc);
  __nv_bfloat16 *qc = static_cast<__nv_bfloat16 *>(a.qc);
  // 1. collapse the heads
  {
    const long long rows = (long long)a.B * a.S;
    ProfScope prof(kKIndexScore, st);
    hca_index_collapse_kernel<<<(unsigned)((rows + kCollapseWarps - 1) / kCollapseWarps), 32 * kCollapseWarps, 0,
                                st>>>(static_cast<const __nv_bfloat16 *>(a.qi), a.w, qc, rows, a.Hi);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, ms;
  if (!make_map_bf16(&mq, qc, kHeadDim, a.S, a.B, kRows, 1) || !make_map_bf16(&mk, a.ki, kHeadDim, Sc, a.B, kBlockKeys, 1))
    return cudaErrorInvalidValue;
  static SmemAttrOnce attr_s, attr_t;
  const int topk_smem = ld * (int)sizeof(uint32_t);
  cudaError_t e = attr_s.ensure(reinterpret_cast<const void *>(hca_index_score_kernel), isk::kSmemBytes);
  if (e == cudaSuccess) e = attr_t.ensure(reinterpret_cast<const void *>(hca_index_topk_kernel), kMaxEntries * (int)sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  for (int row0 = 0; row0 < a.S; row0 += rows_chunk) {
    const int rows = min(rows_chunk, a.S - row0);
    ScoreParams sp;
    sp.sstart = a.sstart; sp.buf = a.buf; sp.B = a.B; sp.S = a.S; sp.m = a.m; sp.Sc = Sc;
    sp.row0 = row0; sp.rows = rows; sp.ld = ld; sp.status = a.status; sp.wait_ns = a.wait_ns;
    const int tiles = a.B * ((rows + kRows - 1) / kRows);
    // enough CTAs for two per SM, each with at least two entry blocks
    const int max_blk = (Sc + kBlockKeys - 1) / kBlockKeys;
    sp.groups = max(1, min((2 * sm_count() + tiles - 1) / tiles, max_blk / 2));
    // the chunk buffer holds `rows` rows at pitch ld (16-byte aligned rows: ld is a multiple of 128)
    if (!make_map_scores(&ms, a.buf, (uint64_t)ld, (uint64_t)rows, (uint64_t)a.B)) return cudaErrorInvalidValue;
    {
      ProfScope prof(kKIndexScore, st);
      hca_index_score_kernel<<<tiles * sp.groups, isk::kThreads, isk::kSmemBytes, st>>>(mq, mk, ms, sp);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    TopkParams tp;
    tp.buf = a.buf; tp.sstart = a.sstart; tp.status = a.status; tp.sel = a.sel; tp.scores = a.scores;
    tp.B = a.B; tp.S = a.S; tp.m = a.m; tp.Sc = Sc; tp.row0 = row0; tp.rows = rows; tp.ld = ld; tp.k = a.k;
    {
      ProfScope prof(kKIndexTopk, st);
      hca_index_topk_kernel<<<a.B * rows, kTopkThreads, topk_smem, st>>>(tp);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hca
