// hca_csa.cu -- compressed sparse attention (CSA): the HCA sets with the
// compressed entries narrowed to the indexer's per-query top-k selection.
//
// "Add HCA Static Compilation for Splash Attention [Deepseek v4]",
// Description: CSA (compress ratio 4) needs a top-k step and runtime indexer
// masks that keep or discard (query, compressed entry) pairs; "DSV4: Route
// compressed and sliding train attention onto the splash kernels" routes the
// compressed attention the same way.  Query i attends, under one softmax, to
// its raw window (as in HCA) and to the selected entries j in sel[b,i,:]
// that HCA would let it see (window complete at i, inside i's document);
// selections outside that set, repeats and -1 padding are ignored.
//
// This file holds the CSA-only parts:
//   - csa_union_mask_kernel / csa_union_kernel: per group of P consecutive
//     positions (a forward pair or a dq tile), the sorted set of entries any
//     of them selected and may see, each with the bit mask of the positions
//     that selected it (from byte masks over the group's entry range, or from
//     a sort of the selections, whichever moves fewer bytes).
//     The attention kernels gather those ckv rows into their key blocks and
//     mask each row by its position's bit.
//   - hca_csa_dckv_kernel: dckv, query-major.  Per query tile and block of
//     its union: S = Q K^T and dP = dO K^T (tcgen05, TMEM), P and scale*dS
//     (bf16) into shared memory, then D = P^T dO + (scale dS)^T Q with both
//     A operands read transposed (MN-major) from those tiles, and each
//     entry's row of D added into an fp32 accumulator with float4 atomics
//     (a random selection gives no key-major block structure to reduce in).
//   - a finalize kernel: dckv = bf16(accumulator).
// The raw-key gradients come from the HCA key-major kernel (raw items only).
#include <cuda_bf16.h>

#include "hca_common.cuh"
#include "hca_internal.h"
#include "tc_ptx.cuh"
#include "tc_tiles.cuh"

namespace hca {
using namespace tc;

namespace {

// ---------------------------------------------------------------------------
// union of the selections of a group of positions
// ---------------------------------------------------------------------------
constexpr int kUnionThreads = 256;
constexpr uint32_t kInvalidKey = 0xffffffffu;

struct UnionArgs {
  const int32_t *sel;     // [B,S,k]
  const int32_t *sstart;  // NULL = one document
  int32_t *cnt;           // [B*ngroups]
  int32_t *ent;           // [B*ngroups][cap]
  uint32_t *mask;         // [B*ngroups][cap]
  int B, S, m, Sc, k, P, ngroups, cap, sortn;
  int chunk;  // byte-mask kernel: entries per shared-memory chunk (a multiple of 64)
};

__global__ void __launch_bounds__(kUnionThreads) csa_union_kernel(const UnionArgs a) {
  extern __shared__ uint32_t keys[];
  __shared__ int wsum[kUnionThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = blockIdx.x;
  const int b = g / a.ngroups, pos0 = (g % a.ngroups) * a.P;
  // key = entry * 32 + position in the group; invalid selections sort last
  for (int t = tid; t < a.sortn; t += kUnionThreads) {
    uint32_t key = kInvalidKey;
    if (t < a.P * a.k) {
      const int p = t / a.k, i = pos0 + p;
      if (i < a.S) {
        const int e = a.sel[((size_t)b * a.S + i) * a.k + t % a.k];
        const RowIv iv = row_interval(a.sstart, b, a.S, i, 1, a.m);
        if (iv.valid && e >= iv.clo && e <= iv.chi && e < a.Sc) key = ((uint32_t)e << 5) | (uint32_t)p;
      }
    }
    keys[t] = key;
  }
  __syncthreads();
  // bitonic sort, ascending
  for (int size = 2; size <= a.sortn; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < a.sortn / 2; t += kUnionThreads) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint32_t x = keys[lo], y = keys[hi];
        if ((x > y) == up) {
          keys[lo] = y;
          keys[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  // one output per run of equal entries, in order, with the OR of the
  // positions' bits
  const size_t base = (size_t)g * a.cap;
  int out = 0;
  for (int t0 = 0; t0 < a.sortn; t0 += kUnionThreads) {
    const int t = t0 + tid;
    const uint32_t key = t < a.sortn ? keys[t] : kInvalidKey;
    const bool start = key != kInvalidKey && (t == 0 || (keys[t - 1] >> 5) != (key >> 5));
    int x = start ? 1 : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kUnionThreads / 32; ++w) {
      if (w < wid) before += wsum[w];
      total += wsum[w];
    }
    __syncthreads();
    if (start) {
      uint32_t msk = 0;
      for (int u = t; u < a.sortn && keys[u] != kInvalidKey && (keys[u] >> 5) == (key >> 5); ++u)
        msk |= 1u << (keys[u] & 31u);
      const int pos = out + before + x - 1;
      a.ent[base + pos] = (int32_t)(key >> 5);
      a.mask[base + pos] = msk;
    }
    out += total;
  }
  // pad to a multiple of 16 with a loadable row that no position sees
  const int padded = (out + 15) & ~15;
  for (int t = out + tid; t < padded; t += kUnionThreads) {
    a.ent[base + t] = 0;
    a.mask[base + t] = 0u;
  }
  if (tid == 0) a.cnt[g] = out;
}

// The same union from one byte of position bits per entry.  The group's
// entries lie in [lo, hi] (the union of its positions' visible compressed
// ranges); a chunk of that range is zeroed in shared memory, every selection
// inside the chunk ORs its position's bit into its entry's byte (a shared
// atomic on the containing word), and the non-zero bytes are compacted in
// entry order.  Its cost follows the range (zeroing and one pass over it)
// instead of the bitonic sort's P k log^2(P k) steps; the output is the same
// sorted list.  Needs P <= 8.
constexpr int kMaskPositions = 8;
constexpr int kMaskChunk = 16384;  // default entries (bytes) per chunk

__global__ void __launch_bounds__(kUnionThreads) csa_union_mask_kernel(const UnionArgs a) {
  extern __shared__ uint4 words4[];  // a.chunk bytes: the chunk's entries
  uint32_t *words = reinterpret_cast<uint32_t *>(words4);
  __shared__ int wsum[kUnionThreads / 32];
  __shared__ int2 civ[kMaskPositions];  // visible compressed range per position (empty: x > y)
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = blockIdx.x;
  const int b = g / a.ngroups, pos0 = (g % a.ngroups) * a.P;
  if (tid < a.P) {
    const int i = pos0 + tid;
    int2 r = make_int2(1, 0);
    if (i < a.S) {
      const RowIv iv = row_interval(a.sstart, b, a.S, i, 1, a.m);
      if (iv.valid) r = make_int2(iv.clo, min(iv.chi, a.Sc - 1));
    }
    civ[tid] = r;
  }
  __syncthreads();
  int lo = 0x7fffffff, hi = -1;
  for (int p = 0; p < a.P; ++p)
    if (civ[p].x <= civ[p].y) {
      lo = min(lo, civ[p].x);
      hi = max(hi, civ[p].y);
    }
  int32_t *ent = a.ent + (size_t)g * a.cap;
  uint32_t *msk = a.mask + (size_t)g * a.cap;
  // each thread's first selection of every position, loaded together (the
  // rest, for k > kUnionThreads, are read per chunk)
  const size_t row0 = (size_t)b * a.S + pos0;
  int ev[kMaskPositions];
#pragma unroll
  for (int p = 0; p < kMaskPositions; ++p) {
    ev[p] = -1;
    if (p < a.P && civ[p].x <= civ[p].y && tid < a.k) ev[p] = a.sel[(row0 + p) * a.k + tid];
  }
  int out = 0;
  for (int c0 = lo; c0 <= hi; c0 += a.chunk) {
    const int width = min(a.chunk, hi - c0 + 1);
    const int n4 = (width + 15) >> 4;  // 16 entries per uint4
    for (int w = tid; w < n4; w += kUnionThreads) words4[w] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    // a selection e of position p counts when it is visible to p and in
    // this chunk: e in [max(clo, c0), min(chi, c0 + width - 1)]
#pragma unroll
    for (int p = 0; p < kMaskPositions; ++p) {
      if (p < a.P) {
        const int elo = max(civ[p].x, c0), ehi = min(civ[p].y, c0 + width - 1);
        const int e = ev[p];
        if (e >= elo && e <= ehi) atomicOr(&words[(e - c0) >> 2], (1u << p) << (8 * ((e - c0) & 3)));
        for (int j = tid + kUnionThreads; j < a.k && elo <= ehi; j += kUnionThreads) {
          const int e2 = a.sel[(row0 + p) * a.k + j];
          if (e2 >= elo && e2 <= ehi) atomicOr(&words[(e2 - c0) >> 2], (1u << p) << (8 * ((e2 - c0) & 3)));
        }
      }
    }
    __syncthreads();
    // ordered compaction: thread tid of round q takes entries
    // [16 (q*256 + tid), +16) of the chunk
    for (int q0 = 0; q0 < n4; q0 += kUnionThreads) {
      const int q = q0 + tid;
      const uint4 v = q < n4 ? words4[q] : make_uint4(0u, 0u, 0u, 0u);
      // bit 4x + y of nz: byte y of word x is non-zero (the byte's high bit
      // after adding 0x7f to its low seven bits, or its own high bit; the
      // four high bits then gathered into a nibble by one multiply whose
      // partial products do not overlap)
      uint32_t nz = 0;
      {
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint32_t hb = (((wv[x] & 0x7f7f7f7fu) + 0x7f7f7f7fu) | wv[x]) & 0x80808080u;
          nz |= (((hb >> 7) * 0x01020408u) >> 24) << (4 * x);
        }
      }
      const int cnt = __popc(nz);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) wsum[wid] = incl;
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < kUnionThreads / 32; ++w) {
        if (w < wid) before += wsum[w];
        total += wsum[w];
      }
      __syncthreads();
      int pos = out + before + incl - cnt;
      while (nz != 0u) {
        const int bi = __ffs(nz) - 1;
        nz &= nz - 1u;
        const uint32_t wsel = (bi & 8) ? ((bi & 4) ? v.w : v.z) : ((bi & 4) ? v.y : v.x);
        ent[pos] = c0 + 16 * q + bi;
        msk[pos] = (wsel >> (8 * (bi & 3))) & 0xffu;
        ++pos;
      }
      out += total;
    }
  }
  // pad to a multiple of 16 with a loadable row that no position sees
  const int padded = (out + 15) & ~15;
  for (int t = out + tid; t < padded; t += kUnionThreads) {
    ent[t] = 0;
    msk[t] = 0u;
  }
  if (tid == 0) a.cnt[g] = out;
}

// ---------------------------------------------------------------------------
// dckv, query-major
// ---------------------------------------------------------------------------
namespace ckk {
constexpr int kStages = 2;
constexpr int kEW = 256;                  // two warpgroups, 64 key columns each
constexpr int kThreads = kEW + 128;       // + TMA warp, MMA warp, gather warp, one idle warp
constexpr int kRegEW = 192, kRegProducer = 120;
static_assert(2 * 128 * kRegEW + 128 * kRegProducer <= kThreads * 168, "register split must fit the launch");
constexpr uint32_t kColS = 0, kColDP = 128, kColD = 256;  // D: two 128-column buffers
constexpr int kTmemCols = 512;
constexpr int kOffQ = 0, kOffDO = kTile, kOffKV = 2 * kTile;
constexpr int kOffP = kOffKV + kStages * kTile, kOffDS = kOffP + kTile;
constexpr int kSmemBytes = kOffDS + kTile + 1024;
constexpr int kMaxPos = 4;                // positions per tile (H a multiple of 32)
constexpr int kGather = 32;               // the gather warp's lanes (each issues TMA gather4 loads)
}  // namespace ckk

struct DckvParams {
  QTiling qt;
  const float *rowstat;       // [ntiles][2][128] from the dq kernel
  const int32_t *u_cnt, *u_ent;
  const uint32_t *u_mask;
  int u_cap;
  float *acc;                 // [B][Sc][D] fp32
  int32_t *status;
  float sl2, scale;
  int pq_shift;
  uint64_t wait_ns;
};

struct DckvBars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[ckk::kStages], kv_empty[ckk::kStages];
  uint64_t s_full, s_free;
  uint64_t pds_full, pds_free;
  uint64_t d_full[2], d_free[2];
  uint64_t drain;
  uint32_t vis[ckk::kStages][ckk::kMaxPos][4];
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(ckk::kThreads, 1)
    hca_csa_dckv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                        const __grid_constant__ CUtensorMap map_ckv, const DckvParams p) {
  using namespace ckk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DckvBars bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int *abort_flag = &bars.abort;
  const QTiling &Q = p.qt;

  if (tid == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.kv_full[s], kGather);
      // the S/dP MMAs' commit and every dS thread once it has read the block's bits
      mbar_init(&bars.kv_empty[s], 1 + kEW);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, kEW);
    mbar_init(&bars.pds_full, kEW);
    mbar_init(&bars.pds_free, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.d_full[x], 1);
      mbar_init(&bars.d_free[x], kEW);
    }
    mbar_init(&bars.drain, 1);
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
  const bool poisoned = *(volatile const int32_t *)p.status != 0;

  // the tiles this CTA owns, and the number of key blocks of each
  auto tile_blocks = [&](long long u, Tile &t, int &cnt) -> int {
    tile_coords(Q, u, t);
    const long long grp = (long long)t.b * Q.ntq + t.i0 / Q.Pq;
    cnt = p.u_cnt[grp];
    return (cnt + kBlockKeys - 1) / kBlockKeys;
  };

  if (warp >= kEW / 32) {
    setmaxnreg_dec<kRegProducer>();
    if (warp == kEW / 32) {
      // ------------------------------------------------------------ TMA: Q and dO tiles
      uint32_t tw = 0;
      int q_par = -1;
      bool ok = !poisoned;
      for (long long u = blockIdx.x; ok && u < Q.ntiles; u += gridDim.x) {
        Tile t;
        int cnt;
        if (tile_blocks(u, t, cnt) == 0) continue;
        if (lane == 0) {
          if (tw > 0) ok = mbar_wait(&bars.q_empty, (tw - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (ok) {
            mbar_arrive_expect_tx(&bars.q_full, 2 * kTile);
            const int c2 = t.b * Q.H + t.g * Q.HG;
            tma_load_3d(&map_q, &bars.q_full, smem + kOffQ, 0, t.i0, c2);
            tma_load_3d(&map_q, &bars.q_full, smem + kOffQ + kHalfTile, 64, t.i0, c2);
            tma_load_3d(&map_do, &bars.q_full, smem + kOffDO, 0, t.i0, c2);
            tma_load_3d(&map_do, &bars.q_full, smem + kOffDO + kHalfTile, 64, t.i0, c2);
            q_par = tw & 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        ++tw;
      }
      if (!ok && !poisoned && lane == 0 && q_par >= 0) {
        volatile int never = 0;
        mbar_wait(&bars.q_full, q_par, &never, p.status, 100000000ull);
      }
    } else if (warp == kEW / 32 + 2) {
      // ------------------------------------------------------------ gather: the union's ckv rows
      // Each block's entries land in the 128B-swizzled tile layout the MMA
      // descriptors read, four rows per TMA gather4 load through the row view
      // of ckv (lane l takes rows 4l .. 4l + 3; 16-byte copies made one warp's
      // issue the limit); the per-position visibility bits of the block go to
      // shared memory beside them.  Warp kEW/32 + 3 is idle.
      uint32_t gb = 0;
      uint32_t issued = 0;  // bit s: stage s loaded at least once; bit 8+s: parity of its last load
      bool ok = !poisoned;
      for (long long u = blockIdx.x; ok && u < Q.ntiles; u += gridDim.x) {
        Tile t;
        int cnt;
        const int nb = tile_blocks(u, t, cnt);
        const long long grp = (long long)t.b * Q.ntq + t.i0 / Q.Pq;
        const int32_t *ent = p.u_ent + grp * p.u_cap;
        const uint32_t *msk = p.u_mask + grp * p.u_cap;
        const int rb = t.b * Q.Sc;  // row of ckv[b][0] in the row view
        for (int j = 0; ok && j < nb; ++j, ++gb) {
          const int s = gb % kStages;
          const int c0 = j * kBlockKeys;
          const int n = min(kBlockKeys, ((cnt + 15) & ~15) - c0);  // a multiple of 16
          // entry ids and selection masks, loaded before the wait for a stage
          const int4 e4 = 4 * lane < n ? *reinterpret_cast<const int4 *>(ent + c0 + 4 * lane) : make_int4(0, 0, 0, 0);
          uint32_t mk[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int c = c0 + 32 * w + lane;
            mk[w] = (32 * w + lane < n && c < cnt) ? msk[c] : 0u;
          }
          if (gb >= (uint32_t)kStages)
            ok = wait_warp(&bars.kv_empty[s], ((gb / kStages) - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (!ok) break;
          uint8_t *dst = smem + kOffKV + s * kTile;
          if (lane == 0) mbar_expect_tx(&bars.kv_full[s], (uint32_t)n * 256u);
          __syncwarp();  // the expected bytes are set before any row lands
          if (4 * lane < n) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              tma_gather4(&map_ckv, &bars.kv_full[s], dst + hh * kHalfTile + 4 * lane * 128, 64 * hh, rb + e4.x,
                          rb + e4.y, rb + e4.z, rb + e4.w);
          }
          // visibility bits: word w of position pp = columns [32 w, 32 w + 32)
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            for (int pp = 0; pp < Q.Pq; ++pp) {
              const uint32_t bits = __ballot_sync(0xffffffffu, (mk[w] >> pp) & 1u);
              if (lane == 0) bars.vis[s][pp][w] = bits;
            }
          }
          mbar_arrive(&bars.kv_full[s]);
          issued = (issued | (1u << s)) & ~(1u << (8 + s));
          issued |= ((gb / kStages) & 1u) << (8 + s);
        }
      }
      if (!ok && !poisoned && lane == 0) {
        // the loads already issued land before the CTA can exit
        volatile int never = 0;
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) mbar_wait(&bars.kv_full[s], (issued >> (8 + s)) & 1u, &never, p.status, 100000000ull);
      }
    } else if (warp == kEW / 32 + 1) {
      // ------------------------------------------------------------ MMA
      const uint64_t dQk = smem_desc_sw128(smem_u32(smem + kOffQ), 16, 1024);          // K-major (S)
      const uint64_t dDOk = smem_desc_sw128(smem_u32(smem + kOffDO), 16, 1024);        // K-major (dP)
      const uint64_t dQm = smem_desc_sw128(smem_u32(smem + kOffQ), kHalfTile, 1024);   // MN-major (D)
      const uint64_t dDOm = smem_desc_sw128(smem_u32(smem + kOffDO), kHalfTile, 1024);
      const uint64_t dK0 = smem_desc_sw128(smem_u32(smem + kOffKV), 16, 1024);
      const uint64_t dP = smem_desc_sw128(smem_u32(smem + kOffP), kHalfTile, 1024);    // P^T: MN-major A
      const uint64_t dDS = smem_desc_sw128(smem_u32(smem + kOffDS), kHalfTile, 1024);  // dS^T: MN-major A
      const uint32_t id_d = idesc_bf16_f32(kRows, kHeadDim, true, true);
      uint32_t gb = 0, tw = 0;
      bool ok = !poisoned, issued = false;
      for (long long u = blockIdx.x; ok && u < Q.ntiles; u += gridDim.x) {
        Tile t;
        int cnt;
        const int nb = tile_blocks(u, t, cnt);
        if (nb == 0) continue;
        ok = wait_warp(&bars.q_full, tw & 1, abort_flag, p.status, p.wait_ns);
        for (int j = 0; ok && j < nb; ++j) {
          const uint32_t g = gb + j;
          const int s = g % kStages;
          const int n = min(kBlockKeys, ((cnt + 15) & ~15) - j * kBlockKeys);
          ok = wait_warp(&bars.kv_full[s], (g / kStages) & 1, abort_flag, p.status, p.wait_ns);
          // the previous block's S and dP have been read out
          if (ok && g > 0) ok = wait_warp(&bars.s_free, (g - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(kRows, n, false, false);
          const uint64_t bk = dK0 + desc_bytes(s * kTile);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < kHeadDim / 16; ++k) mma_ss(tmem + kColS, dQk + kmaj_step(k), bk + kmaj_step(k), idesc, k > 0);
#pragma unroll
            for (int k = 0; k < kHeadDim / 16; ++k)
              mma_ss(tmem + kColDP, dDOk + kmaj_step(k), bk + kmaj_step(k), idesc, k > 0);
            mma_commit(&bars.s_full);
            mma_commit(&bars.kv_empty[s]);  // the key block's last readers (with the dS warps' read of its bits)
          }
          __syncwarp();
          issued = true;
          // D = P^T dO + (scale dS)^T Q once P and dS are in shared memory
          const int x = g & 1;
          ok = wait_warp(&bars.pds_full, g & 1, abort_flag, p.status, p.wait_ns);
          if (ok && g >= 2) ok = wait_warp(&bars.d_free[x], ((g / 2) - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
            const uint32_t d = tmem + kColD + x * 128;
#pragma unroll
            for (int k = 0; k < kRows / 16; ++k) mma_ss(d, dP + mnmaj_step(k), dDOm + mnmaj_step(k), id_d, k > 0);
#pragma unroll
            for (int k = 0; k < kRows / 16; ++k) mma_ss(d, dDS + mnmaj_step(k), dQm + mnmaj_step(k), id_d, 1u);
            mma_commit(&bars.d_full[x]);
            mma_commit(&bars.pds_free);
            if (j == nb - 1) mma_commit(&bars.q_empty);  // Q and dO are last read by the D MMAs
          }
          __syncwarp();
        }
        gb += nb;
        ++tw;
      }
      if (!ok && issued) {
        volatile int never = 0;
        if (elect_one()) mma_commit(&bars.drain);
        __syncwarp();
        if (lane == 0) mbar_wait(&bars.drain, 0, &never, p.status, 100000000ull);
        __syncwarp();
      }
    }
  } else {
    setmaxnreg_inc<kRegEW>();
    // ------------------------------------------------------------ P, dS and the dckv rows
    // thread r of warpgroup wg: query row r (TMEM lane r) and key columns
    // [64 wg, 64 wg + 64) of every block; then entry column r of the block's
    // D, its dims [64 wg, 64 wg + 64), into the fp32 accumulator.
    const int r = tid & (kRows - 1), wg = tid >> 7;
    const int cb = wg * 64;
    const int pq = r & (Q.Pq - 1);
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint64_t sl2x2 = f32x2(__float_as_uint(p.sl2), __float_as_uint(p.sl2));
    uint32_t gb = 0;
    bool ok = !poisoned;
    for (long long u = blockIdx.x; ok && u < Q.ntiles; u += gridDim.x) {
      Tile t;
      int cnt;
      const int nb = tile_blocks(u, t, cnt);
      if (nb == 0) continue;
      const long long tl = ((long long)t.b * Q.groups + t.g) * Q.ntq + t.i0 / Q.Pq;
      const float nl2 = p.rowstat[tl * 2 * kRows + r];             // -lse*log2e (0 for invalid rows)
      const float ndl = p.rowstat[tl * 2 * kRows + kRows + r];     // -scale*Delta
      const int i = t.i0 + pq;
      const bool row_valid = i < Q.S && (Q.sstart == nullptr || Q.sstart[(size_t)t.b * Q.S + i] >= 0);
      const long long grp = (long long)t.b * Q.ntq + t.i0 / Q.Pq;
      const int32_t *ent = p.u_ent + grp * p.u_cap;
      for (int j = 0; j < nb; ++j, ++gb) {
        const int s = gb % kStages;
        const int c0 = j * kBlockKeys;
        if (!wait_warp(&bars.s_full, gb & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        // S and dP of the row's 64 columns, 32 at a time, into P and scale*dS
        // (bf16) in shared memory; the bits say which columns the row sees
        if (!wait_warp(&bars.kv_full[s], (gb / kStages) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        const uint64_t vis = row_valid ? ((uint64_t)bars.vis[s][pq][2 * wg] | ((uint64_t)bars.vis[s][pq][2 * wg + 1] << 32))
                                       : 0ull;
        mbar_arrive(&bars.kv_empty[s]);
        // the previous block's D MMAs must have read the P and dS tiles
        if (gb > 0 && !wait_warp(&bars.pds_free, (gb - 1) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        const uint64_t nl2x2 = f32x2(__float_as_uint(nl2), __float_as_uint(nl2));
        const uint64_t sc2 = f32x2(__float_as_uint(p.scale), __float_as_uint(p.scale));
        const uint64_t nd2 = f32x2(__float_as_uint(ndl), __float_as_uint(ndl));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t sv[32], dv[32];
          tmem_ld32(lane_addr + kColS + cb + 32 * h, sv);
          tmem_ld32(lane_addr + kColDP + cb + 32 * h, dv);
          tmem_wait_ld();
          if (h == 1) {
            tc_fence_before();
            mbar_arrive(&bars.s_free);
          }
          const uint32_t vh = (uint32_t)(vis >> (32 * h));
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t pw[4], dw[4];
#pragma unroll
            for (int y = 0; y < 8; y += 2) {
              const int c = ch * 8 + y;
              float t0, t1;
              f32x2_split(ffma2(f32x2(sv[c], sv[c + 1]), sl2x2, nl2x2), t0, t1);
              float e0 = ex2_approx(t0), e1 = ex2_approx(t1);
              // scale dP - scale Delta, times P
              float g0, g1;
              f32x2_split(fmul2(f32x2(__float_as_uint(e0), __float_as_uint(e1)), ffma2(f32x2(dv[c], dv[c + 1]), sc2, nd2)),
                          g0, g1);
              const bool v0 = (vh >> c) & 1u, v1 = (vh >> (c + 1)) & 1u;
              e0 = v0 ? e0 : 0.f;
              e1 = v1 ? e1 : 0.f;
              g0 = v0 ? g0 : 0.f;
              g1 = v1 ? g1 : 0.f;
              pw[y >> 1] = pack_bf16x2(e0, e1);
              dw[y >> 1] = pack_bf16x2(g0, g1);
            }
            const uint32_t off = sw128_offset(r, (cb + 32 * h) / 8 + ch);
            *reinterpret_cast<uint4 *>(smem + kOffP + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
            *reinterpret_cast<uint4 *>(smem + kOffDS + off) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
          }
        }
        fence_async_smem();
        mbar_arrive(&bars.pds_full);
        // D of this block: entry column r of the block, dims [64 wg, 64 wg + 64)
        const int x = gb & 1;
        if (!wait_warp(&bars.d_full[x], (gb / 2) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        uint32_t o[64];
        tmem_ld32(lane_addr + kColD + x * 128 + cb, *reinterpret_cast<uint32_t(*)[32]>(o));
        tmem_ld32(lane_addr + kColD + x * 128 + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars.d_free[x]);
        // The block's D MMAs (done: d_full) were the last readers of its P
        // and dS tiles, and this warp alone writes their rows [32 (warp & 3),
        // +32) of half wg: 4 KB in each tile, the room for the warp's 32 rows
        // of 64 fp32 values.  Staged there (float4 index XOR row, so no two
        // lanes of an 8-lane phase share banks) and read back transposed,
        // each atomic instruction adds two whole 256-byte row pieces instead
        // of 32 scattered 16-byte pieces.
        {
          const int wl = warp & 3;
          uint8_t *stg_p = smem + kOffP + wg * kHalfTile + wl * 32 * 128;
          uint8_t *stg_d = smem + kOffDS + wg * kHalfTile + wl * 32 * 128;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            uint8_t *base = q < 8 ? stg_p : stg_d;
            const int col = (q & 7) ^ (lane & 7);
            *reinterpret_cast<float4 *>(base + lane * 128 + col * 16) =
                make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]), __uint_as_float(o[4 * q + 2]),
                            __uint_as_float(o[4 * q + 3]));
          }
          __syncwarp();
          const int f = lane & 15;
          const uint8_t *rbase = f < 8 ? stg_p : stg_d;
#pragma unroll 2
          for (int q = 0; q < 16; ++q) {
            const int ri = 2 * q + (lane >> 4);  // the warp's row this lane adds to
            const int e = c0 + wl * 32 + ri;       // its position in the union
            if (e < cnt) {
              const float4 v = *reinterpret_cast<const float4 *>(rbase + ri * 128 + (((f & 7) ^ (ri & 7)) * 16));
              float4 *dst = reinterpret_cast<float4 *>(p.acc + ((size_t)t.b * Q.Sc + ent[e]) * kHeadDim + cb);
              atomicAdd(dst + f, v);
            }
          }
          __syncwarp();  // staging read before the next block's P and dS go there
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void csa_dckv_finalize_kernel(const float *acc, __nv_bfloat16 *dckv, long long n4, const int32_t *status) {
  const bool poisoned = *(volatile const int32_t *)status != 0;
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n4; v += (long long)gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4 *>(acc)[v];
    if (poisoned) a = make_float4(NAN, NAN, NAN, NAN);
    uint2 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    reinterpret_cast<uint2 *>(dckv)[v] = o;
  }
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

size_t csa_union_bytes(int B, int S, int P, int k) {
  const long long ng = ((long long)S + P - 1) / P;
  const long long cap = ((long long)P * k + 15) / 16 * 16;
  return align_up((size_t)B * ng * sizeof(int32_t)) + 2 * align_up((size_t)B * ng * cap * sizeof(int32_t));
}

bool csa_shape_ok(int H, int k) {
  // masks carry one bit per position of a forward pair: Pq <= 4 (H a multiple of 32)
  if (H < 1 || (H % 32) != 0 || k < 1) return false;
  const int Pq = kRows / heads_per_tile(H);
  return Pq <= ckk::kMaxPos && 2 * Pq * k <= 32768;
}

cudaError_t csa_build_union(const int32_t *sel, const int32_t *sstart, int B, int S, int m, int k, int P,
                            CsaUnion &u, void *mem, cudaStream_t st) {
  const int ng = (S + P - 1) / P;
  u.P = P;
  u.cap = (P * k + 15) / 16 * 16;
  u.ngroups = ng;
  char *c = static_cast<char *>(mem);
  u.cnt = reinterpret_cast<int32_t *>(c);
  c += align_up((size_t)B * ng * sizeof(int32_t));
  u.ent = reinterpret_cast<int32_t *>(c);
  c += align_up((size_t)B * ng * u.cap * sizeof(int32_t));
  u.mask = reinterpret_cast<uint32_t *>(c);
  if ((long long)B * ng == 0) return cudaSuccess;
  UnionArgs a;
  a.sel = sel; a.sstart = sstart; a.cnt = u.cnt; a.ent = u.ent; a.mask = u.mask;
  a.B = B; a.S = S; a.m = m; a.Sc = (S + m - 1) / m; a.k = k; a.P = P; a.ngroups = ng; a.cap = u.cap;
  a.sortn = next_pow2(P * k);
  if (a.sortn < 2) a.sortn = 2;
  a.chunk = kMaskChunk;
  // shared-memory bytes moved per group: the sort's compare-exchange stages
  // (two loads, up to two stores each) against zeroing and scanning the
  // entry range (Sc/2 on average) plus one atomic per selection
  int lg = 0;
  while ((1 << lg) < a.sortn) ++lg;
  const long long sort_cost = (long long)a.sortn * (lg * (lg + 1) / 2) * 6;
  const long long mask_cost = (long long)a.Sc + 4LL * P * k;
  bool use_mask = P <= kMaskPositions && mask_cost < sort_cost;
  const int setting = csa_union_setting();
  if (setting == 1) use_mask = false;
  if (setting >= 64) {
    if (P > kMaskPositions) return cudaErrorInvalidValue;
    use_mask = true;
    a.chunk = setting;
  }
  ProfScope prof(kKCsaUnion, st);
  if (use_mask) {
    csa_union_mask_kernel<<<B * ng, kUnionThreads, a.chunk, st>>>(a);
  } else {
    static SmemAttrOnce attr;
    cudaError_t e = attr.ensure(reinterpret_cast<const void *>(csa_union_kernel), 32768 * (int)sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    csa_union_kernel<<<B * ng, kUnionThreads, a.sortn * sizeof(uint32_t), st>>>(a);
  }
  return cudaGetLastError();
}

size_t csa_dckv_acc_bytes(int B, int Sc) { return align_up((size_t)B * Sc * kHeadDim * sizeof(float)); }

cudaError_t csa_dckv(const BwdArgs &a, const CsaUnion &u, const float *rowstat, float *acc, cudaStream_t st) {
  const QTiling q = make_qtiling(a.sstart, a.B, a.H, a.S, a.W, a.m);
  CUtensorMap mq, mdo, mckv;
  if (!make_map_bf16(&mq, a.q, kHeadDim, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mdo, a.dout, kHeadDim, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_rows_bf16(&mckv, a.ckv, kHeadDim, (uint64_t)q.Sc * a.B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(acc, 0, (size_t)a.B * q.Sc * kHeadDim * sizeof(float), st);
  if (e != cudaSuccess) return e;
  static SmemAttrOnce attr;
  e = attr.ensure(reinterpret_cast<const void *>(hca_csa_dckv_kernel), ckk::kSmemBytes);
  if (e != cudaSuccess) return e;
  DckvParams p;
  p.qt = q;
  p.rowstat = rowstat;
  p.u_cnt = u.cnt; p.u_ent = u.ent; p.u_mask = u.mask; p.u_cap = u.cap;
  p.acc = acc;
  p.status = a.status_rw;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.scale = a.scale;
  p.pq_shift = 0;
  while ((1 << p.pq_shift) < q.Pq) ++p.pq_shift;
  p.wait_ns = a.wait_ns;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const long long grid = q.ntiles < sms ? q.ntiles : sms;
  if (grid > 0) {
    ProfScope prof(kKCsaDckv, st);
    hca_csa_dckv_kernel<<<(unsigned)grid, ckk::kThreads, ckk::kSmemBytes, st>>>(mq, mdo, mckv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long long n4 = (long long)a.B * q.Sc * kHeadDim / 4;
  if (n4 > 0) {
    int blocks = (int)((n4 + 255) / 256);
    if (blocks > 8 * sms) blocks = 8 * sms;
    csa_dckv_finalize_kernel<<<blocks, 256, 0, st>>>(acc, static_cast<__nv_bfloat16 *>(a.dckv), n4, a.status_rw);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace hca
