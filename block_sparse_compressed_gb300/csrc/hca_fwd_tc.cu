// hca_fwd_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) HCA forward for sm_103a.
//
// Operation ("Add HCA Static Compilation for Splash Attention [Deepseek v4]",
// Description: sliding window + completed compression windows, MQA dispatch
// with the single kv head; "[DeepSeek-V4] Implement Compressed Attention
// Layers", einsum review suggestions: k = v = kv broadcast over heads).
//
// Tiling.  All heads of a query position share every key row (one kv head),
// so a query tile packs Pq consecutive positions x HG heads into the M = 128
// rows of the MMA (row r = head*Pq + p), loaded by one 3-D TMA box
// {64, Pq, HG} per 64-column half of q.  A CTA works on a *pair* of adjacent
// query tiles (A and B) that share one stream of key blocks: the union of the
// 2*Pq positions' intervals (hca_common.cuh) as one list of columns, the
// compressed ckv entries then the raw kv keys, cut into blocks of <= 128
// columns (a block may hold both kinds; tc_tiles.cuh).  Keys outside those
// ranges are never loaded and no mask exists in memory; inside a block every
// row masks by its own two intervals.
//
// Per half-block k (64 keys of a key block) and tile X in {A, B}:
//   S_X = Q_X K^T            tcgen05 SS, fp32 accumulator in TMEM buffer
//                            (k mod 2) of S_X
//   softmax warpgroup X      loads S_X, masks, online softmax in fp32 with
//                            exp2 (the running max is raised only when a
//                            half-block beats it by more than 2^8, so O_X is
//                            rarely rescaled), writes P_X (bf16) back into
//                            the first half of the buffer's columns
//   O_X += P_X V             tcgen05 TS: A = P_X from TMEM, B = the same kv
//                            rows through an MN-major descriptor (K = V)
// S_X is double-buffered: S_X(k+1) is computed while the softmax works on
// k, and S_X(k+2) is issued right after PV_X(k).  The tensor pipe executes
// one thread's MMAs in order, so S_X(k+2) cannot overwrite P_X(k) before
// PV_X(k) has read it.  The MMA warp interleaves the two tiles so that the
// tensor core runs one tile's GEMMs while the other's softmax works.  A
// softmax that must rescale O_X first waits for PV_X(k-1) (a barrier the
// MMA warp commits after every PV).
//
// q is double-buffered over a CTA's pairs: the next pair's q tiles are
// requested while the current pair runs (their load takes several thousand
// cycles, which a single buffer exposed at every pair boundary).  The buffer
// of a finished pair holds no live q any more -- O_X is final only after
// every MMA of tile X -- so the epilogue stages the pair's output there, and
// the buffer is reloaded once the output stores have read it.
//
// Warp roles (512 threads, persistent CTAs; registers rebalanced with
// setmaxnreg to 160 / 160 / 104 / 88 per thread):
//   warpgroup 0   softmax of tile A (thread r owns row r = TMEM lane r)
//   warpgroup 1   softmax of tile B
//   warpgroup 2   epilogue: O_X * (1/l) -> bf16 -> swizzled smem (the pair's
//                 q buffer) -> TMA store
//   warpgroup 3   warp 12 TMA producer, warps 13 and 14 MMA issuers (tile A,
//                 tile B), warp 15 idle; with CSA warp 13 issues for both
//                 tiles and warps 14-15 are idle (the TMA warp gathers the
//                 selected rows with TMA gather4 loads)
// Every wait is bounded (tc_ptx.cuh): on a timeout the CTA records
// HCA_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>

#include "hca_common.cuh"
#include "hca_internal.h"
#include "tc_ptx.cuh"
#include "tc_tiles.cuh"

namespace hca {
using namespace tc;

namespace {

constexpr int kStages = 3;        // kv ring depth
constexpr int kWG = 128;          // threads per warpgroup
constexpr int kThreads = 4 * kWG;
constexpr int kTmemCols = 512;    // S_A | S_B | O_A | O_B, 128 columns each
constexpr int kHalfKeys = 64;     // keys of a half-block: S_X is two buffers of 64 columns
__host__ __device__ constexpr uint32_t col_s(int x) { return (uint32_t)x * 128u; }        // S_X (P_X aliases it)
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u + (uint32_t)x * 128u; }  // O_X
constexpr float kRescaleLog2 = 8.0f;
constexpr int kRegSoftmax = 160, kRegEpilogue = 104, kRegProducer = 88;
static_assert(2 * kRegSoftmax + kRegEpilogue + kRegProducer == 512, "register split must fit the launch");

// dynamic shared memory: q ring of two pairs (Q_A | Q_B each; a finished
// pair's q buffer becomes its output staging) | kv ring (+1 KB align)
constexpr int kOffQ = 0;
constexpr int kQBuf = 2 * kTile;  // one pair's q tiles, later its output tiles
constexpr int kOffKV = kOffQ + 2 * kQBuf;
constexpr int kSmemBytes = kOffKV + kStages * kTile + 1024;
constexpr int kCsaMaxPos = 8;     // positions of a pair whose bits CSA keeps (Pq <= 4)

// CSA: per pair, the union of its positions' selected entries (hca_csa.cu).
// A kernel argument of its own: growing FwdParams changes how the HCA
// instantiation keeps its parameters and costs it registers.
struct CsaParams {
  const int32_t *u_cnt, *u_ent;
  const uint32_t *u_mask;
  int u_cap;
  const __nv_bfloat16 *ckv;
};

struct FwdParams {
  QTiling qt;          // per query tile (Pq positions)
  long long npairs;    // pair tiles over (b, head group, pair index)
  int ntp;             // pairs per (b, group)
  int32_t *status;
  float *lse;
  __nv_bfloat16 *out;  // direct stores for poisoned calls / pairs without keys
  float sl2;           // scale * log2(e)
  uint64_t wait_ns;    // limit of every bounded wait
  int stall;           // failure-path test: the MMA warp first waits on a barrier nothing arrives at
};

// A pair of adjacent query tiles (A at i0, B at i0 + Pq) shares one key list:
// the union of both tiles' key ranges, i.e. a Tile of 2 Pq positions.
__device__ __forceinline__ void pair_coords(const FwdParams &p, long long u, Tile &t) {
  // longest pairs first: the compressed range grows with the position
  const long long per = (long long)p.qt.B * p.qt.groups;
  const int tp = p.ntp - 1 - (int)(u / per);
  const int rem = (int)(u % per);
  t.b = rem / p.qt.groups;
  t.g = rem % p.qt.groups;
  t.i0 = tp * 2 * p.qt.Pq;
}

template <bool kCsa>
__device__ __forceinline__ void pair_ranges_warp(const FwdParams &p, const CsaParams &cp, Tile &t, int lane) {
  QTiling q2 = p.qt;
  q2.Pq = 2 * p.qt.Pq;
  tile_ranges_warp(q2, t, lane);
  if (kCsa) {
    // compressed columns: the pair's union of selected entries
    const int cnt = cp.u_cnt[(long long)t.b * p.ntp + t.i0 / (2 * p.qt.Pq)];
    t.clo = 0;
    t.chi = cnt;
    t.cpad = (cnt + 15) & ~15;
    t.ncols = t.cpad + (t.rhi - t.rlo);
    t.nb = (t.ncols + kBlockKeys - 1) / kBlockKeys;
  }
}

// Half-blocks of a pair's key list: two per block, one for a last block of
// at most 64 columns.
__device__ __forceinline__ int half_blocks(const Tile &t) {
  return 2 * (t.nb - 1) + (t.ncols - (t.nb - 1) * kBlockKeys > kHalfKeys ? 2 : 1);
}

__device__ __forceinline__ void setmaxnreg_inc_softmax() { asm volatile("setmaxnreg.inc.sync.aligned.u32 160;"); }
__device__ __forceinline__ void setmaxnreg_dec_epilogue() { asm volatile("setmaxnreg.dec.sync.aligned.u32 104;"); }
__device__ __forceinline__ void setmaxnreg_dec_producer() { asm volatile("setmaxnreg.dec.sync.aligned.u32 88;"); }

struct Bars {
  uint64_t q_full[2], q_empty[2];  // q ring; a buffer is empty once the pair's output stores have read it
  Tile tile[2];                    // geometry of the pair in each q buffer (nb < 0: end of the schedule)
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2][2], p_full[2][2], pv_done[2];  // [tile][buffer]: the softmax may finish k + 1 before the MMA waits for k
  uint64_t o_final[2], o_free[2];
  uint64_t st_full[2], st_free[2];
  uint64_t epi, drain[2], never;
  float inv_l[2][kRows];
  uint32_t vis[kStages][kCsaMaxPos][4];  // CSA: per block, each pair position's bits of the compressed columns
  uint32_t tmem_base;
  int abort;
};

template <bool kPosScale, bool kCsa, int kD>
__global__ void __launch_bounds__(kThreads, 1)
    hca_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                      const __grid_constant__ CUtensorMap map_ckv, const __grid_constant__ CUtensorMap map_kv16,
                      const __grid_constant__ CUtensorMap map_ckv16, const __grid_constant__ CUtensorMap map_out,
                      const FwdParams p, const CsaParams cp) {
  static_assert(kD == 64 || kD == 128, "head dim 64 or 128");
  static_assert(!kCsa || kD == 128, "CSA gathers 128-dim rows");
  constexpr int kHalves = kD / 64;   // 64-column (128-byte) halves of a row
  // MMA issue: warp 13 for tile A and warp 14 for tile B; with CSA warp 13
  // issues for both tiles
  constexpr int kMmaWarps = kCsa ? 1 : 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2;
  volatile int *abort_flag = &bars.abort;
  const QTiling &Q = p.qt;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.q_full[b], 1);
      mbar_init(&bars.q_empty[b], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      // CSA: every lane of the TMA warp arrives once it has issued its
      // gather loads and the visibility bits are written
      mbar_init(&bars.kv_full[s], kCsa ? 32 : 1);
      mbar_init(&bars.kv_empty[s], kMmaWarps);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.s_full[x][0], 1);
      mbar_init(&bars.s_full[x][1], 1);
      mbar_init(&bars.pv_done[x], 1);
      mbar_init(&bars.p_full[x][0], kWG);
      mbar_init(&bars.p_full[x][1], kWG);
      mbar_init(&bars.o_final[x], 1);
      mbar_init(&bars.o_free[x], kWG);
      mbar_init(&bars.st_full[x], kWG);
      mbar_init(&bars.st_free[x], kWG);
    }
    mbar_init(&bars.epi, kWG);
    mbar_init(&bars.drain[0], 1);
    mbar_init(&bars.drain[1], 1);
    mbar_init(&bars.never, 1);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const bool poisoned = *(volatile const int32_t *)p.status != 0;

  if (wg == 3) {
    setmaxnreg_dec_producer();
    if (warp == 12) {
      // ---------------------------------------------------------- TMA
      if (!poisoned && lane == 0) {
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_kv);
        tma_prefetch_map(&map_ckv);
        tma_prefetch_map(&map_kv16);
        tma_prefetch_map(&map_ckv16);
      }
      uint32_t gb = 0, gq = 0;
      uint32_t issued = 0;    // bit s: stage s loaded at least once; bit 8+s: parity of its last load
      uint32_t q_issued = 0;  // the same for the two q buffers
      bool ok = !poisoned;
      for (long long u = blockIdx.x; ok && u < p.npairs; u += gridDim.x) {
        Tile t;
        pair_coords(p, u, t);
        pair_ranges_warp<kCsa>(p, cp, t, lane);
        const int nb = t.nb;
        if (nb == 0) {
          // no position of the pair has keys (all padding): zero output, lse -inf
          for (int e = lane; e < 2 * Q.Pq * Q.HG; e += 32) {
            const int i = t.i0 + e % (2 * Q.Pq);
            if (i >= Q.S) continue;
            const size_t lrow = ((size_t)t.b * Q.H + t.g * Q.HG + e / (2 * Q.Pq)) * Q.S + i;
            uint4 *orow = reinterpret_cast<uint4 *>(p.out + lrow * kD);
            for (int c = 0; c < kD / 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[lrow] = -INFINITY;
          }
          continue;
        }
        if (lane == 0) {
          // q buffer gq mod 2: free once pair gq - 2's output has left it, so
          // a pair's q is requested while the pair before it still runs
          const uint32_t qb = gq & 1;
          if (gq >= 2) ok = mbar_wait(&bars.q_empty[qb], ((gq >> 1) - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (ok) {
            // the MMA warps take the pair's geometry from here once q_full completes
            bars.tile[qb] = t;
            const bool has_b = t.i0 + Q.Pq < Q.S;
            mbar_arrive_expect_tx(&bars.q_full[qb], (has_b ? 2 : 1) * kHalves * kHalfTile);
            const int c2 = t.b * Q.H + t.g * Q.HG;
            uint8_t *qdst = smem + kOffQ + qb * kQBuf;
#pragma unroll
            for (int hh = 0; hh < kHalves; ++hh) {
              tma_load_3d(&map_q, &bars.q_full[qb], qdst + hh * kHalfTile, 64 * hh, t.i0, c2);
              if (has_b) tma_load_3d(&map_q, &bars.q_full[qb], qdst + kTile + hh * kHalfTile, 64 * hh, t.i0 + Q.Pq, c2);
            }
            q_issued = (q_issued | (1u << qb)) & ~(1u << (8 + qb));
            q_issued |= ((gq >> 1) & 1u) << (8 + qb);
            // this CTA's next pair: its q rows go to L2 now
            const long long un = u + gridDim.x;
            if (un < p.npairs) {
              Tile tn;
              pair_coords(p, un, tn);
              const int cn = tn.b * Q.H + tn.g * Q.HG;
#pragma unroll
              for (int hh = 0; hh < kHalves; ++hh) {
                tma_prefetch_3d(&map_q, 64 * hh, tn.i0, cn);
                if (tn.i0 + Q.Pq < Q.S) tma_prefetch_3d(&map_q, 64 * hh, tn.i0 + Q.Pq, cn);
              }
            }
          }
          for (int j = 0; !kCsa && ok && j < nb; ++j, ++gb) {
            const int s = gb % kStages;
            if (gb >= (uint32_t)kStages)
              ok = mbar_wait(&bars.kv_empty[s], ((gb / kStages) - 1) & 1, abort_flag, p.status, p.wait_ns);
            if (!ok) break;
            int n, nc;
            block_cols(t, j, n, nc);
            mbar_arrive_expect_tx(&bars.kv_full[s], block_load_bytes<kHalves>(n, nc));
            load_block<kHalves>(t, j, n, nc, &map_kv, &map_ckv, &map_kv16, &map_ckv16, &bars.kv_full[s],
                                smem + kOffKV + s * kTile);
            issued = (issued | (1u << s)) & ~(1u << (8 + s));
            issued |= ((gb / kStages) & 1u) << (8 + s);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        gb = __shfl_sync(0xffffffffu, gb, 0);
        if constexpr (kCsa) {
          // CSA: lane 0 loads the raw rows by TMA; the compressed columns are
          // the pair's union of selected entries, gathered four rows per TMA
          // load (one 16-byte copy per lane and instruction took a warp ~8000
          // cycles per block); every lane joins the block's kv_full arrival
          const long long grp = (long long)t.b * p.ntp + t.i0 / (2 * Q.Pq);
          const int32_t *ent = cp.u_ent + grp * cp.u_cap;
          const uint32_t *msk = cp.u_mask + grp * cp.u_cap;
          const int rb = t.b * Q.Sc;  // row of ckv[b][0] in the row view of map_ckv
          for (int j = 0; ok && j < nb; ++j, ++gb) {
            const int s = gb % kStages;
            int n, nc;
            block_cols(t, j, n, nc);
            // the block's entry ids and selection masks: global loads issued
            // before the wait for a free stage, which hides their latency
            const int4 e4 = 4 * lane < nc ? *reinterpret_cast<const int4 *>(ent + j * kBlockKeys + 4 * lane)
                                          : make_int4(0, 0, 0, 0);
            uint32_t mk[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const int c = 32 * w + lane;
              mk[w] = (c < nc && j * kBlockKeys + c < t.chi) ? msk[j * kBlockKeys + c] : 0u;
            }
            if (gb >= (uint32_t)kStages)
              ok = wait_warp(&bars.kv_empty[s], ((gb / kStages) - 1) & 1, abort_flag, p.status, p.wait_ns);
            if (!ok) break;
            uint8_t *dst = smem + kOffKV + s * kTile;
            if (lane == 0) {
              mbar_expect_tx(&bars.kv_full[s], (nc == n ? 0u : raw_load_bytes(n, nc)) + (uint32_t)nc * 128u * kHalves);
              if (nc < n) load_block_raw(t, j, n, nc, &map_kv, &map_kv16, &bars.kv_full[s], dst);
              issued = (issued | (1u << s)) & ~(1u << (8 + s));
              issued |= ((gb / kStages) & 1u) << (8 + s);
            }
            __syncwarp();  // the expected bytes are set before any gathered row lands
            // compressed columns (nc is a multiple of 16): lane l gathers rows
            // 4l .. 4l + 3, the union's entries, with one TMA gather4 load per
            // 64-column half; padding entries are row 0, which no position sees
            if (4 * lane < nc) {
#pragma unroll
              for (int hh = 0; hh < kHalves; ++hh)
                tma_gather4(&map_ckv, &bars.kv_full[s], dst + hh * kHalfTile + 4 * lane * 128, 64 * hh, rb + e4.x,
                            rb + e4.y, rb + e4.z, rb + e4.w);
            }
            // each pair position's bits for the block's compressed columns
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              for (int pp = 0; pp < 2 * Q.Pq; ++pp) {
                const uint32_t bits = __ballot_sync(0xffffffffu, (mk[w] >> pp) & 1u);
                if (lane == 0) bars.vis[s][pp][w] = bits;
              }
            }
            mbar_arrive(&bars.kv_full[s]);
          }
        }
        ++gq;
      }
      if (ok && lane == 0) {
        // end of the schedule: a pair with nb < 0 in the next slot
        const uint32_t qb = gq & 1;
        if (gq >= 2) ok = mbar_wait(&bars.q_empty[qb], ((gq >> 1) - 1) & 1, abort_flag, p.status, p.wait_ns);
        if (ok) {
          bars.tile[qb].nb = -1;
          mbar_arrive(&bars.q_full[qb]);
        }
      }
      if (!ok && !poisoned && lane == 0) {
        volatile int never = 0;
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) mbar_wait(&bars.kv_full[s], (issued >> (8 + s)) & 1u, &never, p.status, 100000000ull);
        for (int b = 0; b < 2; ++b)
          if (q_issued & (1u << b)) mbar_wait(&bars.q_full[b], (q_issued >> (8 + b)) & 1u, &never, p.status, 100000000ull);
      }
    } else if (warp == 13 || (!kCsa && warp == 14)) {
      // ---------------------------------------------------------- MMA
      // The whole warp runs this loop on warp-uniform values (the pair's
      // ranges are broadcast from lane 0) and one elect.sync lane issues each
      // group of MMAs with its commits.  Operands that the compiler can keep
      // in uniform registers cost ~19 cycles per tcgen05.mma to issue; the
      // same MMAs issued from a lane-0 branch cost 50-80 cycles, more than
      // the tensor pipe needs to execute an M=128, N=128, K=16 step (~65).
      // Descriptors are built once; an MMA only adds a constant offset.
      //
      // Half-block k of a pair is keys [64 (k & 1), 64 (k & 1) + 64) of block
      // k >> 1.  Its S_X goes to TMEM buffer (hb + k) & 1 of tile X, so S_X of
      // half-block k + 1 is ready while the softmax works on k; the order
      //   S_A(0) S_B(0) S_A(1) S_B(1) | PV_A(0) S_A(2) PV_B(0) S_B(2) | ...
      // issues S_X(k + 2) right after PV_X(k), which reads P_X(k) from the
      // same buffer (the tensor pipe runs one thread's MMAs in order).
      const uint64_t dq0 = smem_desc_sw128(smem_u32(smem + kOffQ), 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(smem_u32(smem + kOffQ + kTile), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + kOffKV), 16, 1024);         // K view of stage 0
      const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + kOffKV), kHalfTile, 1024);  // V view of stage 0
      const uint32_t id_pv = idesc_bf16_f32(kRows, kD, false, true);
      const int x0 = kCsa ? 0 : warp - 13, x1 = kCsa ? 2 : x0 + 1;  // tiles this warp issues for
      uint32_t gb = 0, gq = 0, hb = 0;  // blocks, pairs and half-blocks before this pair
      bool ok = !poisoned, issued = false;
      bool ahead = false;  // this pair's S(0) and S(1) went out during the previous pair
      if (ok && p.stall) {
        injected_stall(&bars.never, abort_flag, p.status, p.wait_ns);
        ok = false;
      }
      while (ok) {
        // The pairs with keys, in the TMA warp's order: each one's geometry
        // sits beside its q buffer, so none of it is computed here between
        // two pairs (the range arithmetic took ~2000 cycles of this warp's
        // critical path at every pair boundary).
        ok = wait_warp(&bars.q_full[gq & 1], (gq >> 1) & 1, abort_flag, p.status, p.wait_ns);
        if (!ok) break;
        Tile t = bars.tile[gq & 1];
        uniform_tile(t);
        if (t.nb < 0) break;
        const int nb = t.nb;
        const int nh = half_blocks(t);
        // S_X of half-block k of a pair whose key list has ncols columns, whose
        // q sits in buffer qbuf and whose blocks / half-blocks start at gbb / hbb
        auto issue_s_at = [&](int ncols, uint32_t qbuf, uint32_t gbb, uint32_t hbb, int x, int k) {
          const int n = min(kBlockKeys, ncols - (k >> 1) * kBlockKeys);
          const int h = k & 1;
          const int w = h ? n - kHalfKeys : min(n, kHalfKeys);
          const uint32_t idesc = idesc_bf16_f32(kRows, (w + 15) & ~15, false, false);
          const uint64_t da = (x ? dq1 : dq0) + desc_bytes(qbuf * kQBuf);
          const uint64_t db = dk0 + desc_bytes(((gbb + (k >> 1)) % kStages) * kTile + h * kHalfKeys * 128);
          const uint32_t buf = (hbb + k) & 1;
          const uint32_t d = tmem + col_s(x) + buf * kHalfKeys;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) mma_ss(d, da + kmaj_step(kk), db + kmaj_step(kk), idesc, kk > 0);
            mma_commit(&bars.s_full[x][buf]);
          }
          __syncwarp();
          issued = true;
        };
        auto issue_s = [&](int x, int k) { issue_s_at(t.ncols, gq & 1, gb, hb, x, k); };
        auto issue_pv = [&](int x, int k) {
          int n, nc;
          block_cols(t, k >> 1, n, nc);
          const int h = k & 1;
          const int w = h ? n - kHalfKeys : min(n, kHalfKeys);
          const int nks = (w + 15) >> 4;
          const uint32_t st = (gb + (k >> 1)) % kStages;
          const uint64_t dbv = dv0 + desc_bytes(st * kTile) + mnmaj_step(h * (kHalfKeys / 16));
          const uint32_t d = tmem + col_o(x), a = tmem + col_s(x) + ((hb + k) & 1) * kHalfKeys;
          const uint32_t acc0 = k > 0 ? 1u : 0u;
          if (elect_one()) {
            // a full half goes out as one straight run of MMAs: a branch
            // between tcgen05.mma instructions slows their issue
            if (nks == kHalfKeys / 16) {
              mma_ts(d, a, dbv, id_pv, acc0);
#pragma unroll
              for (int kk = 1; kk < kHalfKeys / 16; ++kk) mma_ts(d, a + kk * 8, dbv + mnmaj_step(kk), id_pv, 1u);
            } else {
              for (int kk = 0; kk < nks; ++kk) mma_ts(d, a + kk * 8, dbv + mnmaj_step(kk), id_pv, kk > 0 ? 1u : acc0);
            }
            mma_commit(&bars.pv_done[x]);
            if (k == nh - 1) mma_commit(&bars.o_final[x]);
            if (x == x1 - 1 && (h == 1 || k == nh - 1)) mma_commit(&bars.kv_empty[st]);
          }
          __syncwarp();
        };
        if (!ahead) {
          ok = wait_warp(&bars.kv_full[gb % kStages], (gb / kStages) & 1, abort_flag, p.status, p.wait_ns);
          if (ok) {
            tc_fence_after();
            for (int x = x0; x < x1; ++x) issue_s(x, 0);
            if (nh > 1)
              for (int x = x0; x < x1; ++x) issue_s(x, 1);
          }
        }
        // The next pair's first two S go out during this pair's last two
        // half-blocks (their buffers are free once PV(nh-2) and PV(nh-1) are
        // issued), so its softmax can start as soon as this pair ends -- if
        // its q and first key block have already landed (checked without
        // waiting; otherwise it starts the usual way).
        int nx_cols = 0;
        for (int k = 0; ok && k < nh; ++k) {
          const int k2 = k + 2;
          if (k2 == nh) {
            const uint32_t gn = gq + 1, bn = gb + nb;
            bool rdy = mbar_test(&bars.q_full[gn & 1], (gn >> 1) & 1);
            const int c = rdy ? bars.tile[gn & 1].ncols : 0;
            rdy = rdy && bars.tile[gn & 1].nb > 0 && mbar_test(&bars.kv_full[bn % kStages], (bn / kStages) & 1);
            nx_cols = __all_sync(0xffffffffu, rdy) ? __shfl_sync(0xffffffffu, c, 0) : 0;
          }
          for (int x = x0; ok && x < x1; ++x) {
            ok = wait_warp(&bars.p_full[x][(hb + k) & 1], ((hb + k) >> 1) & 1, abort_flag, p.status, p.wait_ns);
            if (ok && k == 0 && gq > 0) ok = wait_warp(&bars.o_free[x], (gq - 1) & 1, abort_flag, p.status, p.wait_ns);
            if (!ok) break;
            tc_fence_after();
            issue_pv(x, k);
            if (k2 < nh) {
              if (x == x0 && (k2 & 1) == 0) {
                const uint32_t g2 = gb + (k2 >> 1);
                ok = wait_warp(&bars.kv_full[g2 % kStages], (g2 / kStages) & 1, abort_flag, p.status, p.wait_ns);
                if (!ok) break;
                tc_fence_after();
              }
              issue_s(x, k2);
            } else if (nx_cols > 0 && k2 - nh < 2 && (k2 - nh) * kHalfKeys < nx_cols) {
              tc_fence_after();
              issue_s_at(nx_cols, (gq + 1) & 1, gb + nb, hb + nh, x, k2 - nh);
            }
          }
        }
        ahead = nx_cols > 0;
        gb += nb;
        hb += nh;
        ++gq;
      }
      if (!ok && issued) {
        volatile int never = 0;
        if (elect_one()) mma_commit(&bars.drain[x0]);
        __syncwarp();
        if (lane == 0) mbar_wait(&bars.drain[x0], 0, &never, p.status, 100000000ull);
        __syncwarp();
      }
    }
  } else if (wg == 2) {
    setmaxnreg_dec_epilogue();
    // ------------------------------------------------------------ epilogue
    const int r = tid - 2 * kWG;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t gq = 0, epi_phase = 0;
    bool ok = true;
    auto rendezvous = [&]() -> bool {
      mbar_arrive(&bars.epi);
      const bool rr = wait_warp(&bars.epi, epi_phase & 1, abort_flag, p.status, p.wait_ns);
      ++epi_phase;
      return rr;
    };
    for (long long u = blockIdx.x; ok && !poisoned && u < p.npairs; u += gridDim.x) {
      Tile t;
      pair_coords(p, u, t);
      pair_ranges_warp<kCsa>(p, cp, t, lane);
      const int nb = t.nb;
      if (nb == 0) continue;
      for (int x = 0; ok && x < 2; ++x) {
        const int i0 = t.i0 + x * Q.Pq;
        // tile X's output is staged where its q was: O_X is final only after
        // every MMA of tile X, the S MMAs that read Q_X included, has completed
        uint8_t *obuf = smem + kOffQ + (gq & 1) * kQBuf + x * kTile;
        if (!wait_warp(&bars.o_final[x], gq & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        if (!wait_warp(&bars.st_full[x], gq & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        const float inv = bars.inv_l[x][r];
        mbar_arrive(&bars.st_free[x]);
        tc_fence_after();
        uint32_t o[32];
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          tmem_ld32(lane_addr + col_o(x) + c0, o);
          tmem_wait_ld();
          if (c0 == kD - 32) {
            tc_fence_before();
            mbar_arrive(&bars.o_free[x]);  // O_X may now be overwritten
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv, __uint_as_float(o[ch * 8 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv, __uint_as_float(o[ch * 8 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv, __uint_as_float(o[ch * 8 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv, __uint_as_float(o[ch * 8 + 7]) * inv);
            *reinterpret_cast<uint4 *>(obuf + sw128_offset(r, c0 / 8 + ch)) = v;
          }
        }
        fence_async_smem();
        if (!rendezvous()) { ok = false; break; }
        if (i0 < Q.S) {
          if (r == 0) {
            const int c2 = t.b * Q.H + t.g * Q.HG;
#pragma unroll
            for (int hh = 0; hh < kHalves; ++hh) tma_store_3d(&map_out, obuf + hh * kHalfTile, 64 * hh, i0, c2);
          }
        }
        if (r == 0) bulk_commit();  // one group per staging tile (possibly empty)
      }
      if (!ok) break;
      // the q buffer is free for pair gq + 2 once both stores have read it
      if (r == 0) {
        bulk_wait_read0();
        mbar_arrive(&bars.q_empty[gq & 1]);
      }
      ++gq;
    }
    if (r == 0) bulk_wait0();
  } else {
    setmaxnreg_inc_softmax();
    // ------------------------------------------------------------ softmax of tile X
    const int x = wg;  // 0: tile A, 1: tile B
    const int r = tid - x * kWG;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t hb = 0, gq = 0, scnt = 0;  // half-blocks and pairs before this one; blocks (CSA bits)
    const int pq = r % Q.Pq, hh = r / Q.Pq;
    const int ppos = x * Q.Pq + pq;  // this row's position in the pair (CSA bits)
    if (poisoned) {
      // the ordering check failed: every row is NaN
      for (long long u = blockIdx.x; u < p.npairs; u += gridDim.x) {
        Tile t;
        pair_coords(p, u, t);
        const int i = t.i0 + x * Q.Pq + pq;
        if (i < Q.S) {
          const size_t lrow = ((size_t)t.b * Q.H + t.g * Q.HG + hh) * Q.S + i;
          const float v = __int_as_float(0x7fc00000);
          const uint32_t w2 = pack_bf16x2(v, v);
          uint4 *orow = reinterpret_cast<uint4 *>(p.out + lrow * kD);
#pragma unroll
          for (int c = 0; c < kD / 8; ++c) orow[c] = make_uint4(w2, w2, w2, w2);
          p.lse[lrow] = v;
        }
      }
    }
    bool ok = !poisoned;
    while (ok) {
      // the pairs with keys, in the TMA warp's order, with their geometry
      // (a pair's ranges took this warpgroup ~2000 cycles to work out)
      if (!wait_warp(&bars.q_full[gq & 1], (gq >> 1) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
      const Tile t = bars.tile[gq & 1];
      const int nb = t.nb;
      if (nb < 0) break;
      const int head = t.g * Q.HG + hh;
      const int i = t.i0 + x * Q.Pq + pq;
      const RowIv iv = row_interval(Q.sstart, t.b, Q.S, i, Q.W, Q.m);
      const size_t lrow = ((size_t)t.b * Q.H + head) * Q.S + i;
      const int nh = half_blocks(t);
      float m_run = -INFINITY, l_run = 0.f;
      int a1 = 0, b1 = -1, a2 = 0, b2 = -1;  // the row's visible columns of the block: [a1, b1] compressed, [a2, b2] raw
      uint32_t cbits[4] = {0u, 0u, 0u, 0u};
      for (int k = 0; k < nh; ++k) {
        const int j = k >> 1, h = k & 1;
        int n, nc;
        block_cols(t, j, n, nc);
        const int nk = ((h ? n - kHalfKeys : min(n, kHalfKeys)) + 15) & ~15;
        if (h == 0) row_cols(t, iv, j, n, nc, a1, b1, a2, b2);
        const uint32_t buf = (hb + k) & 1;
        if (!wait_warp(&bars.s_full[x][buf], ((hb + k) >> 1) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        if constexpr (kCsa) {
          if (h == 0) {
            // the block's key tile (with the TMA warp's bits) has landed:
            // the MMA waited for it before S; this wait orders the bits' reads
            const uint32_t sst = scnt % kStages;
            if (!wait_warp(&bars.kv_full[sst], (scnt / kStages) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
#pragma unroll
            for (int w = 0; w < 4; ++w) cbits[w] = iv.valid ? bars.vis[sst][ppos][w] : 0u;
            ++scnt;
          }
        }
        tc_fence_after();
        // One TMEM round trip brings the row's nk scores of this half into
        // registers; the masked row max, then exp2 / row sum / bf16 packing
        // 32 columns at a time.  P_X overwrites the first nk/2 columns of the
        // buffer.  Columns outside the row's two ranges are masked -- that
        // also covers the padding entries and the columns past n of a short
        // block -- and a chunk that every row of the warp sees whole skips
        // the per-element test (warp-uniform).
        const uint32_t sbase = lane_addr + col_s(x) + buf * kHalfKeys;
        uint32_t sv[kHalfKeys];
        tmem_ld32(sbase, *reinterpret_cast<uint32_t(*)[32]>(sv));
        if (32 < nk) tmem_ld32(sbase + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_wait_ld();
        float mx;
        {
          // kPosScale: max of s, scaled after; otherwise min of s (scale < 0)
          const float ninf = kPosScale ? -INFINITY : INFINITY;
          // eight independent 3-input max chains keep the dependency depth short
          float mc[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) mc[q] = ninf;
#pragma unroll
          for (int cc = 0; cc < kHalfKeys; cc += 32) {
            if (cc < nk) {
              const int c0 = h * kHalfKeys + cc;  // column in the block
              if constexpr (kCsa) {
                // compressed columns: this position's selection bits; raw: its window
                const uint32_t vm = cbits[c0 >> 5] | (uint32_t)range_mask64(a2, b2, c0);
                if (!__all_sync(0xffffffffu, vm == 0xffffffffu)) {
#pragma unroll
                  for (int y = 0; y < 32; ++y)
                    if (!((vm >> y) & 1u)) sv[cc + y] = __float_as_uint(ninf);
                }
              } else {
                const bool whole = (c0 >= a1 && c0 + 31 <= b1) || (c0 >= a2 && c0 + 31 <= b2);
                if (!__all_sync(0xffffffffu, whole)) {
                  const uint32_t vm = (uint32_t)(range_mask64(a1, b1, c0) | range_mask64(a2, b2, c0));
#pragma unroll
                  for (int y = 0; y < 32; ++y)
                    if (!((vm >> y) & 1u)) sv[cc + y] = __float_as_uint(ninf);
                }
              }
#pragma unroll
              for (int y = 0; y < 32; y += 16) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const float e0 = __uint_as_float(sv[cc + y + 2 * q]), e1 = __uint_as_float(sv[cc + y + 2 * q + 1]);
                  mc[q] = kPosScale ? fmax3(mc[q], e0, e1) : fmin3(mc[q], e0, e1);
                }
              }
            }
          }
          float m;
          if (kPosScale) {
            const float m0 = fmax3(mc[0], mc[1], mc[2]), m1 = fmax3(mc[3], mc[4], mc[5]);
            m = fmax3(m0, m1, fmaxf(mc[6], mc[7]));
          } else {
            const float m0 = fmin3(mc[0], mc[1], mc[2]), m1 = fmin3(mc[3], mc[4], mc[5]);
            m = fmin3(m0, m1, fminf(mc[6], mc[7]));
          }
          mx = (m == ninf) ? -INFINITY : m * p.sl2;
        }
        float f = 1.f;
        bool rescale_o = false;
        if (mx > m_run + kRescaleLog2 || (m_run == -INFINITY && mx > -INFINITY)) {
          if (m_run > -INFINITY) {
            f = ex2_approx(m_run - mx);
            l_run *= f;
            rescale_o = true;  // an earlier half-block of this pair had visible keys
          }
          m_run = mx;
        }
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        {
          const uint64_t sl2x2 = f32x2(__float_as_uint(p.sl2), __float_as_uint(p.sl2));
          const uint64_t nm2 = f32x2(__float_as_uint(-m_use), __float_as_uint(-m_use));
          uint64_t acc[4] = {0, 0, 0, 0};  // packed row sums (+0.0f bit patterns), four chains
#pragma unroll
          for (int cc = 0; cc < kHalfKeys; cc += 32) {
            if (cc < nk) {
              uint32_t pk[16];
#pragma unroll
              for (int y = 0; y < 32; y += 2) {
                // masked scores are already +-inf, so exp2 gives exactly 0
                float t0, t1;
                f32x2_split(ffma2(f32x2(sv[cc + y], sv[cc + y + 1]), sl2x2, nm2), t0, t1);
                const float e0 = ex2_approx(t0), e1 = ex2_approx(t1);
                const uint64_t e2 = f32x2(__float_as_uint(e0), __float_as_uint(e1));
                acc[(y >> 1) & 3] = fadd2(acc[(y >> 1) & 3], e2);
                pk[y >> 1] = pack_bf16x2(e0, e1);
              }
              tmem_st16(sbase + cc / 2, pk);
            }
          }
          float a0, a1s, b0, b1s;
          f32x2_split(fadd2(acc[0], acc[1]), a0, a1s);
          f32x2_split(fadd2(acc[2], acc[3]), b0, b1s);
          l_run += (a0 + a1s) + (b0 + b1s);
        }
        if (__any_sync(0xffffffffu, rescale_o)) {
          // O_X holds the sum up to half-block k - 1 once that PV completes
          // (S_X(k) only implies PV_X(k - 2))
          if (!wait_warp(&bars.pv_done[x], (hb + k - 1) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[32];
#pragma unroll
          for (int c0 = 0; c0 < kD; c0 += 32) {
            tmem_ld32(lane_addr + col_o(x) + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int y = 0; y < 32; ++y) o[y] = __float_as_uint(__uint_as_float(o[y]) * f);
            tmem_st32(lane_addr + col_o(x) + c0, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.p_full[x][buf]);
      }
      if (!ok) break;
      hb += nh;
      // row statistics: lse to global, 1/l to the epilogue
      if (gq > 0 && !wait_warp(&bars.st_free[x], (gq - 1) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
      bars.inv_l[x][r] = l_run > 0.f ? 1.f / l_run : 0.f;
      mbar_arrive(&bars.st_full[x]);
      if (i < Q.S) {
        float lv = -INFINITY;
        if (l_run > 0.f) {
          float lg;
          asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l_run));
          lv = (m_run + lg) * 0.69314718055994531f;
        }
        p.lse[lrow] = lv;
      }
      ++gq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool tc_fwd_supported(int H, int D, int dtype) { return tc_shape_ok(H, D, dtype); }

int tc_query_tile_positions(int H) { return kRows / heads_per_tile(H); }

cudaError_t tc_fwd(const FwdArgs &a, cudaStream_t st, const CsaUnion *csa) {
  FwdParams p;
  p.qt = make_qtiling(a.sstart, a.B, a.H, a.S, a.W, a.m);
  const QTiling &q = p.qt;
  p.ntp = (q.ntq + 1) / 2;
  p.npairs = (long long)a.B * q.groups * p.ntp;
  CsaParams cp;
  cp.u_cnt = csa ? csa->cnt : nullptr;
  cp.u_ent = csa ? csa->ent : nullptr;
  cp.u_mask = csa ? csa->mask : nullptr;
  cp.u_cap = csa ? csa->cap : 0;
  cp.ckv = static_cast<const __nv_bfloat16 *>(a.ckv);
  CUtensorMap mq, mkv, mckv, mkv16, mckv16, mout;
  const uint64_t D = (uint64_t)a.D;
  if (!make_map_bf16(&mq, a.q, D, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mout, a.out, D, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mkv, a.kv, D, a.S, a.B, kBlockKeys, 1) ||
      // CSA gathers its compressed rows through the 2-D row view of ckv
      !(csa ? make_map_rows_bf16(&mckv, a.ckv, D, (uint64_t)q.Sc * a.B)
            : make_map_bf16(&mckv, a.ckv, D, q.Sc, a.B, kBlockKeys, 1)) ||
      !make_map_bf16(&mkv16, a.kv, D, a.S, a.B, 16, 1) ||
      !make_map_bf16(&mckv16, a.ckv, D, q.Sc, a.B, 16, 1))
    return cudaErrorInvalidValue;
  p.status = a.status_rw;
  p.lse = a.lse;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.sl2 = a.scale * 1.4426950408889634f;
  p.wait_ns = a.wait_ns;
  p.stall = a.stall;
  const bool pos = p.sl2 > 0.f;
  if (csa && a.D != 128) return cudaErrorInvalidValue;
  const int which = (pos ? 1 : 0) + (csa ? 2 : 0) + (a.D == 64 ? 4 : 0);
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               const CUtensorMap, const FwdParams, const CsaParams) =
      which == 0   ? hca_fwd_tc_kernel<false, false, 128>
      : which == 1 ? hca_fwd_tc_kernel<true, false, 128>
      : which == 2 ? hca_fwd_tc_kernel<false, true, 128>
      : which == 3 ? hca_fwd_tc_kernel<true, true, 128>
      : which == 4 ? hca_fwd_tc_kernel<false, false, 64>
                   : hca_fwd_tc_kernel<true, false, 64>;
  static SmemAttrOnce attr[6];
  cudaError_t e = attr[which].ensure(reinterpret_cast<const void *>(kern), kSmemBytes);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const long long grid = p.npairs < sms ? p.npairs : sms;
  if (grid == 0) return cudaSuccess;
  ProfScope prof(kKFwdTc, st);
  kern<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(mq, mkv, mckv, mkv16, mckv16, mout, p, cp);
  return cudaGetLastError();
}

}  // namespace hca
