// hca_bwd_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) HCA backward, sm_103a.
//
// Gradient of the forward in hca_fwd_tc.cu (same visibility, K = V):
//   P = exp(s - lse), dP = dO K^T, Delta = rowsum(dO * out), dS = P (dP - Delta)
//   dq  = scale * dS K
//   dkv = sum over heads and visible queries of (scale * dS^T q + P^T dO),
// i.e. each shared row receives its key-role and its value-role gradient in
// one accumulator ("[DeepSeek-V4] Implement Compressed Attention Layers",
// einsum review suggestions: k and v are the same kv tensor).
//
// Three kernels on the caller's stream:
//  1. dq kernel (query-major, the forward's tiles and key blocks).  Per tile
//     it also forms Delta from the TMA-loaded dO tile and the stored out rows
//     and writes (lse*log2e, Delta) in tile-row order for kernel 2.  Per key
//     block: S = Q K^T and dP = dO K^T share the kv tile; the softmax warps
//     form dS (bf16) straight into TMEM; dq += dS K reads dS from TMEM and the
//     kv tile through an MN-major descriptor.
//  2. dkv kernel (key-major).  A work item is a range of head-packed query
//     tiles and one or two 128-key blocks of one kind; each 64-row query
//     sub-tile is loaded once and serves both blocks:
//       S^T = K Q^T, dP^T = K dO^T  ->  P^T, dS^T (bf16, into TMEM)
//       acc_a += P^T dO + (scale dS^T) Q    (one fp32 TMEM accumulator per block)
//     Raw items cover 128 query positions and the (up to two) raw blocks they
//     see; compressed items cover a slice of the queries that see a pair of
//     compressed blocks.  Every item writes fp32 partial sums.
//     The dQ side needs no atomics: kernel 1 owns dq.  ("Add HCA Static
//     Compilation for Splash Attention [Deepseek v4]" reduces dQ in an on-chip
//     ring buffer on TPU; here dq stays in TMEM for a whole query tile.)
//  3. reduce kernel: dkv and dckv = sums of their partials in a fixed order
//     (deterministic).
#include <cuda_bf16.h>

#include "hca_common.cuh"
#include "hca_internal.h"
#include "tc_ptx.cuh"
#include "tc_tiles.cuh"

namespace hca {
using namespace tc;

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// kernel 1: dq
// ---------------------------------------------------------------------------
namespace dqk {
constexpr int kStages = 3;
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;  // dS: 64 cols of packed bf16
constexpr int kTmemCols = 512;
// two dS warpgroups (each owns 64 of a row's 128 key columns); warpgroup 2:
// TMA warp (also the tile descriptors), MMA warp, two Delta warps
constexpr int kEW = 256;
constexpr int kThreads = kEW + 128;
// 12 warps put 3 on each SM sub-partition (16K registers each): 168 per
// thread at launch; the TMA/MMA warpgroup gives registers to the other two
constexpr int kRegEW = 208, kRegProducer = 88;
static_assert(2 * 128 * kRegEW + 128 * kRegProducer <= kThreads * 168, "register split must fit the launch");
// shared memory: Q | dO | out (for Delta) | kv ring | dq staging (+1 KB align)
constexpr int kOffQ = 0, kOffDO = kTile, kOffO = 2 * kTile, kOffKV = 3 * kTile;
constexpr int kOffOut = kOffKV + kStages * kTile;
constexpr int kSmemBytes = kOffOut + kTile + 1024;
constexpr int kDescSlots = 8;
constexpr int kDescReaders = 11;  // dS warps 0-7, MMA warp 9, Delta warps 10-11 (CSA: warp 11 alone forms Delta)
constexpr int kDeltaThreads = 64;
constexpr int kCsaMaxPos = 4;     // CSA: positions per tile whose bits are kept (Pq <= 4)
}  // namespace dqk

struct DqParams {
  QTiling qt;
  // CSA: per tile, the union of its positions' selected entries (hca_csa.cu)
  const int32_t *u_cnt, *u_ent;
  const uint32_t *u_mask;
  int u_cap;
  const __nv_bfloat16 *ckv;
  int32_t *status;
  const float *lse;
  float *rowstat;            // [ntiles][2][128]: -lse*log2e, then -scale*Delta, per tile row
  __nv_bfloat16 *dq;         // direct stores for poisoned calls / tiles without keys
  float sl2, scale;
  int pq_shift;              // log2(Pq)
  uint64_t wait_ns;          // limit of every bounded wait
  int stall;                 // failure-path test: the MMA warp first waits on a barrier nothing arrives at
};

// One query tile of the CTA's schedule as every role needs it (u < 0 ends it).
struct DqDesc {
  long long u;
  int b, g, i0, rlo, rhi, clo, chi, cpad, ncols, nb;
};

struct DqBars {
  uint64_t qd_full, qd_empty;
  uint64_t kv_full[dqk::kStages], kv_empty[dqk::kStages];
  uint64_t s_full, s_free;   // S of a block in TMEM / read out by the dS warps
  uint64_t dp_full, ds_full; // dP in TMEM / dS stored (and dP read out)
  uint64_t dq_done;          // a tile's last dq MMA complete
  uint64_t stat_full, stat_empty;  // a tile's Delta in shared memory / read by the dS warps
  uint64_t desc_full[dqk::kDescSlots], desc_empty[dqk::kDescSlots];
  uint64_t epi, drain, never;
  DqDesc desc[dqk::kDescSlots];
  float delta[kRows];
  uint32_t vis[dqk::kStages][dqk::kCsaMaxPos][4];  // CSA: per block, each position's bits of the compressed columns
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ long long tile_linear(const QTiling &q, const Tile &t) {
  return ((long long)t.b * q.groups + t.g) * q.ntq + t.i0 / q.Pq;
}

// Reads tile descriptor kd (bounded wait) and releases its slot; false when
// the wait gave up.
__device__ __forceinline__ bool read_dq_desc(DqBars &bars, uint32_t kd, Tile &t, long long &u, volatile int *abort,
                                             int32_t *status, uint64_t wait_ns) {
  const int slot = kd % dqk::kDescSlots;
  if (!wait_warp(&bars.desc_full[slot], (kd / dqk::kDescSlots) & 1, abort, status, wait_ns)) return false;
  const volatile DqDesc &d = bars.desc[slot];
  u = d.u;
  t.b = d.b; t.g = d.g; t.i0 = d.i0;
  t.rlo = d.rlo; t.rhi = d.rhi; t.clo = d.clo; t.chi = d.chi;
  t.cpad = d.cpad; t.ncols = d.ncols; t.nb = d.nb;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&bars.desc_empty[slot]);
  return true;
}

template <bool kCsa, int kD>
__global__ void __launch_bounds__(dqk::kThreads, 1)
    hca_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                      const __grid_constant__ CUtensorMap map_out,
                      const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_ckv,
                      const __grid_constant__ CUtensorMap map_kv16, const __grid_constant__ CUtensorMap map_ckv16,
                      const __grid_constant__ CUtensorMap map_dq, const DqParams p) {
  using namespace dqk;
  static_assert(kD == 64 || kD == 128, "head dim 64 or 128");
  static_assert(!kCsa || kD == 128, "CSA gathers 128-dim rows");
  constexpr int kHalves = kD / 64;   // 64-column (128-byte) halves of a row
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DqBars bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int *abort_flag = &bars.abort;
  const QTiling &Q = p.qt;

  if (tid == 0) {
    mbar_init(&bars.qd_full, 1);
    // released by the last S/dP MMA of a tile and by every Delta thread once
    // it has read the staged dO and out tiles
    mbar_init(&bars.qd_empty, 1 + (kCsa ? 32 : kDeltaThreads));
    for (int s = 0; s < kStages; ++s) {
      // CSA: every lane of the TMA warp arrives once its gather loads are
      // issued and the visibility bits written
      mbar_init(&bars.kv_full[s], kCsa ? 32 : 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, kEW);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.ds_full, kEW);
    mbar_init(&bars.dq_done, 1);
    mbar_init(&bars.stat_full, kCsa ? 32 : kDeltaThreads);
    mbar_init(&bars.stat_empty, kEW);
    for (int s = 0; s < kDescSlots; ++s) {
      mbar_init(&bars.desc_full[s], 32);
      mbar_init(&bars.desc_empty[s], kCsa ? kDescReaders - 1 : kDescReaders);
    }
    mbar_init(&bars.epi, kEW);
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.never, 1);
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

  if (warp >= kEW / 32) {
    setmaxnreg_dec<kRegProducer>();
    if (warp == kEW / 32) {
      // ------------------------------------------------------------ TMA + tile descriptors
      // Every tile of the CTA's schedule (then an end marker) is published
      // to the other roles through a shared-memory ring, so its key ranges
      // are computed once; then its operands are loaded.
      uint32_t gb = 0, tw = 0;
      int last_par[kStages] = {-1, -1, -1};
      int q_par = -1;
      bool ok = true;
      for (uint32_t k = 0; ok; ++k) {
        const long long u = (long long)blockIdx.x + (long long)k * gridDim.x;
        const bool end = u >= Q.ntiles;
        Tile t;
        t.b = t.g = t.i0 = 0;
        t.rlo = t.rhi = t.clo = t.chi = t.cpad = t.ncols = t.nb = 0;
        if (!end) {
          tile_coords(Q, u, t);
          tile_ranges_warp(Q, t, lane);
          if (kCsa) {
            // compressed columns: the tile's union of selected entries
            const int cnt = p.u_cnt[(long long)t.b * Q.ntq + t.i0 / Q.Pq];
            t.clo = 0;
            t.chi = cnt;
            t.cpad = (cnt + 15) & ~15;
            t.ncols = t.cpad + (t.rhi - t.rlo);
            t.nb = (t.ncols + kBlockKeys - 1) / kBlockKeys;
          }
        }
        const int slot = k % kDescSlots;
        if (k >= (uint32_t)kDescSlots &&
            !wait_warp(&bars.desc_empty[slot], ((k / kDescSlots) - 1) & 1, abort_flag, p.status, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          volatile DqDesc &d = bars.desc[slot];
          d.u = end ? -1 : u;
          d.b = t.b; d.g = t.g; d.i0 = t.i0;
          d.rlo = t.rlo; d.rhi = t.rhi; d.clo = t.clo; d.chi = t.chi;
          d.cpad = t.cpad; d.ncols = t.ncols; d.nb = t.nb;
        }
        __syncwarp();
        mbar_arrive(&bars.desc_full[slot]);
        if (end) break;
        const int nb = t.nb;
        if (poisoned || nb == 0) continue;
        if (lane == 0) {
          if (tw > 0) ok = mbar_wait(&bars.qd_empty, (tw - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (ok) {
            mbar_arrive_expect_tx(&bars.qd_full, 3 * kHalves * kHalfTile);
            const int c2 = t.b * Q.H + t.g * Q.HG;
#pragma unroll
            for (int hh = 0; hh < kHalves; ++hh) {
              tma_load_3d(&map_q, &bars.qd_full, smem + kOffQ + hh * kHalfTile, 64 * hh, t.i0, c2);
              tma_load_3d(&map_do, &bars.qd_full, smem + kOffDO + hh * kHalfTile, 64 * hh, t.i0, c2);
              tma_load_3d(&map_out, &bars.qd_full, smem + kOffO + hh * kHalfTile, 64 * hh, t.i0, c2);
            }
            q_par = tw & 1;
            // this CTA's next tile: its q, dO and out rows go to L2 now, so
            // the loads at the tile boundary do not wait on HBM
            const long long un = u + gridDim.x;
            if (un < Q.ntiles) {
              Tile tn;
              tile_coords(Q, un, tn);
              const int cn = tn.b * Q.H + tn.g * Q.HG;
#pragma unroll
              for (int hh = 0; hh < kHalves; ++hh) {
                tma_prefetch_3d(&map_q, 64 * hh, tn.i0, cn);
                tma_prefetch_3d(&map_do, 64 * hh, tn.i0, cn);
                tma_prefetch_3d(&map_out, 64 * hh, tn.i0, cn);
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
            last_par[s] = (gb / kStages) & 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        gb = __shfl_sync(0xffffffffu, gb, 0);
        if constexpr (kCsa) {
          // CSA: lane 0 loads the raw rows by TMA; the compressed columns are
          // the tile's union of selected entries, gathered four rows per TMA
          // load (the row view of ckv in map_ckv); every lane joins the
          // block's kv_full arrival once its loads are issued and the
          // positions' visibility bits are written
          const long long grp = (long long)t.b * Q.ntq + t.i0 / Q.Pq;
          const int32_t *ent = p.u_ent + grp * p.u_cap;
          const uint32_t *msk = p.u_mask + grp * p.u_cap;
          const int rb = t.b * Q.Sc;  // row of ckv[b][0] in the row view
          for (int j = 0; ok && j < nb; ++j, ++gb) {
            const int s = gb % kStages;
            int n, nc;
            block_cols(t, j, n, nc);
            // entry ids and selection masks, loaded before the wait for a stage
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
              last_par[s] = (gb / kStages) & 1;
            }
            __syncwarp();  // the expected bytes are set before any gathered row lands
            // nc is a multiple of 16: lane l gathers rows 4l .. 4l + 3 (padding
            // entries are row 0, which no position sees)
            if (4 * lane < nc) {
#pragma unroll
              for (int hh = 0; hh < kHalves; ++hh)
                tma_gather4(&map_ckv, &bars.kv_full[s], dst + hh * kHalfTile + 4 * lane * 128, 64 * hh, rb + e4.x,
                            rb + e4.y, rb + e4.z, rb + e4.w);
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              for (int pp = 0; pp < Q.Pq; ++pp) {
                const uint32_t bits = __ballot_sync(0xffffffffu, (mk[w] >> pp) & 1u);
                if (lane == 0) bars.vis[s][pp][w] = bits;
              }
            }
            mbar_arrive(&bars.kv_full[s]);
          }
        }
        ++tw;
      }
      if (!ok && !poisoned && lane == 0) {
        volatile int never = 0;
        for (int s = 0; s < kStages; ++s)
          if (last_par[s] >= 0) mbar_wait(&bars.kv_full[s], last_par[s], &never, p.status, 100000000ull);
        if (q_par >= 0) mbar_wait(&bars.qd_full, q_par, &never, p.status, 100000000ull);
      }
    } else if (warp == kEW / 32 + 1) {
      // ------------------------------------------------------------ MMA
      // Whole warp, warp-uniform values, one elect.sync lane issues (cheap
      // tcgen05.mma issue from uniform registers; see the forward kernel).
      // Per key block j the order is  S(j+1) | dq(j) | dP(j+1):  S(j+1) goes
      // out as soon as the dS warps hold P(j) in registers, so the tensor pipe
      // runs it while they form dS(j).  dP(j+1) overwrites dP(j) only after
      // dS(j) is stored, and its commit also covers dq(j) (one thread's MMAs
      // complete in order), so dS(j+1) never overwrites a dS that an
      // unfinished dq MMA still reads.
      const uint64_t dQ = smem_desc_sw128(smem_u32(smem + kOffQ), 16, 1024);
      const uint64_t dDO = smem_desc_sw128(smem_u32(smem + kOffDO), 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(smem_u32(smem + kOffKV), 16, 1024);
      const uint64_t dV0 = smem_desc_sw128(smem_u32(smem + kOffKV), kHalfTile, 1024);
      const uint32_t id_dq = idesc_bf16_f32(kRows, kD, false, true);
      uint32_t gb = 0, tw = 0, kd = 0;
      bool ok = true, issued = false;
      if (!poisoned && p.stall) {
        injected_stall(&bars.never, abort_flag, p.status, p.wait_ns);
        ok = false;
      }
      while (ok) {
        Tile t;
        long long u;
        ok = read_dq_desc(bars, kd++, t, u, abort_flag, p.status, p.wait_ns);
        if (!ok || u < 0) break;
        const int nb = t.nb;
        if (poisoned || nb == 0) continue;
        // S (x = 0) or dP (x = 1) of block j into its TMEM columns
        auto issue_sdp = [&](int x, int j, uint32_t g, bool last_q_use) {
          int n, nc;
          block_cols(t, j, n, nc);
          const uint32_t idesc = idesc_bf16_f32(kRows, (n + 15) & ~15, false, false);
          const uint64_t bk = dK0 + desc_bytes((g % kStages) * kTile);
          const uint64_t da = x ? dDO : dQ;
          const uint32_t d = tmem + (x ? kColDP : kColS);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < kD / 16; ++k) mma_ss(d, da + kmaj_step(k), bk + kmaj_step(k), idesc, k > 0);
            mma_commit(x ? &bars.dp_full : &bars.s_full);
            if (last_q_use) mma_commit(&bars.qd_empty);
          }
          __syncwarp();
          issued = true;
        };
        ok = wait_warp(&bars.qd_full, tw & 1, abort_flag, p.status, p.wait_ns);
        if (ok) ok = wait_warp(&bars.kv_full[gb % kStages], (gb / kStages) & 1, abort_flag, p.status, p.wait_ns);
        // the previous tile's last S must have been read out
        if (ok && gb > 0) ok = wait_warp(&bars.s_free, (gb - 1) & 1, abort_flag, p.status, p.wait_ns);
        if (ok) {
          tc_fence_after();
          issue_sdp(0, 0, gb, false);
          issue_sdp(1, 0, gb, nb == 1);
        }
        for (int j = 0; ok && j < nb; ++j) {
          const uint32_t g = gb + j;
          const bool next = j + 1 < nb;
          if (next) {
            ok = wait_warp(&bars.s_free, g & 1, abort_flag, p.status, p.wait_ns);
            if (ok) ok = wait_warp(&bars.kv_full[(g + 1) % kStages], ((g + 1) / kStages) & 1, abort_flag, p.status, p.wait_ns);
            if (!ok) break;
            tc_fence_after();
            issue_sdp(0, j + 1, g + 1, false);
          }
          ok = wait_warp(&bars.ds_full, g & 1, abort_flag, p.status, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          int n, nc;
          block_cols(t, j, n, nc);
          const int nks = (n + 15) >> 4;
          const int s = g % kStages;
          const uint64_t bv = dV0 + desc_bytes(s * kTile);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
          if (elect_one()) {
            // a full block goes out as one straight run of MMAs: a branch
            // between tcgen05.mma instructions slows their issue
            if (nks == kBlockKeys / 16) {
              mma_ts(tmem + kColDQ, tmem + kColDS, bv, id_dq, acc0);
#pragma unroll
              for (int kk = 1; kk < kBlockKeys / 16; ++kk)
                mma_ts(tmem + kColDQ, tmem + kColDS + kk * 8, bv + mnmaj_step(kk), id_dq, 1u);
            } else {
              for (int kk = 0; kk < nks; ++kk)
                mma_ts(tmem + kColDQ, tmem + kColDS + kk * 8, bv + mnmaj_step(kk), id_dq, kk > 0 ? 1u : acc0);
            }
            mma_commit(&bars.kv_empty[s]);
            if (!next) mma_commit(&bars.dq_done);
          }
          __syncwarp();
          if (next) issue_sdp(1, j + 1, g + 1, j + 1 == nb - 1);
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
    } else if (kCsa && warp == kEW / 32 + 2) {
      // CSA: idle (the TMA warp gathers the selected rows); it is not counted
      // among the tile descriptors' readers
    } else {
      // ------------------------------------------------------------ Delta
      // Delta = <dO, out> of every tile row from the staged dO and out tiles
      // (two warps, 64 rows each, two rows per lane; CSA: one warp, four rows
      // per lane), off the dS warps' critical path; published in shared
      // memory and, as -scale*Delta, in the row records the dkv kernel reads.
      constexpr int kRowsPerLane = kCsa ? 4 : 2;
      const int dt = kCsa ? lane : tid - (kEW + 64);
      uint32_t tw = 0, kd = 0;
      bool ok = true;
      const uint8_t *dobuf = smem + kOffDO;
      const uint8_t *outbuf = smem + kOffO;
      while (ok) {
        Tile t;
        long long u;
        ok = read_dq_desc(bars, kd++, t, u, abort_flag, p.status, p.wait_ns);
        if (!ok || u < 0) break;
        if (poisoned || t.nb == 0) continue;
        if (!wait_warp(&bars.qd_full, tw & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        float dl[kRowsPerLane];
#pragma unroll
        for (int h = 0; h < kRowsPerLane; ++h) {
          dl[h] = 0.f;
          const int r = dt + (kRows / kRowsPerLane) * h;
#pragma unroll 4
          for (int ch = 0; ch < kD / 8; ++ch) {
            const uint4 ov = *reinterpret_cast<const uint4 *>(outbuf + sw128_offset(r, ch));
            const uint4 gv = *reinterpret_cast<const uint4 *>(dobuf + sw128_offset(r, ch));
            const uint32_t oa[4] = {ov.x, ov.y, ov.z, ov.w}, ga[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              dl[h] = fmaf(__uint_as_float(oa[x] << 16), __uint_as_float(ga[x] << 16), dl[h]);
              dl[h] = fmaf(__uint_as_float(oa[x] & 0xffff0000u), __uint_as_float(ga[x] & 0xffff0000u), dl[h]);
            }
          }
        }
        mbar_arrive(&bars.qd_empty);  // dO and out of this tile are read
        float *rs = p.rowstat + tile_linear(Q, t) * 2 * kRows;
#pragma unroll
        for (int h = 0; h < kRowsPerLane; ++h) rs[kRows + dt + (kRows / kRowsPerLane) * h] = -p.scale * dl[h];
        // the dS warps have read the previous tile's Delta
        if (tw > 0 && !wait_warp(&bars.stat_empty, (tw - 1) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
#pragma unroll
        for (int h = 0; h < kRowsPerLane; ++h) bars.delta[dt + (kRows / kRowsPerLane) * h] = dl[h];
        mbar_arrive(&bars.stat_full);
        ++tw;
      }
    }
  } else {
    setmaxnreg_inc<kRegEW>();
    // ------------------------------------------------------------ dS + epilogue
    // thread r of warpgroup wg owns row r (TMEM lane r) and key columns
    // [64 wg, 64 wg + 64) of every block (and dq columns [64 wg, 64 wg + 64))
    const int r = tid & (kRows - 1), wg = tid >> 7;
    const int cb = wg * 64;            // key columns of a block
    const int cbq = wg * (kD / 2);     // dq columns
    const int pq = r & (Q.Pq - 1), hh = r >> p.pq_shift;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint8_t *obuf = smem + kOffOut;
    uint32_t gb = 0, tw = 0, epi_phase = 0, kd = 0;
    const uint64_t sl2x2 = f32x2(__float_as_uint(p.sl2), __float_as_uint(p.sl2));
    bool ok = true, store_pending = false;
    auto rendezvous = [&]() -> bool {
      mbar_arrive(&bars.epi);
      const bool rr = wait_warp(&bars.epi, epi_phase & 1, abort_flag, p.status, p.wait_ns);
      ++epi_phase;
      return rr;
    };
    while (ok) {
      Tile t;
      long long u;
      ok = read_dq_desc(bars, kd++, t, u, abort_flag, p.status, p.wait_ns);
      if (!ok || u < 0) break;
      const int nb = t.nb;
      const int head = t.g * Q.HG + hh;
      const int i = t.i0 + pq;
      const RowIv iv = row_interval(Q.sstart, t.b, Q.S, i, Q.W, Q.m);
      const size_t lrow = ((size_t)t.b * Q.H + head) * Q.S + i;
      float *rs = p.rowstat + tile_linear(Q, t) * 2 * kRows;
      if (poisoned || nb == 0) {
        if (i < Q.S) {
          const float v = poisoned ? __int_as_float(0x7fc00000) : 0.f;
          const uint32_t w2 = pack_bf16x2(v, v);
          uint4 *grow = reinterpret_cast<uint4 *>(p.dq + lrow * kD + cbq);
#pragma unroll
          for (int c = 0; c < kD / 16; ++c) grow[c] = make_uint4(w2, w2, w2, w2);
        }
        if (wg == 0) {
          rs[r] = 0.f;
          rs[kRows + r] = 0.f;
        }
        continue;
      }
      const float lse2 = iv.valid ? p.lse[lrow] * kLog2e : 0.f;
      if (wg == 0) rs[r] = -lse2;
      float delta = 0.f;
      for (int j = 0; j < nb; ++j, ++gb) {
        int n, nc;
        block_cols(t, j, n, nc);
        const int nk = (n + 15) & ~15;
        // visible columns [cb, cb + 64) of this row: its compressed range and
        // its raw range in the block
        int a1, b1, a2, b2;
        row_cols(t, iv, j, n, nc, a1, b1, a2, b2);
        uint64_t vis = kCsa ? range_mask64(a2, b2, cb) : (range_mask64(a1, b1, cb) | range_mask64(a2, b2, cb));
        if (!wait_warp(&bars.s_full, gb & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        if (kCsa) {
          // the block's key tile (with the TMA warp's bits) has landed;
          // this wait orders the bits' reads
          const int s = gb % kStages;
          if (!wait_warp(&bars.kv_full[s], (gb / kStages) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
          if (iv.valid) vis |= (uint64_t)bars.vis[s][pq][2 * wg] | ((uint64_t)bars.vis[s][pq][2 * wg + 1] << 32);
        }
        tc_fence_after();
        // P = exp2(S * scale * log2e - lse * log2e), kept in registers so the
        // S columns can take the next block's scores right away
        uint32_t pv[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          if (cb + c0 < nk) {
            tmem_ld32(lane_addr + kColS + cb + c0, *reinterpret_cast<uint32_t(*)[32]>(pv + c0));
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) pv[c0 + x] = 0u;
          }
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars.s_free);
        const uint64_t nl2 = f32x2(__float_as_uint(-lse2), __float_as_uint(-lse2));
        // warp-uniform cases: nothing visible, everything visible, or a mix
        const bool none = __all_sync(0xffffffffu, vis == 0ull);
        const bool all = __all_sync(0xffffffffu, vis == ~0ull);
        if (none) {
#pragma unroll
          for (int c = 0; c < 64; ++c) pv[c] = 0u;
        } else if (all) {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float t0, t1;
            f32x2_split(ffma2(f32x2(pv[c], pv[c + 1]), sl2x2, nl2), t0, t1);
            pv[c] = __float_as_uint(ex2_approx(t0));
            pv[c + 1] = __float_as_uint(ex2_approx(t1));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float t0, t1;
            f32x2_split(ffma2(f32x2(pv[c], pv[c + 1]), sl2x2, nl2), t0, t1);
            pv[c] = ((vis >> c) & 1ull) ? __float_as_uint(ex2_approx(t0)) : 0u;
            pv[c + 1] = ((vis >> (c + 1)) & 1ull) ? __float_as_uint(ex2_approx(t1)) : 0u;
          }
        }
        if (j == 0) {
          // this tile's Delta, from the Delta warps
          if (!wait_warp(&bars.stat_full, tw & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
          delta = bars.delta[r];
          mbar_arrive(&bars.stat_empty);
        }
        if (!wait_warp(&bars.dp_full, gb & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ndl2 = f32x2(__float_as_uint(-delta), __float_as_uint(-delta));
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          if (cb + c0 >= nk) break;
          uint32_t packed[16];
          if (none) {
#pragma unroll
            for (int x = 0; x < 16; ++x) packed[x] = 0u;
          } else {
            uint32_t dr[32];
            tmem_ld32(lane_addr + kColDP + cb + c0, dr);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; x += 2) {
              const int c = c0 + x;
              // dS = P (dP - Delta); columns past the block (stale TMEM) are zero
              float d0, d1;
              f32x2_split(fmul2(f32x2(pv[c], pv[c + 1]), fadd2(f32x2(dr[x], dr[x + 1]), ndl2)), d0, d1);
              if (!all) {
                d0 = ((vis >> c) & 1ull) ? d0 : 0.f;
                d1 = ((vis >> (c + 1)) & 1ull) ? d1 : 0.f;
              }
              packed[x / 2] = pack_bf16x2(d0, d1);
            }
          }
          tmem_st16(lane_addr + kColDS + (cb + c0) / 2, packed);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.ds_full);
      }
      if (!ok) break;
      // ---------------- epilogue: dq = scale * acc
      if (!wait_warp(&bars.dq_done, tw & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
      tc_fence_after();
      if (store_pending) {
        if (tid == 0) bulk_wait_read0();
        if (!rendezvous()) { ok = false; break; }
        store_pending = false;
      }
      {
        uint32_t o[32];
#pragma unroll
        for (int c0 = cbq; c0 < cbq + kD / 2; c0 += 32) {
          tmem_ld32(lane_addr + kColDQ + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * p.scale, __uint_as_float(o[ch * 8 + 1]) * p.scale);
            v.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * p.scale, __uint_as_float(o[ch * 8 + 3]) * p.scale);
            v.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * p.scale, __uint_as_float(o[ch * 8 + 5]) * p.scale);
            v.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * p.scale, __uint_as_float(o[ch * 8 + 7]) * p.scale);
            *reinterpret_cast<uint4 *>(obuf + sw128_offset(r, c0 / 8 + ch)) = v;
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      if (!rendezvous()) { ok = false; break; }
      if (tid == 0) {
        const int c2 = t.b * Q.H + t.g * Q.HG;
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) tma_store_3d(&map_dq, obuf + hh * kHalfTile, 64 * hh, t.i0, c2);
        bulk_commit();
      }
      store_pending = true;
      ++tw;
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
// kernel 2: dkv / dckv partials
// ---------------------------------------------------------------------------
namespace dkk {
// A work item is a range of query tiles and one or two 128-key blocks of one
// kind (raw or compressed).  The item streams 64-row query sub-tiles through
// shared memory once and uses each for both key blocks, so a query row is
// fetched about half as often as with one key block per item.  Shared memory
// holds a sub-tile as one 128-row operand R = [Q_sub ; dO_sub] (64 rows each,
// per 64-column half): a single N = 128 MMA K R^T yields S^T (columns 0-63)
// and dP^T (columns 64-127) of the sub-tile for one key block.
// two P^T/dS^T warpgroups (each takes 32 of every unit's 64 query columns
// and 64 of a key row's 128 accumulator columns), TMA warp, MMA warp
constexpr int kEW = 256;
constexpr int kThreads = kEW + 128;
// 12 warps put 3 on each SM sub-partition (16K registers each): 168 per
// thread at launch; the TMA/MMA warpgroup gives registers to the other two
constexpr int kRegEW = 208, kRegProducer = 88;
static_assert(2 * 128 * kRegEW + 128 * kRegProducer <= kThreads * 168, "register split must fit the launch");
constexpr int kStages = 4;                     // sub-tiles in flight
constexpr int kSubBytes = kTile;               // one operand R (two halves)
constexpr int kHalfRows = 64;                  // rows of Q_sub (and of dO_sub)
constexpr int kOffRowstat = kSubBytes;         // -lse*log2e [64] then -scale*Delta [64]
constexpr int kOffIv = kOffRowstat + 512;      // per-position intervals (rlo, rhi, clo, chi) [<= 64]
constexpr int kStageBytes = kOffIv + 1024 + 512;  // 34 KB: every stage stays 1 KB aligned
constexpr int kOffK = 0;                       // key block tiles A | B
constexpr int kOffStage = 2 * kTile;
constexpr int kSmemBytes = kOffStage + kStages * kStageBytes + 1024;
// TMEM: two [S^T | dP^T] buffers (packed bf16 P^T and dS^T overwrite the
// S^T columns: query rows 0-31 at columns 0-15 / 16-31, rows 32-63 at 32-47 /
// 48-63), then one fp32 accumulator per key block
constexpr uint32_t kColAcc = 256;
constexpr int kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_buf(uint32_t g) { return (g & 1u) * 128u; }
__host__ __device__ constexpr uint32_t col_acc(int a) { return kColAcc + (uint32_t)a * 128u; }
// Query-range splits of the compressed items.  They are fixed numbers so
// the partial buffers grow linearly with the sequence length.
constexpr int kSplitBoth = 128;  // compressed blocks 2c, 2c+1 where both are visible
constexpr int kSplitLead = 32;   // block 2c alone, before block 2c+1 is visible
constexpr int kSlotsComp = kSplitLead + kSplitBoth;
}  // namespace dkk

struct DkvParams {
  QTiling qt;
  int32_t *status;
  int32_t *next_item;  // work counter (zeroed before the launch)
  const float *rowstat;
  float *rpart;  // raw partials [nslot][B][S_pad][D] fp32: slot = query range - key block
                 // (one slot, accumulated with atomics, when raw_atomic)
  float *cpart;  // compressed partials [kSlotsComp][B][Sc_pad][D] fp32
  int nrb, nkb_comp, S_pad, Sc_pad, nslot, npr;
  int raw_atomic;      // raw partials summed with fp32 atomics into slot 0 (long windows)
  int sub_pq, sub_hg;  // TMA box of a 64-row sub-tile: positions x heads
  long long n_both, n_lead, nitems;
  float sl2, scale;
  uint64_t wait_ns;    // limit of every bounded wait
  int stall;           // failure-path test: the MMA warp first waits on a barrier nothing arrives at
};

struct Item {
  int b, comp, nkb;   // nkb key blocks of one kind (0: nothing to do)
  int k0[2], n[2];    // key blocks [k0, k0 + n)
  int slot[2];        // partial slot of each block
  int tq_lo, tq_hi;   // query tiles [tq_lo, tq_hi), each over all head groups
};

// First query tile with a query that can see compressed entry e (the entry's
// window completes at query (e + 1) m - 1).
__device__ __forceinline__ int first_tile_comp(const QTiling &Q, int e) {
  const long long first = (long long)(e + 1) * Q.m - 1;
  return first >= Q.S ? Q.ntq : (int)(first / Q.Pq);
}

// Items, most work first: compressed pairs, lone even compressed blocks, raw.
//  - compressed pair c: blocks 2c and 2c+1 over the tiles from the first one
//    that sees block 2c+1 on, split kSplitBoth ways (slots kSplitLead + s);
//  - compressed lead c: block 2c over the tiles before that, split kSplitLead
//    ways (slots s);
//  - raw (b, j, pr): query positions [128 j, 128 j + 128) with raw blocks
//    j - 2 pr and j - 2 pr - 1 (the blocks that range can see, two at a time);
//    block kb's partial goes to slot j - kb.
__device__ __forceinline__ void item_of(const DkvParams &p, long long u, Item &it) {
  const QTiling &Q = p.qt;
  it.nkb = 0;
  it.tq_lo = it.tq_hi = 0;
  it.b = 0;
  it.comp = 0;
  if (u < p.n_both) {
    const long long per = (long long)Q.B * dkk::kSplitBoth;
    const int pc = (int)(u / per);
    const int rem = (int)(u % per);
    it.b = rem / dkk::kSplitBoth;
    const int split = rem % dkk::kSplitBoth;
    it.comp = 1;
    it.nkb = 2;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      it.k0[a] = (2 * pc + a) * kBlockKeys;
      it.n[a] = min(kBlockKeys, Q.Sc - it.k0[a]);
      it.slot[a] = dkk::kSplitLead + split;
    }
    const int lo = first_tile_comp(Q, it.k0[1]);
    const int len = Q.ntq - lo;
    it.tq_lo = lo + (int)((long long)len * split / dkk::kSplitBoth);
    it.tq_hi = lo + (int)((long long)len * (split + 1) / dkk::kSplitBoth);
  } else if (u < p.n_both + p.n_lead) {
    const long long v = u - p.n_both;
    const long long per = (long long)Q.B * dkk::kSplitLead;
    const int pc = (int)(v / per);
    const int rem = (int)(v % per);
    it.b = rem / dkk::kSplitLead;
    const int split = rem % dkk::kSplitLead;
    it.comp = 1;
    it.nkb = 1;
    it.k0[0] = 2 * pc * kBlockKeys;
    it.n[0] = min(kBlockKeys, Q.Sc - it.k0[0]);
    it.slot[0] = split;
    const int lo = first_tile_comp(Q, it.k0[0]);
    const int hi = 2 * pc + 1 < p.nkb_comp ? first_tile_comp(Q, it.k0[0] + kBlockKeys) : Q.ntq;
    const int len = hi - lo;
    it.tq_lo = lo + (int)((long long)len * split / dkk::kSplitLead);
    it.tq_hi = lo + (int)((long long)len * (split + 1) / dkk::kSplitLead);
  } else {
    const long long v = u - p.n_both - p.n_lead;
    const int pr = (int)(v % p.npr);
    const long long w = v / p.npr;
    it.b = (int)(w % Q.B);
    const int j = (int)(w / Q.B);
    const long long lo_key = (long long)j * kBlockKeys - Q.W + 1;  // oldest key the range can see
    const int kb_lo = lo_key <= 0 ? 0 : (int)(lo_key / kBlockKeys);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int kb = j - 2 * pr - a;
      if (kb < kb_lo || 2 * pr + a >= p.nslot) break;
      it.k0[a] = kb * kBlockKeys;
      it.n[a] = min(kBlockKeys, Q.S - it.k0[a]);
      it.slot[a] = 2 * pr + a;
      it.nkb = a + 1;
    }
    it.tq_lo = j * kBlockKeys / Q.Pq;
    it.tq_hi = (min(j * kBlockKeys + kBlockKeys, Q.S) + Q.Pq - 1) / Q.Pq;
  }
}

// P^T and (scale dS^T) of one key row for 32 query columns of a unit:
//   p = exp2(s * scale * log2e - lse * log2e),  ds = p * (scale dP - scale Delta)
// sv holds the 32 S^T values then the 32 matching dP^T values; rs4 points at
// the columns' (-lse*log2e) records, their (-scale*Delta) records 16 float4
// further.
// kMasked zeroes the columns whose bit in vis is clear.
template <bool kMasked>
__device__ __forceinline__ void ew_unit(const uint32_t (&sv)[64], const float4 *rs4, uint32_t vis, uint64_t sl2x2,
                                        uint64_t sc2, uint32_t (&pk)[16], uint32_t (&dk)[16]) {
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float4 nl = rs4[c / 4];
    const float4 dl = rs4[16 + c / 4];
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
      const float n0 = h ? nl.z : nl.x, n1 = h ? nl.w : nl.y;
      const float d0 = h ? dl.z : dl.x, d1 = h ? dl.w : dl.y;  // -scale * Delta
      float t0, t1;
      f32x2_split(ffma2(f32x2(sv[c + h], sv[c + h + 1]), sl2x2, f32x2(__float_as_uint(n0), __float_as_uint(n1))), t0,
                  t1);
      float e0 = ex2_approx(t0), e1 = ex2_approx(t1);
      // scale dP - scale Delta, then times p
      const uint64_t g2 =
          ffma2(f32x2(sv[32 + c + h], sv[32 + c + h + 1]), sc2, f32x2(__float_as_uint(d0), __float_as_uint(d1)));
      float g0, g1;
      f32x2_split(fmul2(f32x2(__float_as_uint(e0), __float_as_uint(e1)), g2), g0, g1);
      if (kMasked) {
        const bool v0 = (vis >> (c + h)) & 1u, v1 = (vis >> (c + h + 1)) & 1u;
        e0 = v0 ? e0 : 0.f;
        e1 = v1 ? e1 : 0.f;
        g0 = v0 ? g0 : 0.f;
        g1 = v1 ? g1 : 0.f;
      }
      pk[(c + h) >> 1] = pack_bf16x2(e0, e1);
      dk[(c + h) >> 1] = pack_bf16x2(g0, g1);
    }
  }
}

constexpr int kItemRing = 4;

struct DkvBars {
  uint64_t item_full[kItemRing], item_empty[kItemRing];  // dynamic item queue
  long long item[kItemRing];
  uint64_t k_full, k_empty;
  uint64_t st_full[dkk::kStages], st_empty[dkk::kStages];
  uint64_t s_full[2], p_full[2];  // per TMEM buffer
  uint64_t acc_full, acc_free;
  uint64_t drain, never;
  uint32_t tmem_base;
  int abort;
};

template <int kD>
__global__ void __launch_bounds__(dkk::kThreads, 1)
    hca_bwd_dkv_kernel(const __grid_constant__ CUtensorMap map_qs, const __grid_constant__ CUtensorMap map_dos,
                       const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_ckv,
                       const DkvParams p) {
  using namespace dkk;
  static_assert(kD == 64 || kD == 128, "head dim 64 or 128");
  constexpr int kHalves = kD / 64;   // 64-column (128-byte) halves of a row
  constexpr int kAccCols = kD / 2;   // accumulator columns per warpgroup in the item epilogue
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DkvBars bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int *abort_flag = &bars.abort;
  const QTiling &Q = p.qt;

  if (tid == 0) {
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&bars.item_full[i], 1);
      mbar_init(&bars.item_empty[i], 1 + kEW);
    }
    mbar_init(&bars.k_full, 1);
    mbar_init(&bars.k_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.st_full[s], 1);
      mbar_init(&bars.st_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.s_full[x], 1);
      mbar_init(&bars.p_full[x], kEW);  // both warpgroups write every unit
    }
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.acc_free, kEW);
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.never, 1);
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
  const int per_tile = Q.groups;  // query tiles per position tile (one per head group)
  // a sub-tile is a head range of its query tile when HG >= 2, a position range when one head fills it
  const bool pos_split = p.sub_hg == Q.HG;

  if (warp >= kEW / 32) {
    setmaxnreg_dec<kRegProducer>();
    if (warp == kEW / 32) {
      // ------------------------------------------------------------ TMA
      uint32_t gsub = 0, iw = 0;
      uint32_t issued = 0;  // bit s: stage loaded at least once; bit 8+s: parity of its last load
      int k_par = -1;
      bool ok = true;
      // Items are handed out dynamically (largest first) through a global
      // counter; this warp fetches them and publishes each to the other roles.
      for (uint32_t k = 0; ok; ++k) {
        const int slot = k % kItemRing;
        long long u = -1;
        if (lane == 0) {
          if (k >= (uint32_t)kItemRing)
            ok = mbar_wait(&bars.item_empty[slot], ((k / kItemRing) - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (ok) {
            u = atomicAdd(p.next_item, 1);
            if (u >= p.nitems) u = -1;
            bars.item[slot] = u;
            mbar_arrive(&bars.item_full[slot]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        u = __shfl_sync(0xffffffffu, u, 0);
        if (!ok || u < 0) break;
        if (poisoned) continue;
        Item it;
        item_of(p, u, it);
        const int nsub = 2 * (it.tq_hi - it.tq_lo) * per_tile;
        if (it.nkb == 0 || nsub <= 0) continue;
        if (lane == 0) {
          if (iw > 0) ok = mbar_wait(&bars.k_empty, (iw - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (ok) {
            const CUtensorMap *mp = it.comp ? &map_ckv : &map_kv;
            mbar_arrive_expect_tx(&bars.k_full, it.nkb * kHalves * kHalfTile);
            for (int a = 0; a < it.nkb; ++a) {
              uint8_t *dst = smem + kOffK + a * kTile;
#pragma unroll
              for (int hh = 0; hh < kHalves; ++hh) tma_load_3d(mp, &bars.k_full, dst + hh * kHalfTile, 64 * hh, it.k0[a], it.b);
            }
            k_par = iw & 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        for (int v = 0; ok && v < nsub; ++v, ++gsub) {
          const int x = v >> 1, sub = v & 1;
          const int tq = it.tq_lo + x / per_tile, g = x % per_tile;
          const int s = gsub % kStages;
          uint8_t *st = smem + kOffStage + s * kStageBytes;
          if (lane == 0 && gsub >= (uint32_t)kStages)
            ok = mbar_wait(&bars.st_empty[s], ((gsub / kStages) - 1) & 1, abort_flag, p.status, p.wait_ns);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          const int i0 = tq * Q.Pq;
          const int pos0 = pos_split ? i0 + sub * p.sub_pq : i0;
          const int hd = it.b * Q.H + g * Q.HG + (pos_split ? 0 : sub * p.sub_hg);
          // key intervals of the sub-tile's positions (both kinds)
          int4 *ivs = reinterpret_cast<int4 *>(st + kOffIv);
          for (int c = lane; c < p.sub_pq; c += 32) {
            const RowIv iv = row_interval(Q.sstart, it.b, Q.S, pos0 + c, Q.W, Q.m);
            ivs[c] = iv.valid ? make_int4(iv.rlo, iv.rhi, iv.clo, iv.chi) : make_int4(1, 0, 1, 0);
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars.st_full[s], kHalves * kHalfTile + 512);
#pragma unroll
            for (int h = 0; h < kHalves; ++h) {
              tma_load_3d(&map_qs, &bars.st_full[s], st + h * kHalfTile, 64 * h, pos0, hd);
              tma_load_3d(&map_dos, &bars.st_full[s], st + h * kHalfTile + kHalfRows * 128, 64 * h, pos0, hd);
            }
            // rows [64 sub, 64 sub + 64) of the tile's (-lse*log2e, Delta) record
            const long long tl = ((long long)it.b * Q.groups + g) * Q.ntq + tq;
            const float *rs = p.rowstat + tl * 2 * kRows + sub * kHalfRows;
#pragma unroll
            for (int h = 0; h < 2; ++h)
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                      smem_u32(st + kOffRowstat + h * 256)),
                  "l"(reinterpret_cast<uint64_t>(rs + h * kRows)), "r"(256), "r"(smem_u32(&bars.st_full[s]))
                  : "memory");
            issued = (issued | (1u << s)) & ~(1u << (8 + s));
            issued |= ((gsub / kStages) & 1u) << (8 + s);
          }
          __syncwarp();
        }
        ++iw;
      }
      if (!ok && !poisoned && lane == 0) {
        volatile int never = 0;
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) mbar_wait(&bars.st_full[s], (issued >> (8 + s)) & 1u, &never, p.status, 100000000ull);
        if (k_par >= 0) mbar_wait(&bars.k_full, k_par, &never, p.status, 100000000ull);
      }
    } else if (warp == kEW / 32 + 1) {
      // ------------------------------------------------------------ MMA
      // Whole warp on warp-uniform values; one elect.sync lane issues.  Work
      // unit u of an item is (sub-tile u / nkb, key block u % nkb); its
      // S^T | dP^T goes to TMEM buffer (global unit count) & 1, so the dS warps
      // form P^T, dS^T of one unit while the tensor pipe runs the next.
      const uint64_t dK0 = smem_desc_sw128(smem_u32(smem + kOffK), 16, 1024);
      const uint64_t dR0 = smem_desc_sw128(smem_u32(smem + kOffStage), 16, 1024);          // R, K-major
      const uint64_t dM0 = smem_desc_sw128(smem_u32(smem + kOffStage), kHalfTile, 1024);   // R rows, MN-major
      const uint32_t id_sd = idesc_bf16_f32(kRows, kRows, false, false);
      const uint32_t id_acc = idesc_bf16_f32(kRows, kD, false, true);
      uint32_t gsub = 0, gu = 0, iw = 0;  // sub-tiles, units and items with work so far
      bool ok = true, issued = false;
      if (p.stall && !poisoned) {
        injected_stall(&bars.never, abort_flag, p.status, p.wait_ns);
        ok = false;
      }
      for (uint32_t kq = 0; ok; ++kq) {
        const int slot = kq % kItemRing;
        long long u = -1;
        if (lane == 0) {
          ok = mbar_wait(&bars.item_full[slot], (kq / kItemRing) & 1, abort_flag, p.status, p.wait_ns);
          if (ok) {
            u = bars.item[slot];
            mbar_arrive(&bars.item_empty[slot]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        u = __shfl_sync(0xffffffffu, u, 0);
        if (!ok || u < 0) break;
        if (poisoned) continue;
        Item it;
        item_of(p, u, it);
        const int nsub = 2 * (it.tq_hi - it.tq_lo) * per_tile;
        if (it.nkb == 0 || nsub <= 0) continue;
        const int nkb = it.nkb;
        const int nu = nsub * nkb;
        ok = wait_warp(&bars.k_full, iw & 1, abort_flag, p.status, p.wait_ns);
        // S^T | dP^T of unit w into TMEM buffer (gu + w) & 1
        auto issue_sd = [&](int w) -> bool {
          const int v = nkb == 2 ? (w >> 1) : w, a = nkb == 2 ? (w & 1) : 0;
          const uint32_t sg = gsub + v;
          const int s = sg % kStages;
          if (a == 0 && !wait_warp(&bars.st_full[s], (sg / kStages) & 1, abort_flag, p.status, p.wait_ns)) return false;
          tc_fence_after();
          const uint64_t br = dR0 + desc_bytes(s * kStageBytes);
          const uint64_t bk = dK0 + desc_bytes(a * kTile);
          const uint32_t d = tmem + col_buf(gu + w);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < kD / 16; ++k) mma_ss(d, bk + kmaj_step(k), br + kmaj_step(k), id_sd, k > 0);
            mma_commit(&bars.s_full[(gu + w) & 1]);
            if (w == nu - 1) mma_commit(&bars.k_empty);  // the key tiles are read by these MMAs only
          }
          __syncwarp();
          issued = true;
          return true;
        };
        if (ok) ok = issue_sd(0);
        if (ok && nu > 1) ok = issue_sd(1);
        for (int w = 0; ok && w < nu; ++w) {
          const uint32_t g = gu + w;
          ok = wait_warp(&bars.p_full[g & 1], (g >> 1) & 1, abort_flag, p.status, p.wait_ns);
          if (ok && w == 0 && iw > 0) ok = wait_warp(&bars.acc_free, (iw - 1) & 1, abort_flag, p.status, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const int v = nkb == 2 ? (w >> 1) : w, a = nkb == 2 ? (w & 1) : 0;
          const int s = (gsub + v) % kStages;
          const uint64_t mq = dM0 + desc_bytes(s * kStageBytes), mdo = mq + desc_bytes(kHalfRows * 128);
          const uint32_t buf = tmem + col_buf(g), acc = tmem + col_acc(a);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kHalfRows / 16; ++kk) {
              // acc += P^T dO_sub  and  acc += (scale dS)^T Q_sub; query rows
              // [32 h, 32 h + 32) have P^T at columns 32 h .. 32 h + 15 and dS^T
              // at 32 h + 16 .. 32 h + 31 (8 packed columns per k-step)
              const uint32_t pc = (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8);
              mma_ts(acc, buf + pc, mdo + mnmaj_step(kk), id_acc, (v > 0 || kk > 0) ? 1u : 0u);
              mma_ts(acc, buf + pc + 16, mq + mnmaj_step(kk), id_acc, 1u);
            }
            if (a == nkb - 1) mma_commit(&bars.st_empty[s]);  // the sub-tile's last reader
            if (w == nu - 1) mma_commit(&bars.acc_full);
          }
          __syncwarp();
          if (w + 2 < nu) {
            ok = issue_sd(w + 2);
            if (!ok) break;
          }
        }
        gsub += nsub;
        gu += nu;
        ++iw;
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
    // ------------------------------------------------------------ P^T, dS^T + item epilogue
    // thread kr of warpgroup wg owns key row kr (TMEM lane kr), query columns
    // [32 wg, 32 wg + 32) of every unit and accumulator columns
    // [64 wg, 64 wg + 64) of the item epilogue
    const int kr = tid & (kRows - 1), wg = tid >> 7;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint64_t sl2x2 = f32x2(__float_as_uint(p.sl2), __float_as_uint(p.sl2));
    const uint64_t sc2 = f32x2(__float_as_uint(p.scale), __float_as_uint(p.scale));
    uint32_t gsub = 0, gu = 0, iw = 0;
    bool ok = true;
    for (uint32_t kq = 0; ok; ++kq) {
      const int slot = kq % kItemRing;
      if (!wait_warp(&bars.item_full[slot], (kq / kItemRing) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
      const long long u = *(volatile long long *)&bars.item[slot];
      mbar_arrive(&bars.item_empty[slot]);
      if (u < 0) break;
      Item it;
      item_of(p, u, it);
      const int nkb = it.nkb;
      if (nkb == 0) continue;
      const int nsub = 2 * (it.tq_hi - it.tq_lo) * per_tile;
      float *prow[2];
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const size_t rows = it.comp ? (size_t)p.Sc_pad : (size_t)p.S_pad;
        float *base = it.comp ? p.cpart : p.rpart;
        const int sl = (it.comp || !p.raw_atomic) ? it.slot[a] : 0;
        prow[a] = a < nkb ? base + (((size_t)sl * Q.B + it.b) * rows + it.k0[a] + kr) * kD + wg * kAccCols : nullptr;
      }
      const bool atomic_rows = !it.comp && p.raw_atomic;
      if (poisoned || nsub <= 0) {
        const float val = poisoned ? __int_as_float(0x7fc00000) : 0.f;
        for (int a = 0; a < nkb; ++a) {
          float4 *dst = reinterpret_cast<float4 *>(prow[a]);
          if (atomic_rows) {
            if (poisoned)
              for (int c = 0; c < kAccCols / 4; ++c) atomicAdd(dst + c, make_float4(val, val, val, val));
          } else {
#pragma unroll
            for (int c = 0; c < kAccCols / 4; ++c) dst[c] = make_float4(val, val, val, val);
          }
        }
        continue;
      }
      const int nu = nsub * nkb;
      // both warpgroups work on every unit, warpgroup h on query rows
      // [32 h, 32 h + 32) of its sub-tile: half the latency per unit, which
      // is what the tensor pipe waits on with two TMEM buffers in flight
      const int h = wg;
      for (int w = 0; w < nu; ++w) {
        const int v = nkb == 2 ? (w >> 1) : w, a = nkb == 2 ? (w & 1) : 0;
        const uint32_t g = gu + w;
        const uint32_t sg = gsub + v;
        const uint8_t *st = smem + kOffStage + (sg % kStages) * kStageBytes;
        if (!wait_warp(&bars.st_full[sg % kStages], (sg / kStages) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        if (!wait_warp(&bars.s_full[g & 1], (g >> 1) & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t base = lane_addr + col_buf(g);
        // query rows [32 h, 32 h + 32): S^T columns 32 h.., dP^T columns 64 + 32 h..
        uint32_t sv[64];
        tmem_ld32(base + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(base + 64 + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        // visibility of this key for the 64 columns (query rows) of the
        // sub-tile: column c sits at position c mod sub_pq of the sub-tile
        const int key = it.k0[a] + kr;
        uint64_t vis = 0;
        if (kr < it.n[a]) {
          const int4 *ivs = reinterpret_cast<const int4 *>(st + kOffIv);
          auto sees = [&](int q) -> bool {
            const int4 iv = ivs[q];
            const int lo = it.comp ? iv.z : iv.x, hi = it.comp ? iv.w : iv.y;
            return key >= lo && key <= hi;
          };
          if (p.sub_pq == 1) {  // one position: all 64 columns alike
            vis = sees(0) ? ~0ull : 0ull;
          } else if (p.sub_pq == 2) {  // two positions alternate over the columns
            vis = (sees(0) ? 0x5555555555555555ull : 0ull) | (sees(1) ? 0xAAAAAAAAAAAAAAAAull : 0ull);
          } else {
            uint64_t pat = 0;
            for (int q = 0; q < p.sub_pq; ++q)
              if (sees(q)) pat |= 1ull << q;
            for (int wd = p.sub_pq; wd < kHalfRows; wd *= 2) pat |= pat << wd;
            vis = pat;
          }
        }
        const uint32_t vis32 = (uint32_t)(vis >> (32 * h));
        // -lse*log2e [64] then -scale*Delta [64] of the sub-tile's rows
        const float4 *rs4 = reinterpret_cast<const float4 *>(st + kOffRowstat);
        uint32_t pk[16], dk[16];
        // warp-uniform cases: no visible pair (P^T = dS^T = 0), every pair
        // visible (no masking), or a mix
        const bool none = __all_sync(0xffffffffu, vis32 == 0u);
        const bool all = __all_sync(0xffffffffu, vis32 == ~0u);
        tmem_wait_ld();
        if (none) {
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = dk[c] = 0u;
        } else if (all) {
          ew_unit<false>(sv, rs4 + 8 * h, 0u, sl2x2, sc2, pk, dk);
        } else {
          ew_unit<true>(sv, rs4 + 8 * h, vis32, sl2x2, sc2, pk, dk);
        }
        // packed P^T and dS^T of query rows [32 h, 32 h + 32) go over S^T
        // columns 32 h .. 32 h + 31, which this thread has read
        tmem_st16(base + 32 * h, pk);
        tmem_st16(base + 32 * h + 16, dk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.p_full[g & 1]);
      }
      if (!ok) break;
      // ---------------- item epilogue: this key's accumulator rows
      if (!wait_warp(&bars.acc_full, iw & 1, abort_flag, p.status, p.wait_ns)) { ok = false; break; }
      tc_fence_after();
      for (int a = 0; a < nkb; ++a) {
        uint32_t o[kAccCols];
        const uint32_t ab = lane_addr + col_acc(a) + wg * kAccCols;
#pragma unroll
        for (int c0 = 0; c0 < kAccCols; c0 += 32) tmem_ld32(ab + c0, *reinterpret_cast<uint32_t(*)[32]>(o + c0));
        tmem_wait_ld();
        if (a == nkb - 1) {
          tc_fence_before();
          mbar_arrive(&bars.acc_free);  // the next item's accumulation may start
        }
        float4 *dst = reinterpret_cast<float4 *>(prow[a]);
        if (atomic_rows) {
#pragma unroll
          for (int x = 0; x < kAccCols / 4; ++x)
            atomicAdd(dst + x, make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]),
                                           __uint_as_float(o[4 * x + 2]), __uint_as_float(o[4 * x + 3])));
        } else {
#pragma unroll
          for (int x = 0; x < kAccCols / 4; ++x)
            dst[x] = make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]), __uint_as_float(o[4 * x + 2]),
                                 __uint_as_float(o[4 * x + 3]));
        }
      }
      gsub += nsub;
      gu += nu;
      ++iw;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// kernel 3: dkv and dckv = sums of their partial slots, in a fixed order
// ---------------------------------------------------------------------------
struct ReduceParams {
  const float *rpart, *cpart;
  __nv_bfloat16 *dkv, *dckv;
  int B, S, Sc, S_pad, Sc_pad, nslot, nrb, nkb_comp, raw_atomic;
  int with_comp;  // 0: dkv only (CSA writes dckv itself)
};

// Raw rows: one thread per four columns (a few slots each).  Compressed rows
// have up to kSlotsComp slots: kReduceLanes lanes per four columns, lane l
// summing slots s_lo + l, s_lo + l + kReduceLanes, ... in order, then a fixed
// butterfly over the lanes; both orders are fixed, so the sums are the same
// run to run.  The compressed index range starts at a multiple of 32 (the raw
// range is padded with idle threads), so no warp mixes the two and every
// shuffle has the whole warp.
constexpr int kReduceLanes = 8;

template <int kD>
__global__ void hca_bwd_reduce_kernel(const ReduceParams p) {
  const long long nraw4 = (long long)p.B * p.S * (kD / 4);
  const long long nraw_pad = (nraw4 + 31) & ~31LL;
  const long long ncomp = p.with_comp ? (long long)p.B * p.Sc * (kD / 4) * kReduceLanes : 0;
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nraw_pad + ncomp;
       v += (long long)gridDim.x * blockDim.x) {
    if (v >= nraw4 && v < nraw_pad) continue;  // padding of the raw range
    const bool comp = v >= nraw_pad;
    const int part = comp ? (int)((v - nraw_pad) % kReduceLanes) : 0;
    const long long x = comp ? (v - nraw_pad) / kReduceLanes : v;
    const int d4 = (int)(x % (kD / 4));
    const long long row = x / (kD / 4);
    const int rows = comp ? p.Sc : p.S;
    const int b = (int)(row / rows), key = (int)(row % rows);
    const int kb = key / kBlockKeys;
    int s_lo, s_hi, s_step;
    size_t stride, off;
    const float *base;
    if (comp) {
      // odd blocks only have pair slots; even blocks have lead slots and,
      // when their odd partner exists, pair slots
      s_lo = ((kb & 1) ? dkk::kSplitLead : 0) + part;
      s_hi = ((kb & 1) || kb + 1 < p.nkb_comp) ? dkk::kSlotsComp : dkk::kSplitLead;
      s_step = kReduceLanes;
      stride = (size_t)p.B * p.Sc_pad * kD;
      off = ((size_t)b * p.Sc_pad + key) * kD + d4 * 4;
      base = p.cpart;
    } else {
      // slot s holds query range kb + s; ranges past the sequence do not exist
      s_lo = 0;
      s_hi = p.raw_atomic ? 1 : min(p.nslot, p.nrb - kb);
      s_step = 1;
      stride = (size_t)p.B * p.S_pad * kD;
      off = ((size_t)b * p.S_pad + key) * kD + d4 * 4;
      base = p.rpart;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = s_lo; s < s_hi; s += s_step) {
      const float4 y = *reinterpret_cast<const float4 *>(base + s * stride + off);
      acc.x += y.x; acc.y += y.y; acc.z += y.z; acc.w += y.w;
    }
    if (comp) {
#pragma unroll
      for (int o = kReduceLanes / 2; o > 0; o >>= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
      }
      if (part != 0) continue;
    }
    uint2 o;
    o.x = pack_bf16x2(acc.x, acc.y);
    o.y = pack_bf16x2(acc.z, acc.w);
    __nv_bfloat16 *dst = comp ? p.dckv + ((size_t)b * p.Sc + key) * kD : p.dkv + ((size_t)b * p.S + key) * kD;
    *reinterpret_cast<uint2 *>(dst + d4 * 4) = o;
  }
}

size_t rowstat_bytes(const QTiling &q) { return align_up((size_t)q.ntiles * 2 * kRows * sizeof(float)); }

int sc_pad(int Sc) { return (Sc + kBlockKeys - 1) / kBlockKeys * kBlockKeys; }

// Raw key blocks: query range j (positions [128 j, 128 j + 128)) sees blocks
// j - nslot + 1 .. j, so a block collects nslot partial sums.  Windows longer
// than a few blocks accumulate into one fp32 buffer with atomics instead.
constexpr int kMaxRawSlots = 4;
struct RawGeom {
  int nrb, S_pad, nslot, npr, atomic;
};
RawGeom raw_geom(int S, int W) {
  RawGeom g;
  g.nrb = (S + kBlockKeys - 1) / kBlockKeys;
  g.S_pad = g.nrb * kBlockKeys;
  int ns = (int)(((long long)W + kBlockKeys - 2) / kBlockKeys) + 1;
  if (ns > g.nrb) ns = g.nrb;
  if (ns < 1) ns = 1;
  g.nslot = ns;
  g.npr = (ns + 1) / 2;
  g.atomic = ns > kMaxRawSlots;
  return g;
}
size_t rpart_bytes(int B, const RawGeom &g, int D) {
  return align_up((size_t)(g.atomic ? 1 : g.nslot) * B * g.S_pad * D * sizeof(float));
}
size_t cpart_bytes(int B, int Sc, int D) { return align_up((size_t)dkk::kSlotsComp * B * sc_pad(Sc) * D * sizeof(float)); }

}  // namespace

bool tc_bwd_supported(int H, int D, int dtype) { return tc_shape_ok(H, D, dtype); }

size_t tc_bwd_scratch_bytes(int B, int H, int S, int D, int W, int m, int dtype, bool csa) {
  if (!tc_shape_ok(H, D, dtype)) return 0;
  QTiling q = make_qtiling(nullptr, B, H, S, W, m);
  // CSA keeps no compressed partial slots: its dckv is accumulated query-major
  return rowstat_bytes(q) + (csa ? 0 : cpart_bytes(B, q.Sc, D)) + rpart_bytes(B, raw_geom(S, W), D);
}

cudaError_t tc_bwd(const BwdArgs &a, cudaStream_t st, const CsaBwd *csa) {
  const QTiling q = make_qtiling(a.sstart, a.B, a.H, a.S, a.W, a.m);
  const int Spad = sc_pad(q.Sc);
  const RawGeom rg = raw_geom(a.S, a.W);
  char *ws = static_cast<char *>(a.scratch);
  float *rowstat = reinterpret_cast<float *>(ws);
  float *cpart = csa ? nullptr : reinterpret_cast<float *>(ws + rowstat_bytes(q));
  float *rpart = reinterpret_cast<float *>(ws + rowstat_bytes(q) + (csa ? 0 : cpart_bytes(a.B, q.Sc, a.D)));
  // dkv kernel: a 64-row half of a query tile is a head range when HG >= 2,
  // a position range when one head fills the tile
  const int sub_hg = q.HG >= 2 ? q.HG / 2 : 1;
  const int sub_pq = q.HG >= 2 ? q.Pq : q.Pq / 2;
  CUtensorMap mq, mdo, mout, mkv, mckv, mkv16, mckv16, mdq, mqs, mdos, mckvg;
  const uint64_t D = (uint64_t)a.D;
  if (!make_map_bf16(&mq, a.q, D, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mout, a.out, D, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mdo, a.dout, D, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mdq, a.dq, D, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mqs, a.q, D, a.S, (uint64_t)a.B * a.H, sub_pq, sub_hg) ||
      !make_map_bf16(&mdos, a.dout, D, a.S, (uint64_t)a.B * a.H, sub_pq, sub_hg) ||
      !make_map_bf16(&mkv, a.kv, D, a.S, a.B, kBlockKeys, 1) ||
      !make_map_bf16(&mckv, a.ckv, D, q.Sc, a.B, kBlockKeys, 1) ||
      !make_map_bf16(&mkv16, a.kv, D, a.S, a.B, 16, 1) ||
      !make_map_bf16(&mckv16, a.ckv, D, q.Sc, a.B, 16, 1))
    return cudaErrorInvalidValue;
  if (csa && a.D != 128) return cudaErrorInvalidValue;
  // CSA: the dq kernel gathers its compressed rows through the row view of ckv
  if (csa && !make_map_rows_bf16(&mckvg, a.ckv, D, (uint64_t)q.Sc * a.B)) return cudaErrorInvalidValue;
  const bool d64 = a.D == 64;
  auto dq_kern = csa ? hca_bwd_dq_kernel<true, 128> : (d64 ? hca_bwd_dq_kernel<false, 64> : hca_bwd_dq_kernel<false, 128>);
  auto dkv_kern = d64 ? hca_bwd_dkv_kernel<64> : hca_bwd_dkv_kernel<128>;
  auto reduce_kern = d64 ? hca_bwd_reduce_kernel<64> : hca_bwd_reduce_kernel<128>;
  static SmemAttrOnce attr_dq[3], attr_dkv[2];
  {
    cudaError_t e = attr_dq[csa ? 2 : (d64 ? 1 : 0)].ensure(reinterpret_cast<const void *>(dq_kern), dqk::kSmemBytes);
    if (e == cudaSuccess) e = attr_dkv[d64 ? 1 : 0].ensure(reinterpret_cast<const void *>(dkv_kern), dkk::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const float sl2 = a.scale * kLog2e;

  DqParams dp;
  dp.qt = q;
  dp.u_cnt = csa ? csa->u.cnt : nullptr;
  dp.u_ent = csa ? csa->u.ent : nullptr;
  dp.u_mask = csa ? csa->u.mask : nullptr;
  dp.u_cap = csa ? csa->u.cap : 0;
  dp.ckv = static_cast<const __nv_bfloat16 *>(a.ckv);
  dp.status = a.status_rw;
  dp.lse = a.lse;
  dp.rowstat = rowstat;
  dp.dq = static_cast<__nv_bfloat16 *>(a.dq);
  dp.sl2 = sl2;
  dp.scale = a.scale;
  dp.wait_ns = a.wait_ns;
  dp.stall = (a.stall & HCA_STALL_DQ) != 0;
  dp.pq_shift = 0;
  while ((1 << dp.pq_shift) < q.Pq) ++dp.pq_shift;
  const long long g1 = q.ntiles < sms ? q.ntiles : sms;
  if (g1 == 0) return cudaSuccess;
  cudaError_t e;
  {
    ProfScope prof(kKBwdDq, st);
    dq_kern<<<(unsigned)g1, dqk::kThreads, dqk::kSmemBytes, st>>>(mq, mdo, mout, mkv, csa ? mckvg : mckv, mkv16, mckv16, mdq, dp);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;

  DkvParams kp;
  kp.qt = q;
  kp.status = a.status_rw;
  kp.next_item = a.status_rw + 16;  // in the workspace header (64 bytes past the status word)
  kp.rowstat = rowstat;
  kp.rpart = rpart;
  kp.cpart = cpart;
  kp.nrb = rg.nrb;
  kp.nkb_comp = (q.Sc + kBlockKeys - 1) / kBlockKeys;
  kp.S_pad = rg.S_pad;
  kp.Sc_pad = Spad;
  kp.nslot = rg.nslot;
  kp.npr = rg.npr;
  kp.raw_atomic = rg.atomic;
  kp.sub_pq = sub_pq;
  kp.sub_hg = sub_hg;
  // CSA: raw items only (its compressed entries are handled query-major)
  kp.n_both = csa ? 0 : (long long)a.B * (kp.nkb_comp / 2) * dkk::kSplitBoth;
  kp.n_lead = csa ? 0 : (long long)a.B * ((kp.nkb_comp + 1) / 2) * dkk::kSplitLead;
  kp.nitems = kp.n_both + kp.n_lead + (long long)a.B * rg.nrb * rg.npr;
  kp.sl2 = sl2;
  kp.scale = a.scale;
  kp.wait_ns = a.wait_ns;
  kp.stall = (a.stall & HCA_STALL_DKV) != 0;
  const long long g2 = kp.nitems < sms ? kp.nitems : sms;
  e = cudaMemsetAsync(kp.next_item, 0, sizeof(int32_t), st);
  if (e == cudaSuccess && rg.atomic) e = cudaMemsetAsync(rpart, 0, rpart_bytes(a.B, rg, a.D), st);
  if (e != cudaSuccess) return e;
  {
    ProfScope prof(kKBwdDkv, st);
    dkv_kern<<<(unsigned)g2, dkk::kThreads, dkk::kSmemBytes, st>>>(mqs, mdos, mkv, mckv, kp);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;

  ReduceParams rp;
  rp.rpart = rpart;
  rp.cpart = cpart;
  rp.dkv = static_cast<__nv_bfloat16 *>(a.dkv);
  rp.dckv = static_cast<__nv_bfloat16 *>(a.dckv);
  rp.B = a.B;
  rp.S = a.S;
  rp.Sc = q.Sc;
  rp.S_pad = rg.S_pad;
  rp.Sc_pad = Spad;
  rp.nslot = rg.nslot;
  rp.nrb = rg.nrb;
  rp.nkb_comp = kp.nkb_comp;
  rp.raw_atomic = rg.atomic;
  rp.with_comp = csa ? 0 : 1;
  const long long n4 = (((long long)a.B * a.S * (a.D / 4) + 31) & ~31LL) +
                       (csa ? 0 : (long long)a.B * q.Sc * (a.D / 4) * kReduceLanes);
  if (n4 > 0) {
    int blocks = (int)((n4 + 255) / 256);
    if (blocks > 8 * sms) blocks = 8 * sms;
    ProfScope prof(kKBwdReduce, st);
    reduce_kern<<<blocks, 256, 0, st>>>(rp);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || !csa) return e;
  return csa_dckv(a, csa->u, rowstat, csa->acc, st);
}

}  // namespace hca
