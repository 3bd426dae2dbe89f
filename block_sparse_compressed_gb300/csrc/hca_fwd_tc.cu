// hca_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) HCA forward for sm_103a.
//
// Operation ("Add HCA Static Compilation for Splash Attention [Deepseek v4]",
// Description: sliding window + completed compression windows, MQA dispatch
// with the single kv head; "[DeepSeek-V4] Implement Compressed Attention
// Layers", einsum review suggestions: k = v = kv broadcast over heads).
//
// Tiling.  All heads of a query position share every key row (one kv head),
// so a tile packs Pq consecutive positions x HG heads into the M = 128 rows
// of the MMA (row r = head*Pq + p), loaded by one 3-D TMA box {64, Pq, HG}
// per 64-column half of q.  For every tile the key ranges of the union of its
// rows' intervals (hca_common.cuh) are cut into blocks of <= 128 keys: raw kv
// blocks first, then compressed ckv blocks.  Keys outside those ranges are
// never loaded and no mask exists in memory; inside a block each row masks by
// its own interval.
//
// Per key block: S = Q K^T (tcgen05, fp32 in TMEM) -> softmax warps load S,
// mask, online softmax in fp32 with exp2 (the running max is only raised when
// a block's max exceeds it by more than 2^8, so O in TMEM is rarely rescaled)
// -> P (bf16) in shared memory -> O += P V with V = the same shared-memory
// kv tile read through an MN-major descriptor (K = V: one load serves both).
// Epilogue: out = O / l through a 128B-swizzled staging tile and a TMA store;
// lse = ln-domain logsumexp.
//
// Warp roles (192 threads, persistent CTAs):
//   warps 0-3  softmax + epilogue, thread r owns row r (TMEM lane r)
//   warp 4     TMA producer (Q once per tile, kv/ckv blocks into a 3-stage ring)
//   warp 5     MMA issuer (one elected lane)
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

constexpr int kStages = 3;          // kv ring depth
constexpr int kSoftmaxThreads = 128;
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;      // S: cols [0,128), O: cols [128,256)
constexpr uint32_t kColS = 0, kColO = 128;
constexpr float kRescaleLog2 = 8.0f;

// dynamic shared memory: Q | kv ring | P x2 | out staging  (+1 KB alignment)
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kTile;
constexpr int kOffP = kOffKV + kStages * kTile;
constexpr int kOffOut = kOffP + 2 * kTile;
constexpr int kSmemBytes = kOffOut + kTile + 1024;

struct FwdParams {
  QTiling qt;
  int32_t *status;
  float *lse;
  __nv_bfloat16 *out;  // direct stores for poisoned calls / tiles without keys
  float sl2;           // scale * log2(e)
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full, s_free;
  uint64_t p_full[2], o_done[2];
  uint64_t epi;  // softmax-warp rendezvous before the output store
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
    hca_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                      const __grid_constant__ CUtensorMap map_ckv, const __grid_constant__ CUtensorMap map_out,
                      const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int *abort_flag = &bars.abort;

  if (tid == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, kSoftmaxThreads);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars.p_full[k], kSoftmaxThreads);
      mbar_init(&bars.o_done[k], 1);
    }
    mbar_init(&bars.epi, kSoftmaxThreads);
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

  if (warp == 4) {
    // ------------------------------------------------------------ TMA
    if (!poisoned && lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_kv);
      tma_prefetch_map(&map_ckv);
    }
    uint32_t gb = 0, tiles_with_work = 0;
    int last_par[kStages] = {-1, -1, -1};
    int q_par = -1;
    bool ok = !poisoned;
    for (long long u = blockIdx.x; ok && u < p.qt.ntiles; u += gridDim.x) {
      Tile t;
      tile_coords(p.qt, u, t);
      tile_ranges_warp(p.qt, t, lane);
      const int nb = t.nraw + t.ncomp;
      if (nb == 0) continue;
      if (lane == 0) {
        if (tiles_with_work > 0) ok = mbar_wait(&bars.q_empty, (tiles_with_work - 1) & 1, abort_flag, p.status);
        if (ok) {
          mbar_arrive_expect_tx(&bars.q_full, kTile);
          const int c2 = t.b * p.qt.H + t.g * p.qt.HG;
          tma_load_3d(&map_q, &bars.q_full, smem + kOffQ, 0, t.i0, c2);
          tma_load_3d(&map_q, &bars.q_full, smem + kOffQ + kHalfTile, 64, t.i0, c2);
          q_par = tiles_with_work & 1;
        }
        for (int j = 0; ok && j < nb; ++j, ++gb) {
          const int s = gb % kStages;
          if (gb >= (uint32_t)kStages) ok = mbar_wait(&bars.kv_empty[s], ((gb / kStages) - 1) & 1, abort_flag, p.status);
          if (!ok) break;
          bool comp;
          int start, n;
          block_of(t, j, comp, start, n);
          const CUtensorMap *mp = comp ? &map_ckv : &map_kv;
          uint8_t *dst = smem + kOffKV + s * kTile;
          mbar_arrive_expect_tx(&bars.kv_full[s], kTile);
          tma_load_3d(mp, &bars.kv_full[s], dst, 0, start, t.b);
          tma_load_3d(mp, &bars.kv_full[s], dst + kHalfTile, 64, start, t.b);
          last_par[s] = (gb / kStages) & 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      gb = __shfl_sync(0xffffffffu, gb, 0);
      ++tiles_with_work;
    }
    if (!ok && !poisoned && lane == 0) {
      // drain own copies before leaving (bounded, ignores the abort flag)
      volatile int never = 0;
      for (int s = 0; s < kStages; ++s)
        if (last_par[s] >= 0) mbar_wait(&bars.kv_full[s], last_par[s], &never, p.status, 100000000ull);
      if (q_par >= 0) mbar_wait(&bars.q_full, q_par, &never, p.status, 100000000ull);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA
    const uint32_t qa = smem_u32(smem + kOffQ);
    const uint32_t pa0 = smem_u32(smem + kOffP);
    uint32_t gb = 0, tiles_with_work = 0;
    bool ok = !poisoned;
    bool issued = false;
    for (long long u = blockIdx.x; ok && u < p.qt.ntiles; u += gridDim.x) {
      Tile t;
      tile_coords(p.qt, u, t);
      tile_ranges_warp(p.qt, t, lane);
      const int nb = t.nraw + t.ncomp;
      if (nb == 0) continue;
      if (lane == 0) {
        ok = mbar_wait(&bars.q_full, tiles_with_work & 1, abort_flag, p.status);
        // S(j) for the first block, then S(j+1) ahead of PV(j)
        auto issue_s = [&](int j, uint32_t g) -> bool {
          const int s = g % kStages;
          if (!mbar_wait(&bars.kv_full[s], (g / kStages) & 1, abort_flag, p.status)) return false;
          if (g > 0 && !mbar_wait(&bars.s_free, (g - 1) & 1, abort_flag, p.status)) return false;
          tc_fence_after();
          bool comp;
          int start, n;
          block_of(t, j, comp, start, n);
          const int nk = (n + 15) & ~15;
          const uint32_t idesc = idesc_bf16_f32(kRows, nk, false, false);
          const uint32_t ka = smem_u32(smem + kOffKV + s * kTile);
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t off = (k >> 2) * kHalfTile + (k & 3) * 32;
            mma_ss(tmem + kColS, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024), idesc,
                   k > 0);
          }
          mma_commit(&bars.s_full);
          issued = true;
          return true;
        };
        if (ok) ok = issue_s(0, gb);
        if (ok && nb == 1) mma_commit(&bars.q_empty);
        for (int j = 0; ok && j < nb; ++j) {
          const uint32_t g = gb + j;
          if (j + 1 < nb) {
            ok = issue_s(j + 1, g + 1);
            if (!ok) break;
            if (j + 1 == nb - 1) mma_commit(&bars.q_empty);
          }
          const int pb = g & 1;
          ok = mbar_wait(&bars.p_full[pb], (g >> 1) & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          bool comp;
          int start, n;
          block_of(t, j, comp, start, n);
          const int nk = (n + 15) & ~15;
          const int s = g % kStages;
          const uint32_t va = smem_u32(smem + kOffKV + s * kTile);
          const uint32_t pa = pa0 + pb * kTile;
          const uint32_t idesc = idesc_bf16_f32(kRows, kHeadDim, false, true);
          for (int kk = 0; kk < nk / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * kHalfTile + (kk & 3) * 32;
            mma_ss(tmem + kColO, smem_desc_sw128(pa + aoff, 16, 1024),
                   smem_desc_sw128(va + kk * 2048, kHalfTile, 1024), idesc, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars.kv_empty[s]);
          mma_commit(&bars.o_done[pb]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      gb += nb;
      ++tiles_with_work;
    }
    if (!ok && issued && lane == 0) {
      volatile int never = 0;
      mma_commit(&bars.drain);
      mbar_wait(&bars.drain, 0, &never, p.status, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = tid;  // row == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    uint8_t *pbuf = smem + kOffP;
    uint8_t *obuf = smem + kOffOut;
    uint32_t gb = 0;
    uint32_t done_cnt[2] = {0, 0};
    bool ok = true;
    bool store_pending = false;
    uint32_t epi_phase = 0;
    // all 128 softmax threads meet here (bounded; never a bar.sync, so a
    // CTA that aborted cannot strand a thread)
    auto rendezvous = [&]() -> bool {
      mbar_arrive(&bars.epi);
      const bool r = wait_warp(&bars.epi, epi_phase & 1, abort_flag, p.status);
      ++epi_phase;
      return r;
    };
    // wait until PV number x (global) has completed
    auto wait_pv = [&](uint32_t x) -> bool {
      const int buf = x & 1;
      const uint32_t need = (x >> 1) + 1;
      while (done_cnt[buf] < need) {
        if (!wait_warp(&bars.o_done[buf], done_cnt[buf] & 1, abort_flag, p.status)) return false;
        ++done_cnt[buf];
      }
      return true;
    };
    for (long long u = blockIdx.x; ok && u < p.qt.ntiles; u += gridDim.x) {
      Tile t;
      tile_coords(p.qt, u, t);
      tile_ranges_warp(p.qt, t, lane);
      const int nb = t.nraw + t.ncomp;
      const int pq = r % p.qt.Pq, hh = r / p.qt.Pq;
      const int head = t.g * p.qt.HG + hh;
      const int i = t.i0 + pq;
      const RowIv iv = row_interval(p.qt.sstart, t.b, p.qt.S, i, p.qt.W, p.qt.m);
      const size_t lrow = ((size_t)t.b * p.qt.H + head) * p.qt.S + i;
      if (poisoned || nb == 0) {
        // whole tile without keys (padding) or poisoned call: direct stores
        if (i < p.qt.S) {
          const float v = poisoned ? __int_as_float(0x7fc00000) : 0.f;
          const uint32_t w2 = pack_bf16x2(v, v);
          uint4 *orow = reinterpret_cast<uint4 *>(p.out + lrow * kHeadDim);
#pragma unroll
          for (int c = 0; c < kHeadDim / 8; ++c) orow[c] = make_uint4(w2, w2, w2, w2);
          p.lse[lrow] = poisoned ? v : -INFINITY;
        }
        continue;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nb; ++j, ++gb) {
        bool comp;
        int start, n;
        block_of(t, j, comp, start, n);
        const int nk = (n + 15) & ~15;
        // visible columns of this row inside the block
        int lo_c = 0, hi_c = -1;
        if (iv.valid) {
          const int lo = comp ? iv.clo : iv.rlo, hi = comp ? iv.chi : iv.rhi;
          lo_c = max(lo - start, 0);
          hi_c = min(hi - start, n - 1);
        }
        if (!wait_warp(&bars.s_full, gb & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        float s[kBlockKeys];
        {
          uint32_t rr[32];
#pragma unroll
          for (int c0 = 0; c0 < kBlockKeys; c0 += 32) {
            if (c0 < nk) {
              if (c0 + 32 <= nk) {
                tmem_ld32(lane_addr + kColS + c0, rr);
              } else {
                uint32_t r16[16];
                tmem_ld16(lane_addr + kColS + c0, r16);
#pragma unroll
                for (int x = 0; x < 16; ++x) rr[x] = r16[x];
              }
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) s[c0 + x] = __uint_as_float(rr[x]);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&bars.s_free);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBlockKeys; ++c) {
          const float v = (c >= lo_c && c <= hi_c) ? s[c] * p.sl2 : -INFINITY;
          s[c] = v;
          mx = fmaxf(mx, v);
        }
        // raise the running max only when this block exceeds it by > 2^8
        float f = 1.f;
        bool rescale_o = false;
        if (mx > m_run + kRescaleLog2 || (m_run == -INFINITY && mx > -INFINITY)) {
          if (m_run > -INFINITY) {
            f = ex2_approx(m_run - mx);
            l_run *= f;
            rescale_o = j > 0;  // O holds PV(0..j-1) of this tile
          }
          m_run = mx;
        }
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < kBlockKeys; ++c) {
          const float e = ex2_approx(s[c] - m_use);
          s[c] = e;
          rs += e;
        }
        l_run += rs;
        // P buffer gb&1 was last read by PV(gb-2)
        if (gb >= 2 && !wait_pv(gb - 2)) { ok = false; break; }
        uint8_t *pb = pbuf + (gb & 1) * kTile;
#pragma unroll
        for (int ch = 0; ch < kBlockKeys / 8; ++ch) {
          if (ch * 8 < nk) {
            uint4 v;
            v.x = pack_bf16x2(s[ch * 8 + 0], s[ch * 8 + 1]);
            v.y = pack_bf16x2(s[ch * 8 + 2], s[ch * 8 + 3]);
            v.z = pack_bf16x2(s[ch * 8 + 4], s[ch * 8 + 5]);
            v.w = pack_bf16x2(s[ch * 8 + 6], s[ch * 8 + 7]);
            *reinterpret_cast<uint4 *>(pb + sw128_offset(r, ch)) = v;
          }
        }
        // the TMEM access below is warp-collective: rescale when any row of the
        // warp needs it (rows without a new max use f = 1)
        if (__any_sync(0xffffffffu, rescale_o)) {
          // PV(j) waits for this block's P, so O is stable once PV(j-1) is done
          if (!wait_pv(gb - 1)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[32];
#pragma unroll
          for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
            tmem_ld32(lane_addr + kColO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
            tmem_st32(lane_addr + kColO + c0, o);
          }
          tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&bars.p_full[gb & 1]);
      }
      if (!ok) break;
      // ---------------- epilogue
      if (!wait_pv(gb - 1)) { ok = false; break; }
      tc_fence_after();
      if (store_pending) {
        // the previous tile's TMA store must have read the staging tile
        if (tid == 0) bulk_wait_read0();
        if (!rendezvous()) { ok = false; break; }
        store_pending = false;
      }
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      {
        uint32_t o[32];
#pragma unroll
        for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
          tmem_ld32(lane_addr + kColO + c0, o);
          tmem_wait_ld();
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
      }
      if (i < p.qt.S) {
        float lv;
        if (l_run > 0.f) {
          float lg;
          asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l_run));
          lv = (m_run + lg) * 0.69314718055994531f;
        } else {
          lv = -INFINITY;
        }
        p.lse[lrow] = lv;
      }
      fence_async_smem();
      tc_fence_before();
      if (!rendezvous()) { ok = false; break; }
      if (tid == 0) {
        const int c2 = t.b * p.qt.H + t.g * p.qt.HG;
        tma_store_3d(&map_out, obuf, 0, t.i0, c2);
        tma_store_3d(&map_out, obuf + kHalfTile, 64, t.i0, c2);
        bulk_commit();
      }
      store_pending = true;
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

}  // namespace

bool tc_fwd_supported(int H, int D, int dtype) { return tc_shape_ok(H, D, dtype); }

int tc_query_tile_positions(int H) { return kRows / heads_per_tile(H); }

cudaError_t tc_fwd(const FwdArgs &a, cudaStream_t st) {
  FwdParams p;
  p.qt = make_qtiling(a.sstart, a.B, a.H, a.S, a.W, a.m);
  const QTiling &q = p.qt;
  CUtensorMap mq, mkv, mckv, mout;
  if (!make_map_bf16(&mq, a.q, kHeadDim, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mout, a.out, kHeadDim, a.S, (uint64_t)a.B * a.H, q.Pq, q.HG) ||
      !make_map_bf16(&mkv, a.kv, kHeadDim, a.S, a.B, kBlockKeys, 1) ||
      !make_map_bf16(&mckv, a.ckv, kHeadDim, q.Sc, a.B, kBlockKeys, 1))
    return cudaErrorInvalidValue;
  p.status = a.status_rw;
  p.lse = a.lse;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.sl2 = a.scale * 1.4426950408889634f;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(hca_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const long long grid = q.ntiles < sms ? q.ntiles : sms;
  if (grid == 0) return cudaSuccess;
  ProfScope prof(kKFwdTc, st);
  hca_fwd_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(mq, mkv, mckv, mout, p);
  return cudaGetLastError();
}

}  // namespace hca
