// Split-KV flash-decoding body over the ragged page pool (shared by the decode
// kernel and the fused sparse-layer kernel).  See decode_attn.cu for the design.
#pragma once

#include "ptx.cuh"
#include "tg_internal.h"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

namespace {

using namespace tgk;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // give up a copy wait after 2 s
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct DecodeArgs {
  const tg_work_item *items;
  const tg_work_item *lead;  // [N_CTA]: each CTA's first item; reserved[0] its item count, [1] its index
  const int32_t *cta_off;
  const uint16_t *q;
  uint16_t *out;
  float *lse;
  const int64_t *pt_off;
  const int32_t *pt_ids;
  int64_t pool_pages;
  int32_t *counters;
  float *ws_ml;
  float *ws_o;
  int32_t *status;
  int64_t *cta_time;
  int H, H_q, g, G, H_p, P;
  float scale_log2;
  int wait_tables;  // wait for the previous kernel before reading q, pt_off, pt_ids
  const int32_t *row_ready;  // [batch*H]: wait until the rows of this CTA's items hold `epoch` (or NULL)
  const uint8_t *row_due;    // [batch*H]: only rows marked 1 are waited for (NULL: every row)
  uint64_t wait_ns;          // limit of each row-ready wait
  int epoch;
};

// wait (bounded) until *flag == epoch; false after the time limit
__device__ __forceinline__ bool wait_flag(const int32_t *flag, int epoch, uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (;;) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == epoch) return true;
    const uint64_t t = globaltimer_ns();
    if (!t0) t0 = t;
    else if (t - t0 > limit_ns) return false;
    __nanosleep(128);
  }
}

template <int D>
struct KCfg;
// NW streaming warps (each with an R-stage copy ring) and NE epilogue warps
template <>
struct KCfg<128> {
  // seven streaming warps (112 KB of copies in flight per SM): the SMs' bandwidth shares
  // spread less than with eight (worst-layer CTA skew 1.12-1.13 against 1.14-1.17 at config 2,
  // 1.27-1.28 against 1.31-1.34 at config 3, same box), at 1.6% of back-to-back time at config 2
  static constexpr int NW = 7, R = 2, NE = 4;
};
template <>
struct KCfg<256> {
  static constexpr int NW = 4, R = 2, NE = 4;
};

constexpr int kMaxItems = 16;  // work items per CTA kept in shared memory (more are read from global)
constexpr int kFacMax = 2048;  // merge factors (parts x heads) the epilogue keeps in shared memory

template <int D>
struct Layout {
  static constexpr int NW = KCfg<D>::NW, R = KCfg<D>::R, NE = KCfg<D>::NE;
  static constexpr int THREADS = (NW + NE) * 32;
  static constexpr int TILE = 16 * D * 2;  // bytes of 16 rows of K (or V)
  static constexpr int STAGE = 2 * TILE;   // K tile then V tile
  static constexpr int RING = NW * R * STAGE;
  // small region at the start of dynamic shared memory (16-byte aligned base): copy mbarriers,
  // hand-off mbarriers (full[2], empty[2]), the CTA's start time, item copies and their
  // page-table bases, the hand-off (m, l) of every streaming warp in both buffers, the merged
  // (M, L) per head, flags
  static constexpr int SMALL = NW * R * 8 + 4 * 8 + 8 + kMaxItems * (8 + (int)sizeof(tg_work_item)) +
                               kMaxItems * 4 + 2 * NW * 8 * 4 * 2 + 8 * 4 * 2 + 16;
  // floats per (warp, head) row of a hand-off buffer: padded against bank conflicts when it fits
  __host__ __device__ static int ostride(int g) { return g <= 4 ? D + 4 : D; }
  __host__ __device__ static int comb_floats(int g) { return NW * g * ostride(g); }
  static int smem_bytes(int g) { return SMALL + 1008 + RING + 2 * comb_floats(g) * 4 + kFacMax * 4; }
};

// byte offset of element (row, col) of a TMA tile loaded as D/64 boxes of
// [16 rows][64 cols] bf16 with the 128-byte swizzle (16-byte chunk ^= row % 8)
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)((col >> 6) * 2048 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void item_tiles(const tg_work_item &it, int &k_lo, int &k_hi) {
  if (it.t1 > it.t0) {
    k_lo = it.t0 >> 4;
    k_hi = (it.t1 + 15) >> 4;
  } else {
    k_lo = k_hi = 0;
  }
}

// barrier of the epilogue warps only (named barrier 1)
template <int N>
__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// The decode of one CTA (blockIdx.x = its place in the plan); smem_raw: Layout<D>::smem_bytes
// of dynamic shared memory, 16-byte aligned; Layout<D>::THREADS threads.  The kernel below and
// the fused sparse-layer kernel both run it.
//
// Roles.  Warps 0..NW-1 stream: 16-token tiles of an item go round-robin to them, each warp
// keeps R tiles in flight and refills a stage as soon as it has read it, across item
// boundaries.  At the end of an item a streaming warp leaves its (m, l, O) in one of two
// hand-off buffers (item k uses buffer k & 1) and goes straight on.  Warps NW.. are the
// epilogue: per item they combine the streaming warps' states, write the output (a run this
// CTA owns) or a partial (a shared run), count the partial and, in the last CTA of the run,
// merge every partial.  So no streaming warp waits at an item boundary for the slowest one,
// nor for the combine, the count or a merge.  Items of shared runs are processed first, so
// their merges overlap the streaming of the runs this CTA owns and the CTA ends on a cheap
// epilogue.  Which warp reads a tile, and every summation order, is as in one-role decoding:
// the results do not depend on the processing order.
template <int D>
__device__ __forceinline__ void decode_body(const CUtensorMap *pool_map_p, const DecodeArgs &a, uint8_t *smem_raw) {
  const CUtensorMap &pool_map = *pool_map_p;
  using LY = Layout<D>;
  constexpr int NW = LY::NW, R = LY::R, NE = LY::NE, NT = LY::THREADS, KS = D / 16;
  constexpr int NS = NW * 32, NET = NE * 32;  // streaming and epilogue threads
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);                 // [NW][R] copy stages
  uint64_t *full = bars + NW * R;                                          // [2] hand-off buffer written
  uint64_t *empty = full + 2;                                              // [2] hand-off buffer read
  uint64_t *s_t0 = empty + 2;                                              // CTA start (globaltimer)
  int64_t *s_base = reinterpret_cast<int64_t *>(s_t0 + 1);                 // [kMaxItems]
  tg_work_item *s_items = reinterpret_cast<tg_work_item *>(s_base + kMaxItems);  // [kMaxItems]
  int *s_order = reinterpret_cast<int *>(s_items + kMaxItems);             // [kMaxItems] processing order
  float *comb_m = reinterpret_cast<float *>(s_order + kMaxItems);          // [2][NW][8]
  float *comb_l = comb_m + 2 * NW * 8;                                     // [2][NW][8]
  float *s_mm = comb_l + 2 * NW * 8;                                       // [8] merged M per head
  float *s_ll = s_mm + 8;                                                  // [8] merged L per head
  int *flag = reinterpret_cast<int *>(s_ll + 8);                           // last CTA of a shared run
  volatile int *s_dead = flag + 1;                                         // a hand-off wait gave up
  uint8_t *ring = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + LY::SMALL + 1023) & ~uintptr_t(1023));  // [NW][R][STAGE]
  const int ostride = LY::ostride(a.g);
  const int cfl = LY::comb_floats(a.g);
  float *comb_o = reinterpret_cast<float *>(ring + LY::RING);              // [2][NW][g][ostride]
  float *fac = comb_o + 2 * cfl;                                           // [kFacMax]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int cta = blockIdx.x;
  if (tid == 0) *s_t0 = globaltimer_ns();

  // the next kernel in the stream may start as this grid's CTAs finish (programmatic
  // dependent launch); it waits for this grid before touching shared workspace or outputs.
  // A grid that waits for the page lists (wait_tables) lets it start only after that wait:
  // the kernel that writes the lists (a page-score call) is then complete, so a next
  // page-score call that starts early cannot write the score workspace under its feet
  if (!a.wait_tables) griddep_launch_dependents();

  // ---------------- this CTA's work items and their page-table bases, one parallel round trip.
  // Page tables and q are read from L2 (ld.global.cg): the kernel before this one in the
  // stream may have written them just before this grid started
  // the CTA's first item, its item count and its index in one load (no dependent read of cta_off)
  const tg_work_item lead = a.lead[cta];
  const int n_items = lead.reserved[0];
  const int i_begin = lead.reserved[1];
  const bool items_in_smem = n_items <= kMaxItems;
  if (items_in_smem) {
    // (thread i stores item i: it also reads it below for the page-table base)
    tg_work_item first = lead;
    first.reserved[0] = first.reserved[1] = 0;
    for (int i = tid; i < n_items; i += NT) s_items[i] = i == 0 ? first : a.items[i_begin + i];
  }
  // page tables written by the kernel just before this one (which let this grid start
  // early): wait for it first
  if (a.wait_tables) {
    griddep_wait();
    griddep_launch_dependents();
  }
  // page lists written by other CTAs of this same grid (fused sparse layer): wait for the
  // rows of this CTA's items
  if (a.row_ready)
    for (int i = tid; i < n_items; i += NT) {
      const tg_work_item it = a.items[i_begin + i];
      const int r = it.b * a.H + it.h;
      if (it.t1 > it.t0 && (!a.row_due || a.row_due[r]) && !wait_flag(a.row_ready + r, a.epoch, a.wait_ns))
        report(a.status, TG_STATUS_TIMEOUT);
    }
  if (items_in_smem)
    for (int i = tid; i < n_items; i += NT) s_base[i] = __ldcg(a.pt_off + s_items[i].b * a.G + s_items[i].g);
  if (warp < NW && lane == 0)
    for (int s = 0; s < R; ++s) mbar_init(&bars[warp * R + s], 1);
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&full[b], NS);
      mbar_init(&empty[b], NET);
    }
    *s_dead = 0;
    prefetch_tensormap(&pool_map);
  }
  fence_barrier_init();
  __syncthreads();
  if (tid == 0 && items_in_smem) {  // shared-run pieces first, then owned runs, each in plan order
    int c = 0;
    for (int i = 0; i < n_items; ++i)
      if (s_items[i].nparts > 1) s_order[c++] = i;
    for (int i = 0; i < n_items; ++i)
      if (s_items[i].nparts <= 1) s_order[c++] = i;
  }
  __syncthreads();
  // item and page-table base at processing position k (plan order when the items are in global)
  auto get_item = [&](int k) -> tg_work_item { return items_in_smem ? s_items[s_order[k]] : a.items[i_begin + k]; };
  auto get_base = [&](int k, const tg_work_item &it) -> int64_t {
    return items_in_smem ? s_base[s_order[k]] : __ldcg(a.pt_off + it.b * a.G + it.g);
  };

  if (warp < NW) {
    // ================================================================ streaming warps
    // tiles of item `it` that this warp takes: lo + warp, lo + warp + NW, ...
    auto warp_tiles = [&](const tg_work_item &it, int &lo) -> int {
      int hi;
      item_tiles(it, lo, hi);
      return hi - lo > warp ? (hi - lo - warp + NW - 1) / NW : 0;
    };
    int total_tiles = 0;
    for (int k = 0; k < n_items; ++k) {
      int lo;
      total_tiles += warp_tiles(get_item(k), lo);
    }

    // producer: page ids of the warp's tiles, 32 at a time, one per lane, loaded a batch
    // ahead so no TMA issue waits on a global load
    auto tile_info = [&](int n, int32_t &page, int &row_in_page) {
      page = -1;
      row_in_page = -1;
      if (n >= total_tiles) return;
      int rem = n;
      for (int k = 0; k < n_items; ++k) {
        const tg_work_item it = get_item(k);
        int lo;
        const int cnt = warp_tiles(it, lo);
        if (rem < cnt) {
          const int tok = 16 * (lo + warp + NW * rem);
          page = __ldcg(a.pt_ids + get_base(k, it) + tok / a.P);
          row_in_page = it.hpos * 2 * a.P + tok % a.P;  // first K row of the tile inside its page
          return;
        }
        rem -= cnt;
      }
    };
    int32_t pg_cur, pg_nxt;
    int rw_cur, rw_nxt;
    tile_info(lane, pg_cur, rw_cur);
    tile_info(32 + lane, pg_nxt, rw_nxt);
    int issued = 0, consumed = 0;
    auto issue = [&]() {  // whole warp: tile number `issued` of this warp into stage issued % R
      const int32_t page = __shfl_sync(0xffffffffu, pg_cur, issued & 31);
      const int rip = __shfl_sync(0xffffffffu, rw_cur, issued & 31);
      if (lane == 0) {
        const int s = issued % R;
        uint64_t *bar = &bars[warp * R + s];
        uint8_t *dst = ring + (warp * R + s) * LY::STAGE;
        if (page < 0 || (int64_t)page >= a.pool_pages || rip < 0) {
          report(a.status, TG_STATUS_BAD_PAGE);
          mbar_arrive(bar);  // complete the phase without data
        } else {
          const int row_k = (int)((int64_t)page * a.H_p * 2 * a.P + rip);
          mbar_arrive_expect_tx(bar, LY::STAGE);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(dst + c * 2048, &pool_map, bar, c * 64, row_k);
            tma_load_2d(dst + LY::TILE + c * 2048, &pool_map, bar, c * 64, row_k + a.P);
          }
        }
      }
      ++issued;
      if ((issued & 31) == 0) {
        pg_cur = pg_nxt;
        rw_cur = rw_nxt;
        tile_info(issued + 32 + lane, pg_nxt, rw_nxt);
      }
    };
    for (int s = 0; s < R && issued < total_tiles; ++s) issue();

    bool dead = false;  // a copy wait timed out: skip all further tiles, keep handing off
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // query fragments (B operand of S^T = K Q^T): this item's, and the next item's in flight
    uint32_t qf[KS][2], qn[KS][2];
    auto load_q = [&](int k) {
      if (k >= n_items) return;
      const tg_work_item it = get_item(k);
      const uint16_t *qrow = a.q + ((size_t)it.b * a.H_q + (size_t)it.h * a.g + gid) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qn[ks][0] = gid < a.g ? __ldcg(reinterpret_cast<const unsigned int *>(qrow + 16 * ks + 2 * tig)) : 0u;
        qn[ks][1] = gid < a.g ? __ldcg(reinterpret_cast<const unsigned int *>(qrow + 16 * ks + 8 + 2 * tig)) : 0u;
      }
    };
    auto next_item_with_tiles = [&](int from) {
      for (int k = from; k < n_items; ++k) {
        int lo;
        if (warp_tiles(get_item(k), lo) > 0) return k;
      }
      return n_items;
    };
    load_q(next_item_with_tiles(0));

    for (int k = 0; k < n_items; ++k) {
      const tg_work_item it = get_item(k);
      int k_lo, k_hi;
      item_tiles(it, k_lo, k_hi);
      if (k_hi - k_lo > warp && !dead) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qf[ks][0] = qn[ks][0];
          qf[ks][1] = qn[ks][1];
        }
        load_q(next_item_with_tiles(k + 1));
        for (int kk = k_lo + warp; kk < k_hi; kk += NW) {
          const int s = consumed % R;
          bool ok = mbar_wait(&bars[warp * R + s], (uint32_t)((consumed / R) & 1), kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {
            if (lane == 0) report(a.status, TG_STATUS_TIMEOUT);
            dead = true;
            break;
          }
          const uint32_t kbase = smem_addr(ring + (warp * R + s) * LY::STAGE);
          const uint32_t vbase = kbase + LY::TILE;
          const int r0 = it.t0 - kk * 16, r1 = it.t1 - kk * 16;  // valid rows [r0, r1) of the tile

          // S^T = K . Q^T  (rows: tokens, cols: query heads)
          float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kbase + swz((lane & 7) + ((lane >> 3) & 1) * 8, ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
            mma_16816(sc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
          }
          // online softmax, base 2; thread holds tokens gid, gid+8 of heads 2*tig, 2*tig+1
          const bool v0 = gid >= r0 && gid < r1, v1 = gid + 8 >= r0 && gid + 8 < r1;
          float z0 = v0 ? sc[0] * a.scale_log2 : -INFINITY;
          float z1 = v0 ? sc[1] * a.scale_log2 : -INFINITY;
          float z2 = v1 ? sc[2] * a.scale_log2 : -INFINITY;
          float z3 = v1 ? sc[3] * a.scale_log2 : -INFINITY;
          float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float c0 = ex2(m0 - mn0), c1 = ex2(m1 - mn1);
          const float p0 = ex2(z0 - mn0), p1 = ex2(z1 - mn1), p2 = ex2(z2 - mn0), p3 = ex2(z3 - mn1);
          // the weights go to the P.V product rounded to bf16; the row sums add the same
          // rounded weights, so the output is a weighted mean of V under one set of weights
          const uint32_t pk01 = pack_bf16x2(p0, p1), pk23 = pack_bf16x2(p2, p3);
          l0 = l0 * c0 + __uint_as_float(pk01 << 16) + __uint_as_float(pk23 << 16);
          l1 = l1 * c1 + __uint_as_float(pk01 & 0xffff0000u) + __uint_as_float(pk23 & 0xffff0000u);
          m0 = mn0;
          m1 = mn1;
          const uint32_t b0 = movmatrix_t(pk01);
          const uint32_t b1 = movmatrix_t(pk23);
          // O^T += V^T . P^T
#pragma unroll
          for (int mb = 0; mb < KS; ++mb) {
            o[mb][0] *= c0;
            o[mb][1] *= c1;
            o[mb][2] *= c0;
            o[mb][3] *= c1;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vbase + swz((lane & 7) + (lane >> 4) * 8, mb * 16 + ((lane >> 3) & 1) * 8), a0, a1, a2, a3);
            mma_16816(o[mb], a0, a1, a2, a3, b0, b1);
          }
          ++consumed;
          __syncwarp();
          if (issued < total_tiles) {
            if (lane == 0) fence_proxy_async_smem();  // our ldmatrix reads of this stage come before the refill
            issue();
          }
        }
      }

      // ---- hand this warp's state of item k to the epilogue (buffer k & 1, its use k >> 1)
      const int hb = k & 1, use = k >> 1;
      if (use > 0 && !*s_dead && !mbar_wait(&empty[hb], (uint32_t)((use - 1) & 1), kWaitLimitNs)) {
        if (lane == 0) report(a.status, TG_STATUS_TIMEOUT);
        *s_dead = 1;
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      float *cm = comb_m + (hb * NW + warp) * 8, *cl = comb_l + (hb * NW + warp) * 8;
      if (gid == 0) {
        cm[2 * tig] = m0;
        cm[2 * tig + 1] = m1;
        cl[2 * tig] = l0;
        cl[2 * tig + 1] = l1;
      }
      float *co = comb_o + hb * cfl + warp * a.g * ostride;  // [g][ostride] of this warp
      const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
      for (int mb = 0; mb < KS; ++mb) {
        if (h0 < a.g) {
          co[h0 * ostride + mb * 16 + gid] = o[mb][0];
          co[h0 * ostride + mb * 16 + gid + 8] = o[mb][2];
        }
        if (h1 < a.g) {
          co[h1 * ostride + mb * 16 + gid] = o[mb][1];
          co[h1 * ostride + mb * 16 + gid + 8] = o[mb][3];
        }
        o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;
      }
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
      mbar_arrive(&full[hb]);  // (release: this thread's hand-off writes come first)
      // stream past the first item only once the previous decode launch in the stream is
      // done: racing further ahead of its last CTAs measured slower back to back
      if (k == 0) griddep_wait();
    }

    // drain copies still in flight (only after a timeout; otherwise issued == consumed)
    if (lane == 0) {
      for (int t = consumed; t < issued; ++t)
        if (!mbar_wait(&bars[warp * R + t % R], (uint32_t)((t / R) & 1), kWaitLimitNs)) break;
    }
    __syncwarp();
    return;
  }

  // ================================================================== epilogue warps
  const int etid = tid - NS, ew = warp - NW;
  // the workspace (merge counters, partials) and the outputs may still be in use by the
  // previous decode launch in the stream: wait for it before the first write
  griddep_wait();
  for (int k = 0; k < n_items; ++k) {
    const tg_work_item it = get_item(k);
    const int hb = k & 1, use = k >> 1;
    if (!*s_dead && !mbar_wait_sleep(&full[hb], (uint32_t)(use & 1), kWaitLimitNs)) {
      if (etid == 0) report(a.status, TG_STATUS_TIMEOUT);
      *s_dead = 1;
    }
    const float *cm = comb_m + hb * NW * 8, *cl = comb_l + hb * NW * 8, *co = comb_o + hb * cfl;
    const size_t out_row0 = (size_t)it.b * a.H_q + (size_t)it.h * a.g;
    if (it.t1 <= it.t0) {  // a head with no retained token
      for (int e = etid; e < a.g * D; e += NET) {
        a.out[(out_row0 + e / D) * D + e % D] = 0;
        if (e % D == 0 && a.lse) a.lse[out_row0 + e / D] = -INFINITY;
      }
    } else {
      const int slot = it.slot0 + it.part;
      for (int e = etid; e < a.g * D; e += NET) {
        const int hd = e / D, dd = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[w * 8 + hd]);
        float Ls = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float f = ex2(cm[w * 8 + hd] - M);
          Ls += cl[w * 8 + hd] * f;
          O += co[(w * a.g + hd) * ostride + dd] * f;
        }
        if (it.nparts == 1) {
          __nv_bfloat16 v = __float2bfloat16_rn(O / Ls);
          a.out[(out_row0 + hd) * D + dd] = *reinterpret_cast<uint16_t *>(&v);
          if (dd == 0 && a.lse) a.lse[out_row0 + hd] = (M + log2f(Ls)) * kLn2;
        } else {
          a.ws_o[((size_t)slot * a.g + hd) * D + dd] = O;
          if (dd == 0) {
            a.ws_ml[((size_t)slot * a.g + hd) * 2] = M;
            a.ws_ml[((size_t)slot * a.g + hd) * 2 + 1] = Ls;
          }
        }
      }
    }
    mbar_arrive(&empty[hb]);  // (release: this thread's reads of the buffer come first)
    if (it.t1 > it.t0 && it.nparts > 1) {
      __threadfence();
      epilogue_sync<NET>();
      if (etid == 0) {
        const int prev = atomicAdd(&a.counters[it.b * a.H + it.h], 1);
        *flag = prev == it.nparts - 1;
      }
      epilogue_sync<NET>();
      if (*flag) {  // the last CTA of this run merges every partial
        __threadfence();
        const int np = it.nparts, g = a.g;
        const float *pml = a.ws_ml + (size_t)it.slot0 * g * 2;  // [nparts][g][2]
        const float *po = a.ws_o + (size_t)it.slot0 * g * D;     // [nparts][g][D]
        if (np * g <= kFacMax) {
          // factors 2^(m_p - M) of every part go to shared memory; per head, one warp gathers
          // M and L with its lanes striding over the parts (independent loads).  Up to 64 parts,
          // each lane reads its (m, l) pairs once and keeps them in registers
          for (int hh = ew; hh < g; hh += NE) {
            float M = -INFINITY, Ls = 0.f;
            if (np <= 64) {
              float2 ml[2];
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int p = lane + 32 * j;
                ml[j] = p < np ? __ldcg(reinterpret_cast<const float2 *>(pml + ((size_t)p * g + hh) * 2))
                               : make_float2(-INFINITY, 0.f);
                M = fmaxf(M, ml[j].x);
              }
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int p = lane + 32 * j;
                if (p < np) {
                  const float f = ex2(ml[j].x - M);
                  fac[p * g + hh] = f;
                  Ls += ml[j].y * f;
                }
              }
            } else {
              for (int p = lane; p < np; p += 32) M = fmaxf(M, __ldcg(pml + ((size_t)p * g + hh) * 2));
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
              for (int p = lane; p < np; p += 32) {
                const float f = ex2(__ldcg(pml + ((size_t)p * g + hh) * 2) - M);
                fac[p * g + hh] = f;
                Ls += __ldcg(pml + ((size_t)p * g + hh) * 2 + 1) * f;
              }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
            if (lane == 0) {
              s_mm[hh] = M;
              s_ll[hh] = Ls;
            }
          }
          epilogue_sync<NET>();
          // O = sum_p o_p 2^(m_p - M), parts in order.  A thread takes four consecutive outputs
          // of one head (16-byte loads; partial rows are 16-byte aligned), sixteen parts per
          // batch in flight
          for (int e = 4 * etid; e < g * D; e += 4 * NET) {
            const int hd = e / D, dd = e % D;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int p = 0; p < np; p += 16) {
              float4 v[16];
#pragma unroll
              for (int u = 0; u < 16; ++u)
                v[u] = p + u < np ? __ldcg(reinterpret_cast<const float4 *>(po + (size_t)(p + u) * g * D + e))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int u = 0; u < 16; ++u)
                if (p + u < np) {
                  const float f = fac[(p + u) * g + hd];
                  O.x += v[u].x * f;
                  O.y += v[u].y * f;
                  O.z += v[u].z * f;
                  O.w += v[u].w * f;
                }
            }
            const float Ls = s_ll[hd];
            uint16_t *orow = a.out + (out_row0 + hd) * D + dd;
            const float ov[4] = {O.x, O.y, O.z, O.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              __nv_bfloat16 v = __float2bfloat16_rn(ov[c] / Ls);
              orow[c] = *reinterpret_cast<uint16_t *>(&v);
            }
            if (dd == 0 && a.lse) a.lse[out_row0 + hd] = (s_mm[hd] + log2f(s_ll[hd])) * kLn2;
          }
        } else {  // more parts than the factor buffer holds: straight loops
          for (int e = etid; e < g * D; e += NET) {
            const int hd = e / D, dd = e % D;
            float M = -INFINITY;
            for (int p = 0; p < np; ++p) M = fmaxf(M, __ldcg(pml + ((size_t)p * g + hd) * 2));
            float Ls = 0.f, O = 0.f;
            for (int p = 0; p < np; ++p) {
              const float f = ex2(__ldcg(pml + ((size_t)p * g + hd) * 2) - M);
              Ls += __ldcg(pml + ((size_t)p * g + hd) * 2 + 1) * f;
              O += __ldcg(po + (size_t)p * g * D + e) * f;
            }
            __nv_bfloat16 v = __float2bfloat16_rn(O / Ls);
            a.out[(out_row0 + hd) * D + dd] = *reinterpret_cast<uint16_t *>(&v);
            if (dd == 0 && a.lse) a.lse[out_row0 + hd] = (M + log2f(Ls)) * kLn2;
          }
        }
        if (etid == 0) atomicExch(&a.counters[it.b * a.H + it.h], 0);
      }
      epilogue_sync<NET>();  // the flag, the factors and (M, L) are reused by the next item
    }
  }
  if (etid == 0 && a.cta_time) {
    a.cta_time[2 * cta] = (int64_t)*s_t0;
    a.cta_time[2 * cta + 1] = (int64_t)globaltimer_ns();
  }
}


// ---------------------------------------------------------------- host side, shared by the
// decode entry points and the fused sparse-layer kernel

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// TMA map of the pool seen as rows of d bf16 values (boxes of 16 rows x 64 columns, 128-byte
// swizzle); TG_OK or an error with the message set
inline int make_pool_map(CUtensorMap *map, const uint16_t *pool, int64_t pool_pages, const tg_plan_header *hd,
                         const char *fn) {
  const int64_t rows = pool_pages * hd->H_p * 2 * hd->P;
  if (pool_pages <= 0 || rows > INT32_MAX)
    return tgi::fail(TG_ERR_CAPACITY, "%s: pool_pages=%lld gives %lld rows (1..2^31-1)", fn, (long long)pool_pages,
                     (long long)rows);
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return tgi::fail(TG_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", fn);
  const cuuint64_t gdim[2] = {(cuuint64_t)hd->d, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)hd->d * 2};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estride[2] = {1, 1};
  CUresult cr = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(pool), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return tgi::fail(TG_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", fn, (int)cr);
  return TG_OK;
}

// the checks every decode launch of a plan makes; on success *hd_out / *lt_out point into plan_host
inline int check_decode_call(const char *fn, const void *plan_host, const void *plan_dev, int layer,
                             const uint16_t *q, const uint16_t *pool, float scale, const tg_plan_header **hd_out,
                             const tg_plan_layer **lt_out) {
  const tg_plan_header *hd = static_cast<const tg_plan_header *>(plan_host);
  if (hd->magic != TG_PLAN_MAGIC || hd->version != TG_PLAN_VERSION)
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: plan_host is not a tg_plan_decode buffer", fn);
  if (layer < 0 || layer >= hd->L) return tgi::fail(TG_ERR_INVALID_ARG, "%s: layer %d of %d", fn, layer, hd->L);
  if (!std::isfinite(scale)) return tgi::fail(TG_ERR_NONFINITE, "%s: scale is not finite", fn);
  if ((reinterpret_cast<uintptr_t>(pool) & 15) || (reinterpret_cast<uintptr_t>(plan_dev) & 15) ||
      (reinterpret_cast<uintptr_t>(q) & 3))
    return tgi::fail(TG_ERR_INVALID_ARG, "%s: pool and plan must be 16-byte aligned", fn);
  *hd_out = hd;
  *lt_out = reinterpret_cast<const tg_plan_layer *>(static_cast<const uint8_t *>(plan_host) + hd->layers) + layer;
  return TG_OK;
}

// kernel arguments of one decode launch; ws is the scratch (a caller workspace or the fixed array)
inline DecodeArgs decode_args(const tg_plan_header *hd, const tg_plan_layer *lt, const void *plan_dev, uint8_t *ws,
                              const uint16_t *q, uint16_t *out, float *lse, const int64_t *pt_off,
                              const int32_t *pt_ids, int64_t pool_pages, float scale, int32_t *dev_status,
                              int64_t *cta_time) {
  const int g = hd->H_q / hd->H;
  const tgi::WorkspaceLayout wl = tgi::workspace_layout(hd->batch, hd->H, g, hd->d, hd->max_slots);
  const uint8_t *pd = static_cast<const uint8_t *>(plan_dev);
  DecodeArgs args;
  args.items = reinterpret_cast<const tg_work_item *>(pd + lt->items);
  args.lead = reinterpret_cast<const tg_work_item *>(pd + lt->lead);
  args.cta_off = reinterpret_cast<const int32_t *>(pd + lt->cta_off);
  args.q = q;
  args.out = out;
  args.lse = lse;
  args.pt_off = pt_off;
  args.pt_ids = pt_ids;
  args.pool_pages = pool_pages;
  args.counters = reinterpret_cast<int32_t *>(ws + wl.counters);
  args.ws_ml = reinterpret_cast<float *>(ws + wl.ml);
  args.ws_o = reinterpret_cast<float *>(ws + wl.o);
  // without a caller status word, faults are recorded in the scratch's own
  args.status = dev_status ? dev_status : reinterpret_cast<int32_t *>(ws + wl.status);
  args.cta_time = cta_time;
  args.H = hd->H;
  args.H_q = hd->H_q;
  args.g = g;
  args.G = hd->G;
  args.H_p = hd->H_p;
  args.P = hd->P;
  args.scale_log2 = scale * kLog2e;
  args.wait_tables = (hd->flags & TG_PLAN_WAIT_TABLES) != 0;
  args.row_ready = nullptr;
  args.row_due = nullptr;
  args.wait_ns = kWaitLimitNs;
  args.epoch = 0;
  return args;
}

}  // namespace
