// Block-wide helpers for exact top-k selection with ties to the lower index:
// exclusive scans of per-thread flags (one, or U per thread) and MSB-first radix selects over
// order-preserving uint32 keys (a plain one for short rows, and one with wide digits that
// narrows to a candidate list in shared memory).  Used by the one-shot compaction's copy
// (the scans), the chunked token compaction and the page top-K of long rows.
#pragma once

#include <cstdint>

namespace tgk {

// Exclusive prefix count of `flag` over the block (thread order), plus the total.
// `scratch` holds at least 33 ints of shared memory.  Contains two __syncthreads.
template <int NT>
__device__ __forceinline__ int block_excl_count(bool flag, int *scratch, int &total) {
  static_assert(NT % 32 == 0 && NT <= 1024, "block size");
  constexpr int NWARP = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) scratch[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = lane < NWARP ? scratch[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < NWARP) scratch[lane] = inc - v;
    if (lane == 31) scratch[32] = inc;
  }
  __syncthreads();
  total = scratch[32];
  return scratch[warp] + in_warp;
}

// Exclusive prefix counts of U flags per thread over the block, in the order (u, thread):
// every thread's flag u comes after all flags u' < u and after flag u of lower threads.
// rank[u] is flag u's count of earlier set flags; `total` the block's set flags.  `scratch`
// holds at least U * NT / 32 + 1 ints of shared memory.  Contains two __syncthreads.
template <int NT, int U>
__device__ __forceinline__ void block_excl_count_multi(const bool (&flag)[U], int *scratch, int (&rank)[U],
                                                       int &total) {
  constexpr int NWARP = NT / 32, NV = U * NWARP, PER = NV / 32;
  static_assert(NT % 32 == 0 && NT <= 1024 && NV % 32 == 0, "block size");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  int in_warp[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint32_t bal = __ballot_sync(0xffffffffu, flag[u]);
    in_warp[u] = __popc(bal & lt);
    if (lane == 0) scratch[u * NWARP + warp] = __popc(bal);
  }
  __syncthreads();
  if (warp == 0) {
    // lane l scans values l*PER .. l*PER + PER - 1 of the (u, warp) sequence
    int v[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      v[j] = scratch[lane * PER + j];
      sum += v[j];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    int run = inc - sum;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      scratch[lane * PER + j] = run;
      run += v[j];
    }
    if (lane == 31) scratch[NV] = inc;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < U; ++u) rank[u] = scratch[u * NWARP + warp] + in_warp[u];
  total = scratch[NV];
}

// Find the key T of the k-th largest of `count` keys (1 <= k <= count) and the
// number of keys equal to T that a top-k must take (the lowest-indexed ones):
// need_eq = k - #{key > T}.  get(i) returns key i.  `hist` is 256 ints and
// `scratch` 4 ints of shared memory.
template <int NT, typename GetKey>
__device__ __forceinline__ void block_radix_select(int count, int k, GetKey get, int *hist, int *scratch,
                                                   uint32_t &T, int &need_eq) {
  uint32_t prefix = 0, mask = 0;
  int k_rem = k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
    __syncthreads();
    // histogram of the next digit among keys that match the prefix so far.  In the first
    // pass the leading digits of real scores coincide, and lanes of a warp with the same
    // digit add once; later digits are spread out, where that grouping costs more than
    // the atomics it saves
    for (int base = 0; base < count; base += NT) {
      const int i = base + threadIdx.x;
      uint32_t dg = 256u;  // no digit
      if (i < count) {
        const uint32_t key = get(i);
        if ((key & mask) == prefix) dg = (key >> shift) & 255u;
      }
      if (shift == 24) {
        const uint32_t peers = __match_any_sync(0xffffffffu, dg);
        if (dg < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[dg], __popc(peers));
      } else if (dg < 256u) {
        atomicAdd(&hist[dg], 1);
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255-8l down to 248-8l; scan from the top digit down
      int local[8];
      int s = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        local[t] = hist[255 - 8 * lane - t];
        s += local[t];
      }
      int inc = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const int before = inc - s;  // keys in digits above this lane's block
      if (before < k_rem && k_rem <= inc) {
        int above = before;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (above + local[t] >= k_rem) {
            scratch[0] = 255 - 8 * lane - t;
            scratch[1] = above;
            break;
          }
          above += local[t];
        }
      }
    }
    __syncthreads();
    const uint32_t digit = (uint32_t)scratch[0];
    k_rem -= scratch[1];
    prefix |= digit << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  T = prefix;
  need_eq = k_rem;
}

// The same selection for many keys, also returning n_eq, the number of keys equal to T, with
// digits of 12, 10 and 10 bits and plain shared-memory atomics: the top 12 bits of a float key
// (sign, exponent and three mantissa bits) spread real scores over many counters, where an
// 8-bit first digit piles them into a few (grouping a warp's equal digits with match_any
// instead measured at several hundred cycles a key).  hist0 holds 4096 ints and may share its
// memory with `list` (it is dead once the first digit is chosen); hist1 holds 1024 ints of its
// own; scratch holds NT / 32 + 4 ints.  After the first digit, the keys under it are copied
// into `list` when at most `cap` (NULL: none), and the other passes read only them; passes
// over get() keep four keys in flight per thread.
template <int NT, typename GetKey>
__device__ void block_select_kth_wide(int count, int k, GetKey get, uint32_t *list, int cap, int *hist0, int *hist1,
                                      int *scratch, uint32_t &T, int &need_eq, int &n_eq) {
  constexpr int U = 4;
  static_assert(NT % 32 == 0 && 4096 % NT == 0 && NT <= 1024, "block size");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, mask = 0;
  int k_rem = k, sel_count = count, n_list = -1;
  // the digit (of `bins` counters in h) that holds the k_rem-th key: thread t owns the bins
  // bins-1-t*per .. bins-(t+1)*per (from the top down), a block scan finds the owner
  auto pick = [&](const int *h, int bins, int shift, int bits) {
    const int per = bins / NT, top = bins - 1 - tid * per;
    int s = 0;
    for (int j = 0; j < per; ++j) s += h[top - j];
    int inc = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) scratch[4 + warp] = inc;
    __syncthreads();
    int before = inc - s;
    for (int w = 0; w < warp; ++w) before += scratch[4 + w];
    if (before < k_rem && k_rem <= before + s) {
      int above = before;
      for (int j = 0; j < per; ++j) {
        const int c = h[top - j];
        if (above + c >= k_rem) {
          scratch[0] = top - j;
          scratch[1] = above;
          scratch[2] = c;
          break;
        }
        above += c;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)scratch[0] << shift;
    mask |= ((1u << bits) - 1u) << shift;
    k_rem -= scratch[1];
    sel_count = scratch[2];
    __syncthreads();  // (scratch and the counters are reused)
  };
  // first digit, over every key
  for (int i = tid; i < 4096; i += NT) hist0[i] = 0;
  __syncthreads();
  for (int base = 0; base < count; base += NT * U) {
    uint32_t kk[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NT + tid;
      kk[u] = i < count ? get(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + u * NT + tid < count) atomicAdd(&hist0[kk[u] >> 20], 1);
  }
  __syncthreads();
  pick(hist0, 4096, 20, 12);
  if (list && sel_count <= cap) {
    // copy the keys under the first digit into the list (order does not matter for counts)
    if (tid == 0) scratch[3] = 0;
    __syncthreads();
    for (int base = 0; base < count; base += NT * U) {
      uint32_t kk[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * NT + tid;
        kk[u] = i < count ? get(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool keep = base + u * NT + tid < count && (kk[u] & mask) == prefix;
        const uint32_t bal = __ballot_sync(0xffffffffu, keep);
        int at = 0;
        if (lane == 0 && bal) at = atomicAdd(&scratch[3], __popc(bal));
        at = __shfl_sync(0xffffffffu, at, 0);
        if (keep) list[at + __popc(bal & ((1u << lane) - 1u))] = kk[u];
      }
    }
    n_list = sel_count;
    __syncthreads();
  }
  // two digits of 10 bits over the list (or every key)
  for (int shift = 10; shift >= 0; shift -= 10) {
    for (int i = tid; i < 1024; i += NT) hist1[i] = 0;
    __syncthreads();
    if (n_list >= 0) {
      for (int i = tid; i < n_list; i += NT) {
        const uint32_t key = list[i];
        if ((key & mask) == prefix) atomicAdd(&hist1[(key >> shift) & 1023u], 1);
      }
    } else {
      for (int base = 0; base < count; base += NT * U) {
        uint32_t kk[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = base + u * NT + tid;
          kk[u] = i < count ? get(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (base + u * NT + tid < count && (kk[u] & mask) == prefix) atomicAdd(&hist1[(kk[u] >> shift) & 1023u], 1);
      }
    }
    __syncthreads();
    pick(hist1, 1024, shift, 10);
  }
  T = prefix;
  need_eq = k_rem;
  n_eq = sel_count;
}

}  // namespace tgk
