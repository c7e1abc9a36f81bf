// Page allocator for budget reservation.
//
// Source: "Tangram: Unlocking Non-Uniform KV Cache Compression for Efficient
// Multi-turn LLM Serving" (paper-review page), 3.1 Budget Reservation (each
// request's post-compression footprint is fixed when it is scheduled, so its
// pages are allocated once and no runtime page reclamation is needed) and 3.2
// Ragged Paging (one page table per (layer, request, head group)).
//
// The pool's free pages form a stack held in caller memory (no global state).
// Admission is all-or-nothing: either every list of the request gets its pages
// or nothing is taken.  Pages are handed out lowest id first on a fresh pool;
// released pages are pushed back and reused last-in first-out.  A bitmap of
// allocated pages rejects a double or foreign release.
#include "tg_internal.h"

#include <cstring>

namespace {

using tgi::fail;

constexpr uint32_t kAllocMagic = 0x41504754u;  // "TGPA"

struct AllocHeader {
  uint32_t magic;
  int32_t reserved;
  int64_t n_pages;  // pool size
  int64_t n_free;   // pages on the free stack
  int64_t live;     // pages handed out
};

// state: AllocHeader | int32 stack[n_pages] | uint64 used[ceil(n_pages / 64)]
int64_t state_bytes(int64_t n_pages) {
  return (int64_t)sizeof(AllocHeader) + tgi::align_up(n_pages * 4, 8) + ((n_pages + 63) / 64) * 8;
}
int32_t *stack_of(AllocHeader *h) { return reinterpret_cast<int32_t *>(h + 1); }
uint64_t *used_of(AllocHeader *h) {
  return reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(h + 1) + tgi::align_up(h->n_pages * 4, 8));
}
AllocHeader *checked(void *state, const char *fn) {
  AllocHeader *h = static_cast<AllocHeader *>(state);
  if (!h || h->magic != kAllocMagic) {
    fail(TG_ERR_INVALID_ARG, "%s: not an initialised allocator state", fn);
    return nullptr;
  }
  return h;
}

}  // namespace

extern "C" int tg_alloc_state_bytes(int64_t n_pages, int64_t *bytes) {
  if (n_pages < 0 || n_pages > INT32_MAX) return fail(TG_ERR_INVALID_ARG, "tg_alloc_state_bytes: n_pages=%lld", (long long)n_pages);
  if (!bytes) return fail(TG_ERR_INVALID_ARG, "tg_alloc_state_bytes: NULL bytes");
  *bytes = state_bytes(n_pages);
  return tgi::ok();
}

extern "C" int tg_alloc_init(void *state, int64_t state_cap, int64_t n_pages) {
  if (!state) return fail(TG_ERR_INVALID_ARG, "tg_alloc_init: NULL state");
  if (n_pages < 0 || n_pages > INT32_MAX) return fail(TG_ERR_INVALID_ARG, "tg_alloc_init: n_pages=%lld", (long long)n_pages);
  if (state_cap < state_bytes(n_pages))
    return fail(TG_ERR_CAPACITY, "tg_alloc_init: state %lld < %lld bytes", (long long)state_cap,
                (long long)state_bytes(n_pages));
  AllocHeader *h = static_cast<AllocHeader *>(state);
  std::memset(h, 0, (size_t)state_bytes(n_pages));
  h->magic = kAllocMagic;
  h->n_pages = n_pages;
  h->n_free = n_pages;
  int32_t *st = stack_of(h);
  for (int64_t i = 0; i < n_pages; ++i) st[i] = (int32_t)(n_pages - 1 - i);  // top of the stack = page 0
  return tgi::ok();
}

extern "C" int tg_alloc_admit(void *state, int n_lists, const int32_t *pages_per_list, int32_t *ids,
                              int64_t ids_cap, int64_t *n_ids) {
  AllocHeader *h = checked(state, "tg_alloc_admit");
  if (!h) return TG_ERR_INVALID_ARG;
  if (n_lists < 0 || (n_lists > 0 && !pages_per_list)) return fail(TG_ERR_INVALID_ARG, "tg_alloc_admit: bad lists");
  int64_t need = 0;
  for (int i = 0; i < n_lists; ++i) {
    if (pages_per_list[i] < 0) return fail(TG_ERR_INVALID_ARG, "tg_alloc_admit: list %d asks %d pages", i, pages_per_list[i]);
    need += pages_per_list[i];
  }
  if (n_ids) *n_ids = need;
  if (need > ids_cap || (need > 0 && !ids))
    return fail(TG_ERR_CAPACITY, "tg_alloc_admit: ids holds %lld, the request needs %lld", (long long)ids_cap,
                (long long)need);
  if (need > h->n_free)
    return fail(TG_ERR_CAPACITY, "tg_alloc_admit: %lld pages needed, %lld free", (long long)need, (long long)h->n_free);
  int32_t *st = stack_of(h);
  uint64_t *used = used_of(h);
  for (int64_t k = 0; k < need; ++k) {
    const int32_t p = st[--h->n_free];
    used[p >> 6] |= 1ull << (p & 63);
    ids[k] = p;
  }
  h->live += need;
  return tgi::ok();
}

extern "C" int tg_alloc_release(void *state, int64_t n, const int32_t *ids) {
  AllocHeader *h = checked(state, "tg_alloc_release");
  if (!h) return TG_ERR_INVALID_ARG;
  if (n < 0 || (n > 0 && !ids)) return fail(TG_ERR_INVALID_ARG, "tg_alloc_release: bad ids");
  uint64_t *used = used_of(h);
  // clear each page's bit as it is checked; a page that is free (or listed twice) finds its
  // bit clear, and the bits cleared so far are set again: a rejected release changes nothing
  for (int64_t k = 0; k < n; ++k) {
    const int32_t p = ids[k];
    if (p < 0 || p >= h->n_pages || !((used[p >> 6] >> (p & 63)) & 1ull)) {
      for (int64_t m = 0; m < k; ++m) used[ids[m] >> 6] |= 1ull << (ids[m] & 63);
      return fail(TG_ERR_INVALID_ARG, "tg_alloc_release: page %d is not allocated (or listed twice)", p);
    }
    used[p >> 6] &= ~(1ull << (p & 63));
  }
  int32_t *st = stack_of(h);
  for (int64_t k = n - 1; k >= 0; --k) st[h->n_free++] = ids[k];  // the request's first page ends on top
  h->live -= n;
  return tgi::ok();
}

extern "C" int tg_alloc_query(const void *state, int64_t *n_free, int64_t *n_live) {
  const AllocHeader *h = static_cast<const AllocHeader *>(state);
  if (!h || h->magic != kAllocMagic) return fail(TG_ERR_INVALID_ARG, "tg_alloc_query: not an initialised allocator state");
  if (n_free) *n_free = h->n_free;
  if (n_live) *n_live = h->live;
  return tgi::ok();
}
