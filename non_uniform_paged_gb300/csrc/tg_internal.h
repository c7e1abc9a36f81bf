// Internal helpers shared by the translation units of libtg (not installed).
#pragma once

#include "../../include/tg.h"

#include <cstdint>

namespace tgi {

// Record a message for tg_last_error_string() on this thread and return `code`.
int fail(int code, const char *fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;
// Clear the thread's message and return TG_OK.
int ok();

constexpr int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Byte offsets of the decode workspace sections:
// counters int32 [batch*H] | status int32 (used when the caller passes none) |
// m,l float32 [slots][g][2] | o float32 [slots][g][d]
struct WorkspaceLayout {
  int64_t counters, status, ml, o, total;
};
inline WorkspaceLayout workspace_layout(int batch, int H, int g, int d, int max_slots) {
  WorkspaceLayout w;
  w.counters = 0;
  w.status = align_up((int64_t)batch * H * 4, 256);
  w.ml = w.status + 256;
  w.o = w.ml + align_up((int64_t)max_slots * g * 2 * 4, 256);
  w.total = align_up(w.o + (int64_t)max_slots * g * d * 4, 256);
  return w;
}

}  // namespace tgi
