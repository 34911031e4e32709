// Layout of the caller-provided scratch of the verify / fused-step kernels.
//
//   [0]   uint32 next_unit   dynamic work counter of the persistent grid
//   [4]   uint32 ctas_done   CTAs that have left the work loop
//   [8]   uint32 count[B]    finished argmax units per request
//   [..]  uint64 key[rows]   running (value, column) maximum per logits row
//
// Every field is zero between calls: the last arriving unit of a request
// reads its keys with an exchange against 0 and clears its count; the last
// CTA to leave clears the two scheduler words.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pe {

struct WorkspaceLayout {
  size_t count_off, key_off, bytes;
  WorkspaceLayout(int64_t rows, int64_t B) {
    count_off = 8;
    key_off = (count_off + 4 * (size_t)B + 7) & ~(size_t)7;
    bytes = (key_off + 8 * (size_t)rows + 255) & ~(size_t)255;
  }
};

}  // namespace pe
