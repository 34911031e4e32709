// Layout of the caller-provided scratch of the verify / fused-step kernels.
//
//   [0]   uint32 next_unit     dynamic work counter of the persistent grid
//   [4]   uint32 ctas_done     CTAs that have left the work loop
//   [8]   uint32 count[B]      finished argmax units per request (early exit:
//                              rows known to mismatch before they complete)
//   [..]  uint64 state[B]      early exit: rows done (bits 0-31) and rows
//                              whose argmax matched the draft (bits 32-63)
//   [..]  uint64 xfer[B]       bonus-row hand-off between the copy tiles and
//                              the request's verdict: verified rows whose
//                              default embedding half is written (bits
//                              0-15), verdict known (bit 16), accepted
//                              length (bits 17-24), bonus token (bits 32-63)
//   [..]  uint64 key[rows]     running (value, column) maximum per logits row
//   [..]  uint32 rcount[rows]  early exit: finished chunks per row
//   [..]  int32  amax[rows]    early exit: argmax of each completed row
//   [..]  uint64 slot[1024]    single pass: each argmax unit's chunk key
//
// Every field is zero between calls, so one workspace serves calls of any
// size up to the one it was sized for: the full step clears a request's keys
// and count when its last unit arrives, and its hand-off word when the
// bonus row is written, the early-exit step clears completed
// rows as they complete and everything else (partly read rows, states,
// early-mismatch words, row results) in its last CTA; the last CTA to leave clears the two scheduler
// words; in the single pass, the CTA that collects a request's chunk keys
// clears their slots.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pe {

constexpr int kSinglePassSlots = 1024;  // argmax units of a single-pass step, at most

struct WorkspaceLayout {
  size_t count_off, state_off, xfer_off, key_off, rcount_off, amax_off, slot_off, bytes;
  WorkspaceLayout(int64_t rows, int64_t B) {
    count_off = 8;
    state_off = (count_off + 4 * (size_t)B + 7) & ~(size_t)7;
    xfer_off = state_off + 8 * (size_t)B;
    key_off = xfer_off + 8 * (size_t)B;
    rcount_off = key_off + 8 * (size_t)rows;
    amax_off = rcount_off + 4 * (size_t)rows;
    slot_off = (amax_off + 4 * (size_t)rows + 7) & ~(size_t)7;
    bytes = (slot_off + 8 * (size_t)kSinglePassSlots + 255) & ~(size_t)255;
  }
};

}  // namespace pe
