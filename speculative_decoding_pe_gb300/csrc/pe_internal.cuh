// Internal helpers of libpe.so (device and host).  Not part of the ABI.
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "pe_api.h"

namespace pe {

// ---------------------------------------------------------------- launch shape
constexpr int kThreads = 256;                 // threads per CTA, every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = 8;              // 16-byte loads per thread per batch
constexpr int kBatchVecs = kThreads * kVecPerThread;  // 2048 vectors = 32 KiB
constexpr int kMaxRowsPerUnit = 16;           // X rows per copy unit (upper bound)

// ------------------------------------------------------------- element access
// bf16 is by definition the high half of an IEEE-754 binary32, so widening is
// a shift; both halves of a 32-bit word hold one element each (low = first).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Lane-wise maximum of two pairs of bf16 values (returns one of the inputs,
// so it is exact).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------------------------------- ordering
// Device-scope release/acquire fence.  Every hand-off between CTAs or warps
// here is message passing: data stores, then a counter (or bit) update that
// tells the last arrival to read them.  That needs release ordering at the
// writer (fence, then the counter update, in the updating thread, after any
// barrier that gathers the other threads' stores) and acquire ordering at
// the reader (the update that reveals completion, then the fence, in that
// same thread, before the barrier that releases the other threads' loads).
// Sequential consistency (the fence __threadfence() gives) is not needed.
__device__ __forceinline__ void fence_acq_rel() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Global time in nanoseconds (bounds the few waits).
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Strong (relaxed, device-scope) 64-bit store and load: single-copy atomic,
// so a reader polling the word sees either its old value or the whole new
// one.  Used where the word itself is the message (no other data to order).
__device__ __forceinline__ void st_relaxed(unsigned long long* a, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}
// The two sides of the bonus-row hand-off word.  Each copy tile adds its
// rows with release and acquire semantics (its X writes, gathered by the
// CTA barrier before it, are published; the other tiles' writes are
// acquired); the verdict ORs in its result with acquire semantics only
// (the tiles need nothing but the word from it).  Whichever comes second
// has thereby acquired every default write of the row it overwrites, with
// no separate fence: the atomics' own ordering replaced a fence after the
// clear that cost ~0.45 us at the end of a B=1 step.
__device__ __forceinline__ unsigned long long atom_or_acquire(unsigned long long* a,
                                                          unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acquire.gpu.global.or.b64 %0, [%1], %2;"
               : "=l"(old) : "l"(a), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long* a,
                                                           unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
               : "=l"(old) : "l"(a), "l"(v) : "memory");
  return old;
}
// Counting with release and acquire semantics in the atomic itself: each
// arrival publishes what it wrote before (its key merge, a row's argmax),
// and the arrival that completes the count acquires every other's, with no
// fence on either side.
__device__ __forceinline__ unsigned atom_add_acq_rel_u32(unsigned* a, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_or_acq_rel(unsigned long long* a, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(a), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}

// Total order on non-NaN floats as unsigned integers, with -0.0 == +0.0.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// (value, column) packed so that the unsigned maximum is the largest value
// and, among equal values, the lowest column.  0 is below every real key.
__device__ __forceinline__ unsigned long long make_key(float v, uint32_t col) {
  return ((unsigned long long)ordered_bits(v) << 32) |
         (unsigned long long)(0xffffffffu - col);
}
__device__ __forceinline__ uint32_t key_col(unsigned long long k) {
  return 0xffffffffu - (uint32_t)k;
}

__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    unsigned long long x = __shfl_xor_sync(0xffffffffu, k, o);
    k = x > k ? x : k;
  }
  return k;
}

// ------------------------------------------------------------ checked build
// PE_CHECKED (libpe_checked.so): an internal index invariant that fails
// raises PE_ERR_INTERNAL and the access it guards is skipped; in the
// regular build the condition is not evaluated.
#ifdef PE_CHECKED
#define PE_INVARIANT(err, cond) ((cond) || (atomicOr((err), PE_ERR_INTERNAL), false))
#else
#define PE_INVARIANT(err, cond) true
#endif

// NaN among the elements of a 16-byte vector (exponent all ones, mantissa
// not zero), by the bit patterns of the formats.
__device__ __forceinline__ bool bf16x8_has_nan(uint4 q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  bool n = false;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    n |= (w[i] & 0x7fffu) > 0x7f80u || ((w[i] >> 16) & 0x7fffu) > 0x7f80u;
  return n;
}
__device__ __forceinline__ bool f32x4_has_nan(uint4 q) {
  return (q.x & 0x7fffffffu) > 0x7f800000u || (q.y & 0x7fffffffu) > 0x7f800000u ||
         (q.z & 0x7fffffffu) > 0x7f800000u || (q.w & 0x7fffffffu) > 0x7f800000u;
}

// ------------------------------------------------------------------ KV slots
// Paged-KV slot of a kept position; -1 (and an error bit) outside the table.
__device__ __forceinline__ long long kv_slot(const int32_t* block_table,
                                             int bt_width, int block_size, int b,
                                             int pos, uint32_t* err) {
  if (pos < 0 || pos / block_size >= bt_width) {
    atomicOr(err, PE_ERR_BLOCK_RANGE);
    return -1;
  }
  long long blk = __ldg(block_table + (long long)b * bt_width + pos / block_size);
  return blk * block_size + pos % block_size;
}

// True in every thread of the CTA when in_offsets is a valid partition of R
// rows into B segments of at least min_rows rows each.
__device__ __forceinline__ bool offsets_valid(const int32_t* io, int B, int R,
                                              int min_rows) {
  int bad = 0;
  for (int b = threadIdx.x; b <= B; b += blockDim.x) {
    int v = __ldg(io + b);
    if (b == 0 && v != 0) bad = 1;
    if (b == B && v != R) bad = 1;
    if (b < B && __ldg(io + b + 1) - v < min_rows) bad = 1;
  }
  return !__syncthreads_or(bad);
}

}  // namespace pe

// ------------------------------------------------------------------ host side
namespace pe_host {

struct DeviceInfo {
  int sm_count;
};
// SM count of the current device (cached per device; no synchronisation).
int device_info(DeviceInfo* out);

struct Tuning {
  int ctas_per_sm;
  int chunk_batches;
  int rows_per_unit;
  int variant;
  int queue_order;
  int early_full_read_mb;
  int single_pass;
};
Tuning tuning();

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline int elt_size(int dtype) { return dtype == PE_F32 ? 4 : dtype == PE_BF16 ? 2 : 0; }
inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? PE_OK : PE_ECUDA;
}

// Dynamic shared memory above 48 KiB must be opted into once per kernel and
// device (a host-side attribute; no synchronisation).  The carveout is left
// to the driver: asking for the largest shared-memory share measured slower
// (the argmax loads land in L1, whose size bounds the bytes in flight).
template <class K>
bool allow_smem(K kernel, int bytes, std::atomic<unsigned long long>& done_mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const unsigned long long bit = 1ull << dev;
  if (done_mask.load(std::memory_order_relaxed) & bit) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  done_mask.fetch_or(bit);
  return true;
}

}  // namespace pe_host
