// Row argmax building blocks shared by the fused step's kernels: element
// access for the two logits types and one thread's scan of its share of a
// logits row (16-byte loads, kVecPerThread in flight, first occurrence of
// the maximum kept), reduced into a packed (value, column) key.
#pragma once

#include "pe_internal.cuh"

namespace pe {

// ------------------------------------------------------------ element types
template <int DT>
struct Elem;

template <>
struct Elem<PE_BF16> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ bool has_nan(uint4 q) { return bf16x8_has_nan(q); }
  __device__ static __forceinline__ uint4 neg_inf() {
    return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  }
  // max of the 8 elements of a vector (exact: max returns one of its inputs)
  __device__ static __forceinline__ float vmax(uint4 q) {
    const uint32_t w = bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w));
    return fmaxf(bf16_lo(w), bf16_hi(w));
  }
  // lowest element of q equal to v (v is known to occur in q)
  __device__ static __forceinline__ int first_equal(uint4 q, float v) {
    int e = 7;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 3; i >= 0; --i) {
      if (bf16_hi(w[i]) == v) e = 2 * i + 1;
      if (bf16_lo(w[i]) == v) e = 2 * i;
    }
    return e;
  }
  __device__ static __forceinline__ float scalar(const char* row, int col) {
    uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(row) + col);
    return __uint_as_float(((uint32_t)h) << 16);
  }
};

template <>
struct Elem<PE_F32> {
  static constexpr int kPerVec = 4;
  __device__ static __forceinline__ bool has_nan(uint4 q) { return f32x4_has_nan(q); }
  __device__ static __forceinline__ uint4 neg_inf() {
    return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
  }
  __device__ static __forceinline__ float vmax(uint4 q) {
    return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                 fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
  }
  __device__ static __forceinline__ int first_equal(uint4 q, float v) {
    int e = 3;
    if (__uint_as_float(q.z) == v) e = 2;
    if (__uint_as_float(q.y) == v) e = 1;
    if (__uint_as_float(q.x) == v) e = 0;
    return e;
  }
  __device__ static __forceinline__ float scalar(const char* row, int col) {
    return __ldg(reinterpret_cast<const float*>(row) + col);
  }
};

// Key (value, first column) of this thread's elements of vectors
// [v_lo, v_hi) of one logits row.  Elements are visited in increasing column
// order (batch, then vector i, then element), so a strict '>' keeps the
// first occurrence.
// Checked build: a NaN among the elements read raises PE_ERR_NAN in *err.
template <int DT, int NT>
__device__ __forceinline__ unsigned long long thread_key(const uint4* row, int v_lo, int v_hi,
                                                         uint32_t* err) {
  using E = Elem<DT>;
  const int tid = threadIdx.x;
  float m = 0.f;
  int col = -1;
#ifdef PE_CHECKED
  bool nan = false;
#endif
  for (int base = v_lo; base < v_hi; base += NT * kVecPerThread) {
    if (base + tid >= v_hi) break;  // this thread has no vector here or later
    uint4 x[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int v = base + i * NT + tid;
      x[i] = v < v_hi ? __ldcs(row + v) : E::neg_inf();
    }
#ifdef PE_CHECKED
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) nan |= E::has_nan(x[i]);
#endif
    float vm[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) vm[i] = E::vmax(x[i]);
    float gm = vm[0];
#pragma unroll
    for (int i = 1; i < kVecPerThread; ++i) gm = fmaxf(gm, vm[i]);
    if (col < 0 || gm > m) {
      // locate the first vector, then the first element, holding gm
      uint4 q = x[kVecPerThread - 1];
      int vi = kVecPerThread - 1;
#pragma unroll
      for (int i = kVecPerThread - 2; i >= 0; --i)
        if (vm[i] == gm) {
          q = x[i];
          vi = i;
        }
      m = gm;
      col = (base + vi * NT + tid) * E::kPerVec + E::first_equal(q, gm);
    }
  }
#ifdef PE_CHECKED
  if (nan) atomicOr(err, PE_ERR_NAN);
#else
  (void)err;
#endif
  return col >= 0 ? make_key(m, (uint32_t)col) : 0ull;
}

// Key of the leftover elements of a row past its last whole vector
// (columns nvec*kPerVec .. +tail-1; tail >= 1), scanned by one thread in
// column order.  Checked build: a NaN among them raises PE_ERR_NAN.
template <int DT>
__device__ __forceinline__ unsigned long long tail_key(const char* rowp, int nvec, int tail,
                                                       uint32_t* err) {
  using E = Elem<DT>;
  const int c0 = nvec * E::kPerVec;
  float tm = E::scalar(rowp, c0);
  int tc = c0;
#ifdef PE_CHECKED
  bool nan = tm != tm;
#endif
  for (int e = 1; e < tail; ++e) {
    const float x = E::scalar(rowp, c0 + e);
#ifdef PE_CHECKED
    nan |= x != x;
#endif
    if (x > tm) {
      tm = x;
      tc = c0 + e;
    }
  }
#ifdef PE_CHECKED
  if (nan) atomicOr(err, PE_ERR_NAN);
#else
  (void)err;
#endif
  return make_key(tm, (uint32_t)tc);
}

}  // namespace pe
