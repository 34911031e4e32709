// Rejection-sampling verification (pe_verify_sampled): the acceptance rule
// of speculative sampling, for callers that draw instead of taking argmax.
//
// Source: "并行草稿机制解析：从P-EAGLE到DSpark的投机采样加速" §1.2 -- the target
// checks drafts one by one against its own distribution, accepts when they
// agree well enough, otherwise replaces from that position with its own
// output, so that the result keeps the target's distribution.  Read as the
// standard rule: accept draft x with probability min(1, p(x)/q(x)); at the
// first rejection draw from the normalised max(0, p - q); when every draft
// is accepted draw the bonus from p of the last verified row.
//
// Two launches on the caller's stream:
//  1. stats: every target row and every draft row is streamed once in
//     chunks; each chunk yields a (max, sum of 2^(y - max)) pair of its
//     logits in the log2 domain (y = logit * log2(e) / T), merged in chunk
//     order by the chunk that completes the row, which also evaluates p(x)
//     or q(x) of the row's draft token.  The last row of a request decides
//     its accepted length.  For the bonus row of every request the same pass
//     also draws the Gumbel-max sample of softmax(row / T), used when every
//     draft is accepted.
//  2. residual: for requests with a rejection, the chunks of their target
//     and draft rows at the rejected position are streamed again to draw from
//     max(0, p - q) (and, should that be empty, from p).
// Everything is compared in the log2 domain: argmax of y(v) + G(v) log2(e)
// is argmax of logit(v) / T + G(v), and G(v) log2(e) = -log2(E(v)) with
// E = -ln U (computed as -log2 U, a constant multiple).  Draws use U from Philox4x32-10 (Salmon et al., SC'11),
// counter (v / 4, request, 0, 0), key = the seed's two words.
#include "pe_internal.cuh"

namespace pe {

constexpr int kMaxChunksSampled = 32;  // warp units per row (partial stats slots)
constexpr int kStatsChunkVecs = 1024;  // vectors per stats unit (16 KB), at least
constexpr int kResidChunkVecs = 256;   // vectors per residual unit and row (4 KB)
constexpr float kLog2e = 1.4426950408889634f;

struct SampledParams {
  int B, Kp, V, nvec, tail, C, chunk_vecs, Rt, Rd, C2, chunk2_vecs;
  float c2;                   // log2(e) / temperature
  uint32_t rk0[10], rk1[10];  // Philox round keys (key + r * Weyl constants)
  long long t_row_bytes, d_row_bytes;
  const void* tlogits;
  const void* dlogits;
  const int32_t* tokens;
  const float* u_accept;
  int32_t* accepted_len;
  int32_t* bonus_token;
  uint32_t* err;
  // workspace
  uint32_t* sched;            // [3] residual warps done; [4] requests listed for a
                              // residual draw; [8 + 64 i] stats unit counter i
  unsigned long long* partial;  // [Rt+Rd][kMaxChunksSampled] (max, sum) per chunk,
                                // packed by pack_partial (0: not yet written)
  float* lse;                 // [Rt+Rd] log2 of the row's normaliser (log2 domain)
  float* prob;                // [Rt+Rd] p(x) or q(x) of the row's draft token
  uint32_t* rcount;           // [Rt+Rd] finished chunks per row
  uint32_t* qcount;           // [B] finished rows per request (stats pass)
  uint32_t* dcount;           // [B] finished chunks per request (residual pass)
  int32_t* acc;               // [B] accepted length, for the residual pass
  unsigned long long* gkey;   // [B] Gumbel draw from the bonus row
  unsigned long long* rkey;   // [B] Gumbel draw from the residual
  int32_t* rlist;             // [sched[4]] requests with a rejection, in decision order
};

// ------------------------------------------------------------ Philox4x32-10
// Counter (g, b, 0, 0); the ten round keys come precomputed from the host.
__device__ __forceinline__ uint4 philox(const SampledParams& p, uint32_t g, uint32_t b) {
  uint32_t c0 = g, c1 = b, c2 = 0u, c3 = 0u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long m0 = (unsigned long long)0xD2511F53u * c0;
    const unsigned long long m1 = (unsigned long long)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(m1 >> 32) ^ c1 ^ p.rk0[r];
    const uint32_t n2 = (uint32_t)(m0 >> 32) ^ c3 ^ p.rk1[r];
    c1 = (uint32_t)m1;
    c3 = (uint32_t)m0;
    c0 = n0;
    c2 = n2;
  }
  return make_uint4(c0, c1, c2, c3);
}

// word k (0..3) of a Philox output, without a local-memory array
__device__ __forceinline__ uint32_t word(uint4 w, int k) {
  const uint32_t lo = (k & 1) ? w.y : w.x;
  const uint32_t hi = (k & 1) ? w.w : w.z;
  return (k & 2) ? hi : lo;
}

// Packed fp32 pairs (Blackwell's two-wide FP32 SIMD): (d0, d1) = (a * b + c)
// and (a + b) lane by lane, one instruction for both.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
      "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1) {
  asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "add.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ float ex2(float x) {  // 2^x, subnormal results flushed
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {  // log2 x (approximate)
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Gumbel noise of one Philox word in the log2 domain, up to a constant that
// shifts every score of a draw alike: -log2(E2) with E2 = -log2 U = E log2(e),
// E = -ln U, U = ((w >> 9) + 0.5) / 2^23.  U and t = 1 - U are formed exactly:
// 23 bits (k, and 2^23 - 1 - k) become the mantissa of a float in [1, 2) and
// one exact subtraction shifts it to [2^-24, 1 - 2^-24].  E2 needs a small
// RELATIVE error: below t = 1/64 it is the series log2(e) (t + t^2/2 + ... +
// t^5/5) of -log2(1 - t) (truncation error under t^4/6 relative); above, the
// hardware log2 has absolute error near 2^-22, relative error under 1e-5 of
// an E2 that is then at least 0.0227.
__device__ __forceinline__ float noise2(uint32_t w) {
  constexpr float kOneMinus = 1.0f - 5.9604644775390625e-8f;  // 1 - 2^-24
  const uint32_t k = w >> 9;
  const float u = __uint_as_float(k | 0x3f800000u) - kOneMinus;
  const float t = __uint_as_float((k ^ 0x7fffffu) | 0x3f800000u) - kOneMinus;
  const float series =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kLog2e / 5.f, kLog2e / 4.f), kLog2e / 3.f),
                       kLog2e / 2.f),
               kLog2e);
  const float e2 = t < 0.015625f ? series : -lg2(u);
  return -lg2(e2);
}

// t = 1 - U of one Philox word, exact (see noise2).
__device__ __forceinline__ float one_minus_u(uint32_t w) {
  return __uint_as_float(((w >> 9) ^ 0x7fffffu) | 0x3f800000u) - (1.0f - 5.9604644775390625e-8f);
}

// Pruning bound.  -ln(1 - t) >= t, so E2 = -log2 U >= t log2(e) and a
// column's score y - log2(E2) is at most y - log2(t log2(e)).  With
// e = 2^(y - m) a column can only exceed a threshold thr when
// e > 2^(thr - m) log2(e) t; columns failing that test are skipped without
// computing their noise.  kBound keeps the test conservative by far more
// than the rounding of the quantities it compares.
constexpr float kBound = 1.4426950408889634f * (1.0f - 1.0f / 4096.0f);

// Warp maximum of a float through one integer reduction (redux.sync)
// instead of five shuffles: a float's bits, with the magnitude bits of a
// negative one flipped, order as signed integers the way the floats do (no
// NaN here).  Used once per batch in the draws (237.7 us per B=256 call
// against 239.9 with the shuffles).
__device__ __forceinline__ float warp_max_redux(float x) {
  int i = __float_as_int(x);
  i = i >= 0 ? i : i ^ 0x7fffffff;
  i = __reduce_max_sync(0xffffffffu, i);
  return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff);
}

// ----------------------------------------------------------- element access
template <int DT>
struct Vec;

template <>
struct Vec<PE_BF16> {
  static constexpr int kN = 8;
  static constexpr uint32_t kNegInf = 0xff80ff80u;  // a pair of bf16 -inf
  __device__ static __forceinline__ void unpack(uint4 q, float (&z)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      z[2 * i] = bf16_lo(w[i]);
      z[2 * i + 1] = bf16_hi(w[i]);
    }
  }
  // element e (a compile-time index after unrolling) of a vector
  __device__ static __forceinline__ float elem(uint4 q, int e) {
    const uint32_t w = (e >> 1) == 0 ? q.x : (e >> 1) == 1 ? q.y : (e >> 1) == 2 ? q.z : q.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
  // running maximum of raw values, two at a time
  __device__ static __forceinline__ uint32_t max_init() { return kNegInf; }
  __device__ static __forceinline__ uint32_t max_fold(uint32_t m, uint4 q) {
    return bf16x2_max(m, bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w)));
  }
  __device__ static __forceinline__ float max_value(uint32_t m) {
    return fmaxf(bf16_lo(m), bf16_hi(m));
  }
  __device__ static __forceinline__ float at(const char* row, int col) {
    return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + col))
                           << 16);
  }
};

template <>
struct Vec<PE_F32> {
  static constexpr int kN = 4;
  static constexpr uint32_t kNegInf = 0xff800000u;
  __device__ static __forceinline__ void unpack(uint4 q, float (&z)[4]) {
    z[0] = __uint_as_float(q.x);
    z[1] = __uint_as_float(q.y);
    z[2] = __uint_as_float(q.z);
    z[3] = __uint_as_float(q.w);
  }
  __device__ static __forceinline__ float elem(uint4 q, int e) {
    return __uint_as_float(e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w);
  }
  __device__ static __forceinline__ uint32_t max_init() { return kNegInf; }
  __device__ static __forceinline__ uint32_t max_fold(uint32_t m, uint4 q) {
    const float a = fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                          fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
    return __float_as_uint(fmaxf(__uint_as_float(m), a));
  }
  __device__ static __forceinline__ float max_value(uint32_t m) { return __uint_as_float(m); }
  __device__ static __forceinline__ float at(const char* row, int col) {
    return __ldg(reinterpret_cast<const float*>(row) + col);
  }
};

// (max, sum of 2^(y - max)) of two disjoint sets, merged.
__device__ __forceinline__ float2 combine(float2 a, float2 b) {
  if (a.y == 0.f) return b;
  if (b.y == 0.f) return a;
  const float m = fmaxf(a.x, b.x);
  return make_float2(m, a.y * ex2(a.x - m) + b.y * ex2(b.x - m));
}

__device__ __forceinline__ float2 warp_combine(float2 v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    float2 w;
    w.x = __shfl_xor_sync(0xffffffffu, v.x, o);
    w.y = __shfl_xor_sync(0xffffffffu, v.y, o);
    v = combine(v, w);
  }
  return v;
}

// Per-thread best (value, column): strict > over ascending columns keeps
// the lowest column among equal values.
struct Best {
  float v = -INFINITY;
  int col = 0;
  __device__ __forceinline__ void offer(float x, int c) {
    if (x > v) {
      v = x;
      col = c;
    }
  }
  __device__ __forceinline__ unsigned long long key() const {
    return v == -INFINITY ? 0ull : make_key(v, (uint32_t)col);
  }
};

// Virtual row vr: target rows [0, Rt), then draft rows [Rt, Rt + Rd).
__device__ __forceinline__ const char* vrow_ptr(const SampledParams& p, int vr) {
  return vr < p.Rt ? static_cast<const char*>(p.tlogits) + (long long)vr * p.t_row_bytes
                   : static_cast<const char*>(p.dlogits) + (long long)(vr - p.Rt) * p.d_row_bytes;
}

}  // namespace pe

namespace pe {

// Every unit of work below belongs to ONE warp: a warp takes a unit from the
// dynamic counter, streams it, reduces with shuffles and publishes its
// result with atomics.  No CTA barrier anywhere, so each warp keeps its
// loads in flight regardless of what the other warps of its CTA are doing.

// One row chunk folded into (m, s) = (max, sum of 2^(y - max)) with
// y = logit * c2, and, for the bonus row (DRAW), into the lane's best Gumbel
// score y + G log2(e), pruned by the bound above against the best score of
// the warp (shared after every batch).  Vectors past the chunk read as -inf
// and contribute nothing.  The bonus row takes a quarter of the vectors per
// batch: the noise needs the registers, and with half of them the kernel
// spilled at its 64 registers (248.5 us per B=256 call against 241.2
// without the spill).
template <int DT, bool DRAW>
__device__ __forceinline__ void fold_chunk(const SampledParams& p, const char* rowp, int v_lo,
                                           int v_hi, int b, int lane, float& m, float& s,
                                           Best& best) {
  using E = Vec<DT>;
  constexpr int kV = DRAW ? kVecPerThread / 4 : kVecPerThread;
  const uint4* row = reinterpret_cast<const uint4*>(rowp);
  const uint4 neg = make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
  float thr = -INFINITY;
  for (int base = v_lo; base < v_hi; base += 32 * kV) {
    uint4 x[kV];
    if (base + 32 * kV <= v_hi) {  // a whole batch: no bounds to check
#pragma unroll
      for (int i = 0; i < kV; ++i) x[i] = __ldcs(row + base + i * 32 + lane);
    } else {
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = base + i * 32 + lane;
        x[i] = v < v_hi ? __ldcs(row + v) : neg;
      }
    }
    uint32_t mr = E::max_init();
#pragma unroll
    for (int i = 0; i < kV; ++i) mr = E::max_fold(mr, x[i]);
    const float bm = E::max_value(mr) * p.c2;  // monotone: max of the scaled values
    if (bm > m) {
      s *= ex2(m - bm);
      m = bm;
    }
    if (!DRAW) {  // pairs of elements: two sums, packed arithmetic
      float s1 = 0.f;
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        float z[E::kN];
        E::unpack(x[i], z);
#pragma unroll
        for (int e = 0; e < E::kN; e += 2) {
          float y0, y1;
          fma2(y0, y1, z[e], z[e + 1], p.c2, p.c2, -m, -m);
          add2(s, s1, s, s1, ex2(y0), ex2(y1));
        }
      }
      s += s1;
    } else {
      float K = ex2(thr - m) * kBound;
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = base + i * 32 + lane;
        float z[E::kN];
        E::unpack(x[i], z);
#pragma unroll
        for (int g = 0; g < E::kN / 4; ++g) {
          const uint4 w = philox(p, (uint32_t)((v * E::kN) / 4 + g), (uint32_t)b);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float y = z[4 * g + k] * p.c2;
            const float ev = ex2(y - m);
            s += ev;
            const uint32_t wk = word(w, k);
            if (ev > K * one_minus_u(wk)) {  // may beat the threshold
              const float sc = y + noise2(wk);
              best.offer(sc, v * E::kN + 4 * g + k);
              if (sc > thr) {
                thr = sc;
                K = ex2(thr - m) * kBound;
              }
            }
          }
        }
      }
      thr = warp_max_redux(thr);
    }
  }
}

// A chunk's (max, sum) in one 64-bit word that is never zero, so that zero
// (the workspace's resting state) marks a slot not yet written: the max is
// never NaN (it starts finite and only takes larger values), and its bits
// are stored XOR a quiet-NaN pattern.
constexpr uint32_t kPartialMark = 0x7fc00000u;
constexpr unsigned long long kPollLimitNs = 2000000ull;  // 2 ms per slot before giving up

__device__ __forceinline__ unsigned long long pack_partial(float2 t) {
  return ((unsigned long long)(__float_as_uint(t.x) ^ kPartialMark) << 32) | __float_as_uint(t.y);
}
__device__ __forceinline__ float2 unpack_partial(unsigned long long w) {
  return make_float2(__uint_as_float((uint32_t)(w >> 32) ^ kPartialMark),
                     __uint_as_float((uint32_t)w));
}

// Accepted length of request b from its rows' draft-token probabilities.
// Leaves the workspace zeroed except the normalisers the residual draw of
// this request reads (target and draft row a); that draw clears them.
__device__ __forceinline__ void decide(const SampledParams& p, int b) {
  int a = p.Kp;
  for (int j = 0; j < p.Kp; ++j) {
    const float px = __ldcg(p.prob + b * (p.Kp + 1) + j);
    const float qx = __ldcg(p.prob + p.Rt + b * p.Kp + j);
    if (px < 0.f || !(__ldg(p.u_accept + b * p.Kp + j) * qx < px)) {  // px < 0: bad token
      a = j;
      break;
    }
  }
  p.accepted_len[b] = a;
  if (a < p.Kp) {  // a rejection: list the request for the residual pass
    p.acc[b] = a;  // (the residual draw clears it)
    const unsigned at = atomicAdd(p.sched + 4, 1u);
    if (at < (unsigned)p.B)
      p.rlist[at] = b;
    else  // the list count did not start at zero
      atomicOr(p.err, PE_ERR_WORKSPACE);
  }
  const unsigned long long gk = atomicExch(p.gkey + b, 0ull);
  // the bonus row's draw names a column of the row (a finite row always
  // yields one)
  if (gk == 0ull || key_col(gk) >= (uint32_t)p.V) atomicOr(p.err, PE_ERR_WORKSPACE);
  if (a == p.Kp) p.bonus_token[b] = (int)key_col(gk);  // else the residual pass draws
  for (int j = 0; j <= p.Kp; ++j) {
    const int vt = b * (p.Kp + 1) + j;
    if (j != a || a == p.Kp) p.lse[vt] = 0.f;
    if (j < p.Kp) {
      const int vd = p.Rt + b * p.Kp + j;
      p.prob[vt] = 0.f;
      p.prob[vd] = 0.f;
      if (j != a) p.lse[vd] = 0.f;
    }
  }
}

// The end of a unit (row vr, chunk c): the scalar tail of the row, the
// warp's reduction and its publication.  The warp that completes a row
// merges its partials (lane-strided, then a shuffle tree: a fixed order, so
// the result does not depend on timing), stores the row's log2-normaliser
// and the draft token's probability; the warp that completes a request
// decides its accepted length.
template <int DT>
__device__ __forceinline__ void stats_finish(const SampledParams& p, int vr, int c, int lane,
                                             float m, float s, const Best& best) {
  using E = Vec<DT>;
  int b, j;
  if (vr < p.Rt) {
    b = vr / (p.Kp + 1);
    j = vr - b * (p.Kp + 1);
  } else {
    b = (vr - p.Rt) / p.Kp;
    j = (vr - p.Rt) - b * p.Kp;
  }
  const bool draw = vr < p.Rt && j == p.Kp;  // the bonus row
  const char* rowp = vrow_ptr(p, vr);
  Best bt = best;
  if (p.tail && c == p.C - 1 && lane == 0) {  // elements after the last whole vector
    for (int e = 0; e < p.tail; ++e) {
      const int col = p.nvec * E::kN + e;
      const float y = E::at(rowp, col) * p.c2;
      if (y > m) {
        s *= ex2(m - y);
        m = y;
      }
      s += ex2(y - m);
      if (draw) {
        const uint4 w = philox(p, (uint32_t)(col / 4), (uint32_t)b);
        bt.offer(y + noise2(word(w, col & 3)), col);
      }
    }
  }
  const float2 t = warp_combine(make_float2(m, s));
  const unsigned long long gk = draw ? warp_max_key(bt.key()) : 0ull;
  // The partial goes out without a fence: the warp that completes the row
  // polls each slot until it holds a value.  Only the bonus row's key (an
  // atomicMax elsewhere) needs ordering: its count is an acq_rel atomic,
  // which releases the key and, for the last chunk, acquires the others'
  // (every count here works that way; with fence pairs instead the call
  // took 238.0 us against 234.2).
  int last = 0;
  if (lane == 0) {
    st_relaxed(p.partial + vr * kMaxChunksSampled + c, pack_partial(t));
    unsigned done;
    if (draw) {  // the key merge released with the count, acquired by the last
      atomicMax(p.gkey + b, gk);
      done = atom_add_acq_rel_u32(p.rcount + vr, 1u);
    } else {
      done = atomicAdd(p.rcount + vr, 1u);
    }
    if (done >= (unsigned)p.C) atomicOr(p.err, PE_ERR_WORKSPACE);  // did not start at zero
    last = done == (unsigned)(p.C - 1);
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __syncwarp();  // orders lane 0's acquire before the other lanes' accesses
  float2 acc = make_float2(-3.0e38f, 0.f);
  for (int cc = lane; cc < p.C; cc += 32) {
    unsigned long long* slot = p.partial + vr * kMaxChunksSampled + cc;
    unsigned long long w = ld_relaxed(slot);
    if (w == 0ull) {
      const unsigned long long t0 = global_ns();
      while (w == 0ull && global_ns() - t0 < kPollLimitNs) w = ld_relaxed(slot);
    }
    if (w == 0ull)
      atomicOr(p.err, PE_ERR_TIMEOUT);  // never expected: the chunk was counted
    else
      acc = combine(acc, unpack_partial(w));
    *slot = 0ull;
  }
  acc = warp_combine(acc);
  if (lane == 0) {
    p.rcount[vr] = 0u;
    const float L = acc.x + log2f(acc.y);  // log2 of the sum of 2^y
    p.lse[vr] = L;
    if (!draw) {  // probability of the row's draft token
      const int x = __ldg(p.tokens + b * (p.Kp + 1) + j + 1);
      p.prob[vr] = (x >= 0 && x < p.V) ? ex2(E::at(rowp, x) * p.c2 - L) : -1.f;
    }
    const unsigned rows_done = atom_add_acq_rel_u32(p.qcount + b, 1u);
    if (rows_done > (unsigned)(2 * p.Kp)) atomicOr(p.err, PE_ERR_WORKSPACE);
    if (rows_done == (unsigned)(2 * p.Kp)) {  // all 2Kp+1 rows
      p.qcount[b] = 0u;
      decide(p, b);
    }
  }
}

// Stats of one warp unit u = row * C + chunk.
template <int DT>
__device__ __forceinline__ void stats_unit(const SampledParams& p, int u, int lane) {
  const int vr = u / p.C;
  const int c = u - vr * p.C;
  const int b = vr < p.Rt ? vr / (p.Kp + 1) : (vr - p.Rt) / p.Kp;
  const bool draw = vr < p.Rt && vr - b * (p.Kp + 1) == p.Kp;  // the bonus row
  const char* rowp = vrow_ptr(p, vr);
  const int v_lo = c * p.chunk_vecs;
  const int v_hi = min(v_lo + p.chunk_vecs, p.nvec);
  float m = -3.0e38f, s = 0.f;  // finite: an empty lane never forms -inf + inf
  Best best;
  if (draw) fold_chunk<DT, true>(p, rowp, v_lo, v_hi, b, lane, m, s, best);
  else fold_chunk<DT, false>(p, rowp, v_lo, v_hi, b, lane, m, s, best);
  stats_finish<DT>(p, vr, c, lane, m, s, best);
}

// Persistent warps over dynamic unit counters; the next unit is fetched
// before the current one is processed.  Counter i (kStatsCounters of them,
// 256 bytes apart in the workspace) hands out units i, i + k, i + 2k, ...,
// so each counter word takes half the claims: one word for all ~4900 warps
// measured slower on some GPUs (its atomics queue).  A warp draws from its
// own counter, then from the other, each until it runs out, so every warp
// makes exactly one failing claim on every counter, and the claim that
// returns a counter's last position (its units plus one per warp) resets it.
constexpr int kStatsCtasPerSm = 4;  // 32 warps per SM: 64 registers a thread
constexpr int kStatsCounters = 2;
constexpr int kCounterWords = 64;   // words between counters

__device__ __forceinline__ uint32_t* stats_counter(const SampledParams& p, int i) {
  return p.sched + 8 + i * kCounterWords;
}

// Next unit for this warp (lane 0), or n_units once every counter ran out.
// A counter hands out its n_i units and then one failing claim per warp, so
// a value above n_i + warps - 1 means it did not start at zero.
__device__ __forceinline__ int stats_next(const SampledParams& p, int n_units, int& ci,
                                          int& ndone) {
  while (ndone < kStatsCounters) {
    const int n_i = (n_units - ci + kStatsCounters - 1) / kStatsCounters;
    uint32_t* ctr = stats_counter(p, ci);
    const unsigned v = atomicAdd(ctr, 1u);
    const unsigned last = (unsigned)n_i + gridDim.x * kWarps - 1u;
    if (v == last) atomicExch(ctr, 0u);
    if (v > last) atomicOr(p.err, PE_ERR_WORKSPACE);
    if (v < (unsigned)n_i) return ci + (int)v * kStatsCounters;
    ++ndone;
    ci = ci + 1 == kStatsCounters ? 0 : ci + 1;
  }
  return n_units;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, kStatsCtasPerSm) sampled_stats_kernel(
    const SampledParams p) {
  const int lane = threadIdx.x & 31;
  const int n_units = (p.Rt + p.Rd) * p.C;
  int ci = (blockIdx.x * kWarps + (threadIdx.x >> 5)) % kStatsCounters, ndone = 0;
  int u = 0;
  if (lane == 0) u = stats_next(p, n_units, ci, ndone);
  u = __shfl_sync(0xffffffffu, u, 0);
  while (u < n_units) {
    int next = 0;
    if (lane == 0) next = stats_next(p, n_units, ci, ndone);
    stats_unit<DT>(p, u, lane);
    u = __shfl_sync(0xffffffffu, next, 0);
  }
  // this warp is done: the residual launch may start as SMs free up
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Residual draw of request b, chunk c (u = b * C2 + c; only listed requests,
// which all have a rejection, get units): Gumbel-max
// over log2 max(0, p - q) with p = 2^(y_t - L_t), q = 2^(y_d - L_d).  The
// warp that completes the request publishes the draw; should the residual be
// empty (p == q everywhere, possible only for identical rows) that warp
// draws from p over the whole target row instead.
template <int DT>
__device__ __forceinline__ void residual_unit(const SampledParams& p, int u, int lane) {
  using E = Vec<DT>;
  const int b = u / p.C2;
  const int c = u - b * p.C2;
  int a = __ldcg(p.acc + b);
  if (a < 0 || a >= p.Kp) {  // a listed request has a rejection at a < K'
    if (c == 0) atomicOr(p.err, PE_ERR_WORKSPACE);
    a = p.Kp;  // nothing to draw
  }
  const bool draw = a < p.Kp;
  const int vt = b * (p.Kp + 1) + a;
  const int vd = p.Rt + b * p.Kp + a;
  Best best;
  if (draw) {
    const float Lt = __ldcg(p.lse + vt);
    const float Ld = __ldcg(p.lse + vd);
    const char* trow = vrow_ptr(p, vt);
    const char* drow = vrow_ptr(p, vd);
    const uint4* tr = reinterpret_cast<const uint4*>(trow);
    const uint4* dr = reinterpret_cast<const uint4*>(drow);
    const int v_lo = c * p.chunk2_vecs;
    const int v_hi = min(v_lo + p.chunk2_vecs, p.nvec);
    // one vector of each row per batch: with two the kernel spilled at its
    // 64 registers (241.2 us per B=256 call against 239.3 without)
    constexpr int kV = kVecPerThread / 8;
    float thr = -INFINITY;  // best score of the warp so far (absolute log2 units)
    for (int base = v_lo; base < v_hi; base += 32 * kV) {
      const float K = ex2(thr) * kBound;  // d > K t: the column may beat thr
      const bool whole = base + 32 * kV <= v_hi;  // no bounds to check
      uint4 xt[kV], xd[kV];
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = base + i * 32 + lane;
        xt[i] = (whole || v < v_hi) ? __ldcs(tr + v) : make_uint4(0u, 0u, 0u, 0u);
        xd[i] = (whole || v < v_hi) ? __ldcs(dr + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = base + i * 32 + lane;
        if (!whole && v >= v_hi) continue;
#pragma unroll
        for (int g = 0; g < E::kN / 4; ++g) {
          const uint4 w = philox(p, (uint32_t)((v * E::kN) / 4 + g), (uint32_t)b);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = 4 * g + k;
            float at, ad;  // exponents of p and q, one packed instruction
            fma2(at, ad, E::elem(xt[i], e), E::elem(xd[i], e), p.c2, p.c2, -Lt, -Ld);
            const float d = ex2(at) - ex2(ad);
            const uint32_t wk = word(w, k);
            if (d > K * one_minus_u(wk)) {  // d > 0 and the column may beat thr
              const float sc = lg2(d) + noise2(wk);
              best.offer(sc, v * E::kN + e);
              thr = fmaxf(thr, sc);
            }
          }
        }
      }
      thr = warp_max_redux(thr);
    }
    if (p.tail && c == p.C2 - 1 && lane == 0) {
      for (int e = 0; e < p.tail; ++e) {
        const int col = p.nvec * E::kN + e;
        const float d = ex2(fmaf(E::at(trow, col), p.c2, -Lt)) -
                        ex2(fmaf(E::at(drow, col), p.c2, -Ld));
        if (d > 0.f) {
          const uint4 w = philox(p, (uint32_t)(col / 4), (uint32_t)b);
          best.offer(lg2(d) + noise2(word(w, col & 3)), col);
        }
      }
    }
  }
  const unsigned long long k = warp_max_key(best.key());
  int last = 0;
  if (lane == 0) {
    if (draw) atomicMax(p.rkey + b, k);
    const unsigned done = atom_add_acq_rel_u32(p.dcount + b, 1u);
    if (done >= (unsigned)p.C2) atomicOr(p.err, PE_ERR_WORKSPACE);  // did not start at zero
    last = done == (unsigned)(p.C2 - 1);  // every unit of b is done
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __syncwarp();
  int fallback = 0;
  if (lane == 0) {
    p.dcount[b] = 0u;
    p.acc[b] = 0;
    if (draw) {
      const unsigned long long r = atomicExch(p.rkey + b, 0ull);
      if (r && key_col(r) >= (uint32_t)p.V) atomicOr(p.err, PE_ERR_WORKSPACE);
      if (r) p.bonus_token[b] = (int)key_col(r);
      else fallback = 1;
      p.lse[vt] = 0.f;
      p.lse[vd] = 0.f;
    }
  }
  if (__shfl_sync(0xffffffffu, fallback, 0)) {  // empty residual: draw from p (rare)
    const char* trow = vrow_ptr(p, vt);
    Best bp;
    for (int col = lane; col < p.V; col += 32) {
      const uint4 w = philox(p, (uint32_t)(col / 4), (uint32_t)b);
      bp.offer(E::at(trow, col) * p.c2 + noise2(word(w, col & 3)), col);
    }
    const unsigned long long kf = warp_max_key(bp.key());
    if (lane == 0) p.bonus_token[b] = (int)key_col(kf);
  }
}

// Persistent warps over the residual units of the listed requests, handed
// out statically (warp w takes units w, w + warps, ...: the units are all
// the same size, so a work counter would only add same-address atomics);
// the list is complete, the stats pass having finished.  The last warp to
// leave (sched[3]: warps done) clears the list and the counter words.
template <int DT>
__global__ void __launch_bounds__(kThreads, 4) sampled_residual_kernel(const SampledParams p) {
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kWarps + (threadIdx.x >> 5);
  // Launched as a programmatic dependent of the stats pass: wait until that
  // grid has finished and its writes are visible (a no-op for a plain
  // launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // at most B requests are listed; more means the count did not start at
  // zero (every warp reads the same value, one warp reports it)
  unsigned listed = __ldcg(p.sched + 4);
  if (listed > (unsigned)p.B) {
    if (warp == 0 && lane == 0) atomicOr(p.err, PE_ERR_WORKSPACE);
    listed = (unsigned)p.B;
  }
  const int n_units = (int)listed * p.C2;
  const int nw = gridDim.x * kWarps;
  for (int u = warp; u < n_units; u += nw) {
    const int k = u / p.C2;
    const int b = __ldcg(p.rlist + k);
    if (b < 0 || b >= p.B) {  // an entry this call did not write
      if (lane == 0 && u == k * p.C2) atomicOr(p.err, PE_ERR_WORKSPACE);
      continue;
    }
    residual_unit<DT>(p, b * p.C2 + (u - k * p.C2), lane);
  }
  if (lane == 0) {
    const unsigned left = atom_add_acq_rel_u32(p.sched + 3, 1u);
    if (left > gridDim.x * kWarps - 1u) atomicOr(p.err, PE_ERR_WORKSPACE);
    if (left == gridDim.x * kWarps - 1u) {  // every other warp has left
      for (unsigned k = 0; k < listed; ++k) p.rlist[k] = 0;
      atomicExch(p.sched + 3, 0u);
      atomicExch(p.sched + 4, 0u);
    }
  }
}

}  // namespace pe

// ---------------------------------------------------------------- host side
namespace {

struct SampledLayout {
  size_t partial_off, lse_off, prob_off, rcount_off, qcount_off, dcount_off, acc_off, gkey_off,
      rkey_off, rlist_off, bytes;
  SampledLayout(long long B, long long Kp) {
    const long long rows = B * (Kp + 1) + B * Kp;
    // eight scheduler words, then the stats counters 256 bytes apart
    size_t o = 32 + 4 * pe::kCounterWords * pe::kStatsCounters;
    auto take = [&](size_t n, size_t align) {
      o = (o + align - 1) / align * align;
      const size_t at = o;
      o += n;
      return at;
    };
    partial_off = take(8 * rows * pe::kMaxChunksSampled, 16);
    lse_off = take(4 * rows, 16);
    prob_off = take(4 * rows, 16);
    rcount_off = take(4 * rows, 16);
    qcount_off = take(4 * B, 16);
    dcount_off = take(4 * B, 16);
    acc_off = take(4 * B, 16);
    gkey_off = take(8 * B, 16);
    rkey_off = take(8 * B, 16);
    rlist_off = take(4 * B, 16);
    bytes = (o + 255) / 256 * 256;
  }
};

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

}  // namespace

extern "C" {

size_t pe_workspace_bytes_sampled(int32_t B, int32_t Kp) {
  if (B < 0 || Kp < 0) return 0;
  return SampledLayout(B, Kp).bytes;
}

int pe_verify_sampled(const void* target_logits, const void* draft_logits, int dtype,
                      int64_t target_stride, int64_t draft_stride, int32_t B, int32_t Kp,
                      int32_t V, const int32_t* in_tokens, const float* u_accept,
                      float temperature, uint64_t seed, int32_t* accepted_len,
                      int32_t* bonus_token, void* workspace, uint32_t* err, void* stream) {
  const int elt = pe_host::elt_size(dtype);
  if (!elt) return PE_EDTYPE;
  if (B < 0 || Kp < 0 || Kp > PE_MAX_KP || V < 1 || !(temperature > 0.f)) return PE_EINVAL;
  if (B == 0) return PE_OK;
  if (!target_logits || !accepted_len || !bonus_token || !workspace || !err) return PE_EINVAL;
  if (Kp > 0 && (!draft_logits || !in_tokens || !u_accept)) return PE_EINVAL;
  if (target_stride < V || (Kp > 0 && draft_stride < V)) return PE_EINVAL;
  if (!pe_host::aligned16(target_logits) || !pe_host::aligned16(workspace) ||
      (target_stride * elt) % 16 ||
      (Kp > 0 && (!pe_host::aligned16(draft_logits) || (draft_stride * elt) % 16)))
    return PE_EALIGN;
  const long long rows = (long long)B * (Kp + 1) + (long long)B * Kp;
  if (rows * pe::kMaxChunksSampled > 0x7fffffffLL) return PE_EINVAL;
  const float c2 = pe::kLog2e / temperature;
  if (!(c2 < 3.0e38f)) return PE_EINVAL;  // temperature so small that 1/T overflows
  pe_host::DeviceInfo dev;
  if (pe_host::device_info(&dev) != PE_OK) return PE_ECUDA;

  pe::SampledParams p = {};
  p.B = B;
  p.Kp = Kp;
  p.V = V;
  const int epv = 16 / elt;
  p.nvec = V / epv;
  p.tail = V % epv;
  p.Rt = B * (Kp + 1);
  p.Rd = B * Kp;
  // stats units: at least kStatsChunkVecs vectors, at most kMaxChunksSampled
  // per row; residual units: kResidChunkVecs vectors of each of two rows
  int C = 1, C2 = 1;
  if (p.nvec > 0) {
    p.chunk_vecs = ceil_div(p.nvec, pe::kMaxChunksSampled);
    if (p.chunk_vecs < pe::kStatsChunkVecs) p.chunk_vecs = pe::kStatsChunkVecs;
    if (p.chunk_vecs > p.nvec) p.chunk_vecs = p.nvec;
    C = ceil_div(p.nvec, p.chunk_vecs);
    p.chunk2_vecs = p.nvec < pe::kResidChunkVecs ? p.nvec : pe::kResidChunkVecs;
    C2 = ceil_div(p.nvec, p.chunk2_vecs);
  }
  p.C = C;
  p.C2 = C2;
  if ((long long)B * C2 > 0x7fffffffLL || rows * C > 0x7fffffffLL) return PE_EINVAL;
  p.c2 = c2;
  const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {  // Philox key schedule: Weyl sequence
    p.rk0[r] = k0 + (uint32_t)r * 0x9E3779B9u;
    p.rk1[r] = k1 + (uint32_t)r * 0xBB67AE85u;
  }
  p.t_row_bytes = target_stride * elt;
  p.d_row_bytes = draft_stride * elt;
  p.tlogits = target_logits;
  p.dlogits = draft_logits;
  p.tokens = in_tokens;
  p.u_accept = u_accept;
  p.accepted_len = accepted_len;
  p.bonus_token = bonus_token;
  p.err = err;
  const SampledLayout L(B, Kp);
  char* w = static_cast<char*>(workspace);
  p.sched = reinterpret_cast<uint32_t*>(w);
  p.partial = reinterpret_cast<unsigned long long*>(w + L.partial_off);
  p.lse = reinterpret_cast<float*>(w + L.lse_off);
  p.prob = reinterpret_cast<float*>(w + L.prob_off);
  p.rcount = reinterpret_cast<uint32_t*>(w + L.rcount_off);
  p.qcount = reinterpret_cast<uint32_t*>(w + L.qcount_off);
  p.dcount = reinterpret_cast<uint32_t*>(w + L.dcount_off);
  p.acc = reinterpret_cast<int32_t*>(w + L.acc_off);
  p.gkey = reinterpret_cast<unsigned long long*>(w + L.gkey_off);
  p.rkey = reinterpret_cast<unsigned long long*>(w + L.rkey_off);
  p.rlist = reinterpret_cast<int32_t*>(w + L.rlist_off);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // persistent grids: kStatsCtasPerSm CTAs (32 warps) per SM, fewer for small problems
  const long long n1 = ceil_div(rows * p.C, pe::kWarps);
  const int g1_max = dev.sm_count * pe::kStatsCtasPerSm;
  const int g1 = n1 < g1_max ? (int)n1 : g1_max;
  const long long n2 = ceil_div((long long)B * p.C2, pe::kWarps);
  const int g2 = n2 < g1_max ? (int)n2 : g1_max;
  if (dtype == PE_BF16)
    pe::sampled_stats_kernel<PE_BF16><<<g1, pe::kThreads, 0, st>>>(p);
  else
    pe::sampled_stats_kernel<PE_F32><<<g1, pe::kThreads, 0, st>>>(p);
  // The residual pass as a programmatic dependent launch: its CTAs may be
  // scheduled while the stats pass drains and wait in the kernel for it
  // (237.3 us per B=256 call against 238.4 with a plain launch).  Should the
  // runtime refuse that form, the plain launch follows the stats pass.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(g2);
  cfg.blockDim = dim3(pe::kThreads);
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const cudaError_t rc = dtype == PE_BF16
                             ? cudaLaunchKernelEx(&cfg, pe::sampled_residual_kernel<PE_BF16>, p)
                             : cudaLaunchKernelEx(&cfg, pe::sampled_residual_kernel<PE_F32>, p);
  if (rc != cudaSuccess) {
    (void)cudaGetLastError();
    if (dtype == PE_BF16)
      pe::sampled_residual_kernel<PE_BF16><<<g2, pe::kThreads, 0, st>>>(p);
    else
      pe::sampled_residual_kernel<PE_F32><<<g2, pe::kThreads, 0, st>>>(p);
  }
  return pe_host::launch_status();
}

}  // extern "C"
