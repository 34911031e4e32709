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
// E = -ln U.  Draws use U from Philox4x32-10 (Salmon et al., SC'11),
// counter (v / 4, request, 0, 0), key = the seed's two words.
#include "pe_internal.cuh"

namespace pe {

constexpr int kMaxChunksSampled = 16;  // chunks per row (partial stats slots)
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
  uint32_t* sched;            // [4] stats: unit counter, CTAs done; residual: same
  float2* partial;            // [Rt+Rd][kMaxChunksSampled] (max, sum) per chunk
  float* lse;                 // [Rt+Rd] log2 of the row's normaliser (log2 domain)
  float* prob;                // [Rt+Rd] p(x) or q(x) of the row's draft token
  uint32_t* rcount;           // [Rt+Rd] finished chunks per row
  uint32_t* qcount;           // [B] finished rows per request (stats pass)
  uint32_t* dcount;           // [B] finished chunks per request (residual pass)
  int32_t* acc;               // [B] accepted length, for the residual pass
  unsigned long long* gkey;   // [B] Gumbel draw from the bonus row
  unsigned long long* rkey;   // [B] Gumbel draw from the residual
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

// Gumbel noise of one Philox word in the log2 domain: G log2(e) = -log2(E),
// E = -ln U, U = ((w >> 9) + 0.5) / 2^23.  U is formed exactly: the 23 bits
// become the mantissa of a float in [1, 2) and one subtraction (exact, the
// result needs 24 significant bits) shifts it to [2^-24, 1 - 2^-24].  The
// inner logarithm is CUDA's logf, accurate near U = 1 where E is tiny.
__device__ __forceinline__ float noise2(uint32_t w) {
  const float f = __uint_as_float((w >> 9) | 0x3f800000u);
  const float u = f - (1.0f - 5.9604644775390625e-8f);  // (k + 0.5) / 2^23
  return -lg2(-logf(u));
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

struct SampledShared {
  float2 red[kWarps];
  unsigned long long kred[kWarps];
  int unit;
  int acc;
  int fallback;
};

// Virtual row vr: target rows [0, Rt), then draft rows [Rt, Rt + Rd).
__device__ __forceinline__ const char* vrow_ptr(const SampledParams& p, int vr) {
  return vr < p.Rt ? static_cast<const char*>(p.tlogits) + (long long)vr * p.t_row_bytes
                   : static_cast<const char*>(p.dlogits) + (long long)(vr - p.Rt) * p.d_row_bytes;
}

// Block-wide maximum key; valid in thread 0.
__device__ __forceinline__ unsigned long long block_max_key(SampledShared& sh,
                                                            unsigned long long k) {
  const int tid = threadIdx.x;
  k = warp_max_key(k);
  if ((tid & 31) == 0) sh.kred[tid >> 5] = k;
  __syncthreads();
  if (tid < 32) {
    k = tid < kWarps ? sh.kred[tid] : 0ull;
    k = warp_max_key(k);
  }
  __syncthreads();
  return k;
}

}  // namespace pe

namespace pe {

// One row chunk folded into (m, s) = (max, sum of 2^(y - max)) with
// y = logit * c2, and, for the bonus row (draw), into the thread's best
// Gumbel score y + G log2(e).  Vectors past the chunk read as -inf.
template <int DT>
__device__ __forceinline__ void fold_chunk(const SampledParams& p, const char* rowp, int v_lo,
                                           int v_hi, bool tail, bool draw, int b, float& m,
                                           float& s, Best& best) {
  using E = Vec<DT>;
  const int tid = threadIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(rowp);
  const uint4 neg = make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
  for (int base = v_lo; base < v_hi; base += kBatchVecs) {
    if (base + tid >= v_hi) break;
    uint4 x[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int v = base + i * kThreads + tid;
      x[i] = v < v_hi ? __ldcs(row + v) : neg;
    }
    uint32_t mr = E::max_init();
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) mr = E::max_fold(mr, x[i]);
    const float bm = E::max_value(mr) * p.c2;  // monotone: max of the scaled values
    if (bm > m) {
      s *= ex2(m - bm);
      m = bm;
    }
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      float z[E::kN];
      E::unpack(x[i], z);
#pragma unroll
      for (int e = 0; e < E::kN; ++e) s += ex2(fmaf(z[e], p.c2, -m));
    }
    if (draw) {
#pragma unroll
      for (int i = 0; i < kVecPerThread; ++i) {
        const int v = base + i * kThreads + tid;
        if (v >= v_hi) continue;
        float z[E::kN];
        E::unpack(x[i], z);
#pragma unroll
        for (int g = 0; g < E::kN / 4; ++g) {
          const uint4 w = philox(p, (uint32_t)((v * E::kN) / 4 + g), (uint32_t)b);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            best.offer(z[4 * g + k] * p.c2 + noise2(ws[k]), v * E::kN + 4 * g + k);
        }
      }
    }
  }
  if (tail && tid == 0) {  // elements after the last whole vector
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
        best.offer(y + noise2(word(w, col & 3)), col);
      }
    }
  }
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
  p.acc[b] = a;
  const unsigned long long gk = atomicExch(p.gkey + b, 0ull);
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

template <int DT>
__device__ __forceinline__ void stats_unit(const SampledParams& p, SampledShared& sh, int u) {
  using E = Vec<DT>;
  const int tid = threadIdx.x;
  const int vr = u / p.C;
  const int c = u - vr * p.C;
  int b, j;
  if (vr < p.Rt) {
    b = vr / (p.Kp + 1);
    j = vr - b * (p.Kp + 1);
  } else {
    b = (vr - p.Rt) / p.Kp;
    j = -1;  // draft row
  }
  const bool draw = j == p.Kp;  // the bonus row
  const char* rowp = vrow_ptr(p, vr);
  const int v_lo = c * p.chunk_vecs;
  const int v_hi = min(v_lo + p.chunk_vecs, p.nvec);
  float m = -INFINITY, s = 0.f;
  Best best;
  fold_chunk<DT>(p, rowp, v_lo, v_hi, p.tail && c == p.C - 1, draw, b, m, s, best);

  const float2 st = warp_combine(make_float2(m, s));
  if ((tid & 31) == 0) sh.red[tid >> 5] = st;
  unsigned long long gk = 0ull;
  if (draw) gk = block_max_key(sh, best.key());  // includes the barrier
  else __syncthreads();
  if (tid < 32) {
    float2 t = tid < kWarps ? sh.red[tid] : make_float2(-INFINITY, 0.f);
    t = warp_combine(t);
    if (tid == 0) {
      p.partial[vr * kMaxChunksSampled + c] = t;
      if (draw) atomicMax(p.gkey + b, gk);
      __threadfence();
      if (atomicAdd(p.rcount + vr, 1u) == (unsigned)(p.C - 1)) {  // row complete
        atomicExch(p.rcount + vr, 0u);
        float2 acc = __ldcg(p.partial + vr * kMaxChunksSampled);
        for (int cc = 1; cc < p.C; ++cc)  // chunk order: deterministic
          acc = combine(acc, __ldcg(p.partial + vr * kMaxChunksSampled + cc));
        for (int cc = 0; cc < p.C; ++cc)
          p.partial[vr * kMaxChunksSampled + cc] = make_float2(0.f, 0.f);
        const float L = acc.x + log2f(acc.y);  // log2 of sum of 2^y
        p.lse[vr] = L;
        if (!draw) {  // probability of the row's draft token
          const int jj = vr < p.Rt ? j : (vr - p.Rt) - b * p.Kp;
          const int x = __ldg(p.tokens + b * (p.Kp + 1) + jj + 1);
          p.prob[vr] = (x >= 0 && x < p.V) ? ex2(E::at(rowp, x) * p.c2 - L) : -1.f;
        }
        __threadfence();
        if (atomicAdd(p.qcount + b, 1u) == (unsigned)(2 * p.Kp)) {  // all 2Kp+1 rows
          atomicExch(p.qcount + b, 0u);
          __threadfence();
          decide(p, b);
        }
      }
    }
  }
  __syncthreads();
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 3) sampled_stats_kernel(const SampledParams p) {
  __shared__ SampledShared sh;
  const int n_units = (p.Rt + p.Rd) * p.C;
  int u = blockIdx.x;
  while (u < n_units) {
    unsigned next = 0;
    if (threadIdx.x == 0) next = gridDim.x + atomicAdd(p.sched, 1u);
    stats_unit<DT>(p, sh, u);
    if (threadIdx.x == 0) sh.unit = (int)next;
    __syncthreads();
    u = sh.unit;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
}

}  // namespace pe

namespace pe {

// Residual draw of request b, chunk c: Gumbel-max over log2 max(0, p - q)
// with p = 2^(y_t - L_t), q = 2^(y_d - L_d).  The unit that completes the
// request publishes the draw; should the residual be empty (p == q
// everywhere, possible only for identical rows) that CTA draws from p over
// the whole target row instead.
template <int DT>
__device__ __forceinline__ void residual_unit(const SampledParams& p, SampledShared& sh, int u) {
  using E = Vec<DT>;
  const int tid = threadIdx.x;
  const int b = u / p.C2;
  const int c = u - b * p.C2;
  if (tid == 0) sh.acc = __ldcg(p.acc + b);
  __syncthreads();
  const int a = sh.acc;
  const bool draw = a < p.Kp;  // else the stats pass drew the bonus already
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
    constexpr int kV = kVecPerThread / 2;  // two rows: half the vectors each
    for (int base = v_lo; base < v_hi; base += kThreads * kV) {
      if (base + tid >= v_hi) break;
      uint4 xt[kV], xd[kV];
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = base + i * kThreads + tid;
        xt[i] = v < v_hi ? __ldcs(tr + v) : make_uint4(0u, 0u, 0u, 0u);
        xd[i] = v < v_hi ? __ldcs(dr + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = base + i * kThreads + tid;
        if (v >= v_hi) continue;
        float zt[E::kN], zd[E::kN];
        E::unpack(xt[i], zt);
        E::unpack(xd[i], zd);
#pragma unroll
        for (int g = 0; g < E::kN / 4; ++g) {
          const uint4 w = philox(p, (uint32_t)((v * E::kN) / 4 + g), (uint32_t)b);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = 4 * g + k;
            const float d = ex2(fmaf(zt[e], p.c2, -Lt)) - ex2(fmaf(zd[e], p.c2, -Ld));
            if (d > 0.f) best.offer(lg2(d) + noise2(ws[k]), v * E::kN + e);
          }
        }
      }
    }
    if (p.tail && c == p.C2 - 1 && tid == 0) {
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
  const unsigned long long k = block_max_key(sh, best.key());
  if (tid == 0) {
    sh.fallback = 0;
    if (draw) atomicMax(p.rkey + b, k);
    __threadfence();
    if (atomicAdd(p.dcount + b, 1u) == (unsigned)(p.C2 - 1)) {  // every unit of b is done
      atomicExch(p.dcount + b, 0u);
      p.acc[b] = 0;
      if (draw) {
        const unsigned long long r = atomicExch(p.rkey + b, 0ull);
        if (r) p.bonus_token[b] = (int)key_col(r);
        else sh.fallback = 1;
        p.lse[vt] = 0.f;
        p.lse[vd] = 0.f;
      }
    }
  }
  __syncthreads();
  if (sh.fallback) {  // empty residual: draw from p (rare; one CTA, whole row)
    const char* trow = vrow_ptr(p, vt);
    Best bp;
    for (int col = tid; col < p.V; col += kThreads) {
      const uint4 w = philox(p, (uint32_t)(col / 4), (uint32_t)b);
      bp.offer(E::at(trow, col) * p.c2 + noise2(word(w, col & 3)), col);
    }
    const unsigned long long kf = block_max_key(sh, bp.key());
    if (tid == 0) p.bonus_token[b] = (int)key_col(kf);
  }
  __syncthreads();
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 3) sampled_residual_kernel(const SampledParams p) {
  __shared__ SampledShared sh;
  const int n_units = p.B * p.C2;
  int u = blockIdx.x;
  while (u < n_units) {
    unsigned next = 0;
    if (threadIdx.x == 0) next = gridDim.x + atomicAdd(p.sched + 2, 1u);
    residual_unit<DT>(p, sh, u);
    if (threadIdx.x == 0) sh.unit = (int)next;
    __syncthreads();
    u = sh.unit;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 3, 1u) == gridDim.x - 1) {
      atomicExch(p.sched + 2, 0u);
      atomicExch(p.sched + 3, 0u);
    }
  }
}

}  // namespace pe

// ---------------------------------------------------------------- host side
namespace {

struct SampledLayout {
  size_t partial_off, lse_off, prob_off, rcount_off, qcount_off, dcount_off, acc_off, gkey_off,
      rkey_off, bytes;
  SampledLayout(long long B, long long Kp) {
    const long long rows = B * (Kp + 1) + B * Kp;
    size_t o = 16;  // four scheduler words
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
  const int grid_max = dev.sm_count * 3;

  pe::SampledParams p = {};
  p.B = B;
  p.Kp = Kp;
  p.V = V;
  const int epv = 16 / elt;
  p.nvec = V / epv;
  p.tail = V % epv;
  p.Rt = B * (Kp + 1);
  p.Rd = B * Kp;
  // stats chunks: whole batches of kBatchVecs vectors, at most 4 per chunk,
  // enough chunks for about one unit per CTA, at most the partial slots
  int C = 1;
  if (p.nvec > 0) {
    const int nb = ceil_div(p.nvec, pe::kBatchVecs);
    C = ceil_div(nb, 4);
    const int want = ceil_div(grid_max, rows);
    if (C < want) C = want;
    const int c_max = ceil_div(p.nvec, pe::kThreads);
    if (C > c_max) C = c_max;
    if (C > pe::kMaxChunksSampled) C = pe::kMaxChunksSampled;
    p.chunk_vecs = C <= nb ? ceil_div(nb, C) * pe::kBatchVecs : ceil_div(p.nvec, C);
    if (p.chunk_vecs > p.nvec) p.chunk_vecs = p.nvec;
    C = ceil_div(p.nvec, p.chunk_vecs);
  }
  p.C = C;
  // residual chunks: about four units per CTA over all requests (those
  // without a rejection leave at once)
  int C2 = 1;
  if (p.nvec > 0) {
    C2 = ceil_div(4LL * grid_max, B);
    const int c_max = ceil_div(p.nvec, pe::kThreads);
    if (C2 > c_max) C2 = c_max;
    if (C2 < 1) C2 = 1;
    p.chunk2_vecs = ceil_div(p.nvec, C2);
    C2 = ceil_div(p.nvec, p.chunk2_vecs);
  }
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
  p.partial = reinterpret_cast<float2*>(w + L.partial_off);
  p.lse = reinterpret_cast<float*>(w + L.lse_off);
  p.prob = reinterpret_cast<float*>(w + L.prob_off);
  p.rcount = reinterpret_cast<uint32_t*>(w + L.rcount_off);
  p.qcount = reinterpret_cast<uint32_t*>(w + L.qcount_off);
  p.dcount = reinterpret_cast<uint32_t*>(w + L.dcount_off);
  p.acc = reinterpret_cast<int32_t*>(w + L.acc_off);
  p.gkey = reinterpret_cast<unsigned long long*>(w + L.gkey_off);
  p.rkey = reinterpret_cast<unsigned long long*>(w + L.rkey_off);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long n1 = rows * p.C;
  const int g1 = n1 < grid_max ? (int)n1 : grid_max;
  const long long n2 = (long long)B * p.C2;
  const int g2 = n2 < grid_max ? (int)n2 : grid_max;
  if (dtype == PE_BF16) {
    pe::sampled_stats_kernel<PE_BF16><<<g1, pe::kThreads, 0, st>>>(p);
    pe::sampled_residual_kernel<PE_BF16><<<g2, pe::kThreads, 0, st>>>(p);
  } else {
    pe::sampled_stats_kernel<PE_F32><<<g1, pe::kThreads, 0, st>>>(p);
    pe::sampled_residual_kernel<PE_F32><<<g2, pe::kThreads, 0, st>>>(p);
  }
  return pe_host::launch_status();
}

}  // extern "C"
