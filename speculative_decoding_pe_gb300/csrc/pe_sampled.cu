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
//     chunks; each chunk yields a (max, sum of exp) pair of its scaled
//     logits, merged in chunk order by the chunk that completes the row,
//     which also evaluates p(x) or q(x) of the row's draft token.  The last
//     row of a request decides its accepted length.  For the bonus row of
//     every request the same pass also draws the Gumbel-max sample of
//     softmax(row / temperature), used when every draft is accepted.
//  2. residual: for requests with a rejection, the chunks of their target
//     and draft rows at the rejected position are streamed again to draw from
//     max(0, p - q) (and, should that be empty, from p).
// Draws use Gumbel noise -log(-log(U)) with U from Philox4x32-10 (Salmon et
// al., SC'11), counter (i / 4, request, 0, 0), key = the seed's two words.
#include <atomic>

#include "pe_internal.cuh"

namespace pe {

constexpr int kMaxChunksSampled = 16;  // chunks per row (partial stats slots)

struct SampledParams {
  int B, Kp, V, nvec, tail, C, chunk_vecs, Rt, Rd;
  float inv_t;
  unsigned long long seed;
  long long t_row_bytes, d_row_bytes;
  const void* tlogits;
  const void* dlogits;
  const int32_t* tokens;
  const float* u_accept;
  int32_t* accepted_len;
  int32_t* bonus_token;
  uint32_t* err;
  // workspace
  uint32_t* sched;            // [2] unit counter, CTAs done
  float2* partial;            // [Rt+Rd][kMaxChunksSampled] (max, sum) per chunk
  float2* stats;              // [Rt+Rd] (max, sum) per row
  float* prob;                // [Rt+Rd] p(x) or q(x) of the row's draft token
  uint32_t* rcount;           // [Rt+Rd] finished chunks per row
  uint32_t* qcount;           // [B] finished rows per request (stats pass)
  uint32_t* dcount;           // [B] finished chunks per request (residual pass)
  int32_t* acc;               // [B] accepted length, for the residual pass
  unsigned long long* gkey;   // [B] Gumbel draw from the bonus row
  unsigned long long* rkey;   // [B] Gumbel draw from the residual
  unsigned long long* fkey;   // [B] Gumbel draw from p (empty residual)
};

// ------------------------------------------------------------ Philox4x32-10
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Gumbel noise of the four elements 4g..4g+3 of the draw of request b.
__device__ __forceinline__ void gumbel4(const SampledParams& p, int b, int g, float (&out)[4]) {
  const uint4 w = philox4x32_10(make_uint4((uint32_t)g, (uint32_t)b, 0u, 0u),
                                (uint32_t)p.seed, (uint32_t)(p.seed >> 32));
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float u = ((float)(ws[k] >> 8) + 0.5f) * (1.0f / 16777216.0f);  // exact, in (0,1)
    out[k] = -logf(-logf(u));
  }
}

// ----------------------------------------------------------- element access
template <int DT>
struct Vec;

template <>
struct Vec<PE_BF16> {
  static constexpr int kN = 8;
  __device__ static __forceinline__ void unpack(uint4 q, float (&z)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      z[2 * i] = bf16_lo(w[i]);
      z[2 * i + 1] = bf16_hi(w[i]);
    }
  }
  __device__ static __forceinline__ float at(const char* row, int col) {
    return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + col))
                           << 16);
  }
};

template <>
struct Vec<PE_F32> {
  static constexpr int kN = 4;
  __device__ static __forceinline__ void unpack(uint4 q, float (&z)[4]) {
    z[0] = __uint_as_float(q.x);
    z[1] = __uint_as_float(q.y);
    z[2] = __uint_as_float(q.z);
    z[3] = __uint_as_float(q.w);
  }
  __device__ static __forceinline__ float at(const char* row, int col) {
    return __ldg(reinterpret_cast<const float*>(row) + col);
  }
};

// (max, sum of exp(z - max)) of two disjoint sets, merged.
__device__ __forceinline__ float2 combine(float2 a, float2 b) {
  if (a.y == 0.f) return b;
  if (b.y == 0.f) return a;
  const float m = fmaxf(a.x, b.x);
  return make_float2(m, a.y * expf(a.x - m) + b.y * expf(b.x - m));
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

}  // namespace pe

namespace pe {

struct SampledShared {
  float2 red[kWarps];
  unsigned long long kred[kWarps];
  unsigned long long kred2[kWarps];
  int unit;
  int done_req;
  int acc;
};

// Virtual row vr: target rows [0, Rt), then draft rows [Rt, Rt + Rd).
__device__ __forceinline__ const char* vrow_ptr(const SampledParams& p, int vr) {
  return vr < p.Rt ? static_cast<const char*>(p.tlogits) + (long long)vr * p.t_row_bytes
                   : static_cast<const char*>(p.dlogits) + (long long)(vr - p.Rt) * p.d_row_bytes;
}

// Scaled logits of one row chunk folded into (max, sum of exp) and, for the
// bonus row (draw), into the Gumbel-max key of softmax(row / temperature).
template <int DT>
__device__ __forceinline__ void fold_chunk(const SampledParams& p, const char* rowp, int v_lo,
                                           int v_hi, bool tail, bool draw, int b, float& m,
                                           float& s, unsigned long long& gk) {
  using E = Vec<DT>;
  const int tid = threadIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(rowp);
  for (int base = v_lo; base < v_hi; base += kBatchVecs) {
    if (base + tid >= v_hi) break;
    uint4 x[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int v = base + i * kThreads + tid;
      x[i] = v < v_hi ? __ldcs(row + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    float bm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      if (base + i * kThreads + tid >= v_hi) continue;
      float z[E::kN];
      E::unpack(x[i], z);
#pragma unroll
      for (int e = 0; e < E::kN; ++e) bm = fmaxf(bm, z[e] * p.inv_t);
    }
    if (bm > m) {
      s = (m == -INFINITY) ? 0.f : s * __expf(m - bm);
      m = bm;
    }
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int v = base + i * kThreads + tid;
      if (v >= v_hi) continue;
      float z[E::kN];
      E::unpack(x[i], z);
#pragma unroll
      for (int e = 0; e < E::kN; ++e) s += __expf(z[e] * p.inv_t - m);
      if (draw) {
#pragma unroll
        for (int g = 0; g < E::kN / 4; ++g) {
          float gn[4];
          gumbel4(p, b, (v * E::kN) / 4 + g, gn);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int col = v * E::kN + 4 * g + k;
            const unsigned long long key = make_key(z[4 * g + k] * p.inv_t + gn[k], (uint32_t)col);
            gk = key > gk ? key : gk;
          }
        }
      }
    }
  }
  if (tail && tid == 0) {  // elements after the last whole vector
    for (int e = 0; e < p.tail; ++e) {
      const int col = p.nvec * E::kN + e;
      const float z = E::at(rowp, col) * p.inv_t;
      if (z > m) {
        s = (m == -INFINITY) ? 0.f : s * __expf(m - z);
        m = z;
      }
      s += __expf(z - m);
      if (draw) {
        float gn[4];
        gumbel4(p, b, col / 4, gn);
        const unsigned long long key = make_key(z + gn[col & 3], (uint32_t)col);
        gk = key > gk ? key : gk;
      }
    }
  }
}

// Accepted length of request b from its rows' draft-token probabilities.
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
  // leave the workspace zeroed: what this request's residual draw reads
  // (the statistics of target and draft row a) is cleared by that draw
  for (int j = 0; j <= p.Kp; ++j) {
    const int vt = b * (p.Kp + 1) + j;
    if (j < p.Kp) p.prob[vt] = 0.f;
    if (j != a || a == p.Kp) p.stats[vt] = make_float2(0.f, 0.f);
    if (j < p.Kp) {
      const int vd = p.Rt + b * p.Kp + j;
      p.prob[vd] = 0.f;
      if (j != a) p.stats[vd] = make_float2(0.f, 0.f);
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
  bool target;
  if (vr < p.Rt) {
    target = true;
    b = vr / (p.Kp + 1);
    j = vr - b * (p.Kp + 1);
  } else {
    target = false;
    b = (vr - p.Rt) / p.Kp;
    j = (vr - p.Rt) - b * p.Kp;
  }
  const bool draw = target && j == p.Kp;  // the bonus row
  const char* rowp = vrow_ptr(p, vr);
  const int v_lo = c * p.chunk_vecs;
  const int v_hi = min(v_lo + p.chunk_vecs, p.nvec);
  float m = -INFINITY, s = 0.f;
  unsigned long long gk = 0ull;
  fold_chunk<DT>(p, rowp, v_lo, v_hi, p.tail && c == p.C - 1, draw, b, m, s, gk);

  float2 st = warp_combine(make_float2(m, s));
  gk = warp_max_key(gk);
  if ((tid & 31) == 0) {
    sh.red[tid >> 5] = st;
    sh.kred[tid >> 5] = gk;
  }
  __syncthreads();
  if (tid < 32) {
    float2 t = tid < kWarps ? sh.red[tid] : make_float2(-INFINITY, 0.f);
    unsigned long long k = tid < kWarps ? sh.kred[tid] : 0ull;
    t = warp_combine(t);
    k = warp_max_key(k);
    if (tid == 0) {
      p.partial[vr * kMaxChunksSampled + c] = t;
      if (draw) atomicMax(p.gkey + b, k);
      __threadfence();
      if (atomicAdd(p.rcount + vr, 1u) == (unsigned)(p.C - 1)) {  // row complete
        atomicExch(p.rcount + vr, 0u);
        float2 acc = __ldcg(p.partial + vr * kMaxChunksSampled);
        for (int cc = 1; cc < p.C; ++cc)  // chunk order: deterministic
          acc = combine(acc, __ldcg(p.partial + vr * kMaxChunksSampled + cc));
        for (int cc = 0; cc < p.C; ++cc) p.partial[vr * kMaxChunksSampled + cc] = make_float2(0.f, 0.f);
        p.stats[vr] = acc;
        if (!draw) {  // probability of the row's draft token
          const int x = __ldg(p.tokens + b * (p.Kp + 1) + j + 1);
          p.prob[vr] = (x >= 0 && x < p.V)
                           ? __expf(E::at(rowp, x) * p.inv_t - acc.x) / acc.y
                           : -1.f;
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

// Residual draw of request b, chunk c: Gumbel-max over log max(0, p - q),
// and over log p in case the residual is empty (p == q everywhere).
template <int DT>
__device__ __forceinline__ void residual_unit(const SampledParams& p, SampledShared& sh, int u) {
  using E = Vec<DT>;
  const int tid = threadIdx.x;
  const int b = u / p.C;
  const int c = u - b * p.C;
  if (tid == 0) sh.acc = __ldcg(p.acc + b);
  __syncthreads();
  const int a = sh.acc;
  const bool draw = a < p.Kp;  // else the stats pass drew the bonus already
  const int vt = b * (p.Kp + 1) + a;
  const int vd = p.Rt + b * p.Kp + a;
  unsigned long long rk = 0ull, fk = 0ull;
  if (draw) {
    const float2 sp = __ldcg(p.stats + vt);
    const float2 sq = __ldcg(p.stats + vd);
    const float isp = 1.f / sp.y, isq = 1.f / sq.y;
    const char* trow = vrow_ptr(p, vt);
    const char* drow = vrow_ptr(p, vd);
    const uint4* tr = reinterpret_cast<const uint4*>(trow);
    const uint4* dr = reinterpret_cast<const uint4*>(drow);
    const int v_lo = c * p.chunk_vecs;
    const int v_hi = min(v_lo + p.chunk_vecs, p.nvec);
    auto score = [&](float zt, float zd, int col, float gn) {
      const float pr = __expf(zt - sp.x) * isp;
      const float qr = __expf(zd - sq.x) * isq;
      if (pr - qr > 0.f) {
        const unsigned long long k = make_key(__logf(pr - qr) + gn, (uint32_t)col);
        rk = k > rk ? k : rk;
      }
      const unsigned long long k2 = make_key(zt + gn, (uint32_t)col);
      fk = k2 > fk ? k2 : fk;
    };
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
          float gn[4];
          gumbel4(p, b, (v * E::kN) / 4 + g, gn);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            score(zt[4 * g + k] * p.inv_t, zd[4 * g + k] * p.inv_t, v * E::kN + 4 * g + k, gn[k]);
        }
      }
    }
    if (p.tail && c == p.C - 1 && tid == 0) {
      for (int e = 0; e < p.tail; ++e) {
        const int col = p.nvec * E::kN + e;
        float gn[4];
        gumbel4(p, b, col / 4, gn);
        score(E::at(trow, col) * p.inv_t, E::at(drow, col) * p.inv_t, col, gn[col & 3]);
      }
    }
  }
  rk = warp_max_key(rk);
  fk = warp_max_key(fk);
  if ((tid & 31) == 0) {
    sh.kred[tid >> 5] = rk;
    sh.kred2[tid >> 5] = fk;
  }
  __syncthreads();
  if (tid < 32) {
    unsigned long long k = tid < kWarps ? sh.kred[tid] : 0ull;
    unsigned long long f = tid < kWarps ? sh.kred2[tid] : 0ull;
    k = warp_max_key(k);
    f = warp_max_key(f);
    if (tid == 0) {
      if (draw) {
        atomicMax(p.rkey + b, k);
        atomicMax(p.fkey + b, f);
      }
      __threadfence();
      if (atomicAdd(p.dcount + b, 1u) == (unsigned)(p.C - 1)) {  // every unit of b is done
        atomicExch(p.dcount + b, 0u);
        if (draw) {
          const unsigned long long r = atomicExch(p.rkey + b, 0ull);
          const unsigned long long f2 = atomicExch(p.fkey + b, 0ull);
          p.bonus_token[b] = (int)key_col(r ? r : f2);
          p.stats[vt] = make_float2(0.f, 0.f);
          p.stats[vd] = make_float2(0.f, 0.f);
        }
        p.acc[b] = 0;
      }
    }
  }
  __syncthreads();
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 3) sampled_residual_kernel(const SampledParams p) {
  __shared__ SampledShared sh;
  for (int u = blockIdx.x; u < p.B * p.C; u += gridDim.x) residual_unit<DT>(p, sh, u);
}

}  // namespace pe

// ---------------------------------------------------------------- host side
namespace {

struct SampledLayout {
  size_t partial_off, stats_off, prob_off, rcount_off, qcount_off, dcount_off, acc_off,
      gkey_off, rkey_off, fkey_off, bytes;
  SampledLayout(long long B, long long Kp) {
    const long long rows = B * (Kp + 1) + B * Kp;
    size_t o = 16;
    auto take = [&](size_t n, size_t align) {
      o = (o + align - 1) / align * align;
      const size_t at = o;
      o += n;
      return at;
    };
    partial_off = take(8 * rows * pe::kMaxChunksSampled, 16);
    stats_off = take(8 * rows, 16);
    prob_off = take(4 * rows, 16);
    rcount_off = take(4 * rows, 16);
    qcount_off = take(4 * B, 16);
    dcount_off = take(4 * B, 16);
    acc_off = take(4 * B, 16);
    gkey_off = take(8 * B, 16);
    rkey_off = take(8 * B, 16);
    fkey_off = take(8 * B, 16);
    bytes = (o + 255) / 256 * 256;
  }
};

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
  // chunks per row: ~4 batches each, at least ~one unit per CTA, at most the
  // partial-statistics slots
  int C = 1;
  if (p.nvec > 0) {
    const int cap = 4 * pe::kBatchVecs;
    C = (p.nvec + cap - 1) / cap;
    const int want = (int)((grid_max + rows - 1) / rows);
    if (C < want) C = want;
    const int c_max = (p.nvec + pe::kThreads - 1) / pe::kThreads;
    if (C > c_max) C = c_max;
    if (C > pe::kMaxChunksSampled) C = pe::kMaxChunksSampled;
    if (C < 1) C = 1;
  }
  p.chunk_vecs = p.nvec ? (p.nvec + C - 1) / C : 0;
  p.C = p.nvec ? (p.nvec + p.chunk_vecs - 1) / p.chunk_vecs : 1;
  p.inv_t = 1.f / temperature;
  p.seed = seed;
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
  p.stats = reinterpret_cast<float2*>(w + L.stats_off);
  p.prob = reinterpret_cast<float*>(w + L.prob_off);
  p.rcount = reinterpret_cast<uint32_t*>(w + L.rcount_off);
  p.qcount = reinterpret_cast<uint32_t*>(w + L.qcount_off);
  p.dcount = reinterpret_cast<uint32_t*>(w + L.dcount_off);
  p.acc = reinterpret_cast<int32_t*>(w + L.acc_off);
  p.gkey = reinterpret_cast<unsigned long long*>(w + L.gkey_off);
  p.rkey = reinterpret_cast<unsigned long long*>(w + L.rkey_off);
  p.fkey = reinterpret_cast<unsigned long long*>(w + L.fkey_off);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int n1 = (int)rows * p.C;
  const int g1 = n1 < grid_max ? n1 : grid_max;
  const int n2 = B * p.C;
  const int g2 = n2 < grid_max ? n2 : grid_max;
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
