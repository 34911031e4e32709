/*
 * CPU oracle for the P-EAGLE parallel-drafting step.  TEST INFRASTRUCTURE
 * ONLY (tests, smoke check, benchmark CPU baseline); never on the product
 * path.  Plain single-threaded C, one element at a time, no blocking, no
 * fusion.  Shares nothing with the CUDA library.
 *
 * Sources (page title -- section):
 *  [P1] "P-EAGLE: Faster LLM Inference with Parallel Speculative Decoding in
 *       vLLM" -- quick-read section, input equation Input_i; and the vLLM
 *       engineering-details listing (hidden-state scatter, then MASK fill).
 *  [P2] "P-EAGLE: Parallel Speculative Decoding in vLLM" -- "Step 2: Parallel
 *       Drafting" (prompt positions shifted by one; NTP; MTP placeholders),
 *       "Fused Triton Kernel" (outputs of the rebuild), "Hidden State
 *       Management", "KV Cache and CUDA Graphs" (rejected -> slot -1).
 *  Greedy acceptance: the acceptance-length definition in [P1] quick-read
 *  results paragraph, read as "longest prefix of drafts equal to the
 *  target's argmax, plus the target's token at the first mismatch".
 *
 * Readings where the pages are silent (each is a convention of this
 * project, applied identically by the CUDA path):
 *  - argmax ties go to the lowest index; -0.0 equals +0.0 (numeric compare).
 *  - rejected slot k < n-1 keeps the shifted copy in[k+1] as its token; the
 *    last slot k = n-1, when rejected, holds the MASK id.
 *  - every slot keeps its own target position; MASK slot i (1..K-1) sits at
 *    the bonus slot's position + i.
 *  - emb(mask) is the embedding row of the MASK id.
 *  - rejected slots keep their own target hidden row (identity mapping).
 *  - data errors: a gathered token outside [0,V) gives a zero embedding half;
 *    a position outside the block table gives slot -1; both raise a bit.
 */
#include "pe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- element access -------------------------------------------------- */

/* bf16 is by definition the high 16 bits of an IEEE-754 binary32. */
static double load_elem(const void* base, int dtype, int64_t i) {
  if (dtype == ORC_F32) {
    float f;
    memcpy(&f, (const char*)base + 4 * i, 4);
    return (double)f;
  } else {
    uint16_t h;
    uint32_t bits;
    float f;
    memcpy(&h, (const char*)base + 2 * i, 2);
    bits = ((uint32_t)h) << 16;
    memcpy(&f, &bits, 4);
    return (double)f;
  }
}

static int elt_of(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* ---- a1: row argmax --------------------------------------------------- */

int oracle_argmax_rows(const void* logits, int dtype, int64_t row_stride,
                       int32_t rows, int32_t V, int32_t* out) {
  int32_t r, v;
  if (rows < 0 || V < 1 || (rows > 0 && (!logits || !out))) return -1;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return -1;
  for (r = 0; r < rows; ++r) {
    int64_t base = (int64_t)r * row_stride;
    int32_t best = 0;
    double best_val = load_elem(logits, dtype, base);
    for (v = 1; v < V; ++v) {
      double x = load_elem(logits, dtype, base + v);
      if (x > best_val) { /* strict: the first maximum stays */
        best_val = x;
        best = v;
      }
    }
    out[r] = best;
  }
  return 0;
}

/* ---- drafter readout: greedy t_1..t_K from the drafter's logits -------- */
/* "P-EAGLE: Parallel Speculative Decoding in vLLM" -- Step 2: the LM head
   predicts draft tokens t_1..t_K; greedy drafting takes each row's argmax. */

int oracle_draft_readout(const void* logits, int dtype, int64_t row_stride,
                         int32_t rows, int32_t V, const int32_t* sample_idx,
                         int32_t n, int32_t* out, uint32_t* err) {
  int32_t i;
  if (rows < 0 || V < 1 || n < 0 || !err) return -1;
  if (n > 0 && (!logits || !out)) return -1;
  for (i = 0; i < n; ++i) {
    int32_t r = sample_idx ? sample_idx[i] : i;
    if (r < 0 || r >= rows) {
      *err |= ORC_ERR_ROW_RANGE;
      out[i] = -1;
      continue;
    }
    oracle_argmax_rows((const char*)logits +
                           (int64_t)r * row_stride * elt_of(dtype),
                       dtype, row_stride, 1, V, &out[i]);
  }
  return 0;
}

/* ---- a2: greedy acceptance and bonus token ---------------------------- */

int oracle_verify_greedy(const void* logits, int dtype, int64_t row_stride,
                         int32_t B, int32_t Kp, int32_t V,
                         const int32_t* tokens, int32_t* accepted_len,
                         int32_t* bonus_token, int32_t* target_argmax) {
  int32_t rows, b, j;
  int32_t* amax;
  if (B < 0 || Kp < 0 || V < 1) return -1;
  if (B == 0) return 0;
  if (!logits || !accepted_len || !bonus_token) return -1;
  if (Kp > 0 && !tokens) return -1;
  rows = B * (Kp + 1);
  amax = target_argmax ? target_argmax
                       : (int32_t*)malloc(sizeof(int32_t) * (size_t)rows);
  if (!amax) return -1;
  oracle_argmax_rows(logits, dtype, row_stride, rows, V, amax);
  for (b = 0; b < B; ++b) {
    int32_t first = b * (Kp + 1);
    int32_t a = Kp; /* all drafts accepted unless a mismatch is found */
    for (j = 0; j < Kp; ++j) {
      /* the target's choice after row j is compared with draft d_{j+1} */
      if (amax[first + j] != tokens[first + j + 1]) {
        a = j;
        break;
      }
    }
    accepted_len[b] = a;
    bonus_token[b] = amax[first + a]; /* target token at the first mismatch */
  }
  if (!target_argmax) free(amax);
  return 0;
}

/* ---- rejection-sampling verification ----------------------------------- */
/* "并行草稿机制解析：从P-EAGLE到DSpark的投机采样加速" §1.2: the target checks the
   drafts one by one against its own distribution, accepts when they agree
   well enough and otherwise replaces from that position with its own output,
   so that the result has exactly the target's distribution.  Read as the
   standard rule: accept with probability min(1, p/q); on rejection draw from
   the normalised max(0, p - q); after all acceptances draw from p. */

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  int r;
  for (r = 0; r < 10; ++r) {
    uint64_t p0, p1;
    uint32_t n0, n2;
    if (r > 0) { /* key schedule: Weyl increments */
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    p0 = (uint64_t)0xD2511F53u * c0;
    p1 = (uint64_t)0xCD9E8D57u * c2;
    n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* Gumbel noise for element i of draw `stream` */
static double gumbel(uint64_t seed, uint32_t stream, int32_t i) {
  uint32_t ctr[4], key[2], w[4];
  double u;
  ctr[0] = (uint32_t)i >> 2;
  ctr[1] = stream;
  ctr[2] = 0;
  ctr[3] = 0;
  key[0] = (uint32_t)seed;
  key[1] = (uint32_t)(seed >> 32);
  oracle_philox4x32_10(ctr, key, w);
  /* 23 bits: (k + 0.5) / 2^23 needs 24 significant bits, so U is exact in
   * fp32 as well and lies in [2^-24, 1 - 2^-24] */
  u = ((double)(w[i & 3] >> 9) + 0.5) / 8388608.0;
  return -log(-log(u));
}

/* probability of column x under softmax(row / temperature) */
static double softmax_at(const void* logits, int dtype, int64_t base, int32_t V,
                         double inv_t, int32_t x) {
  double m = -INFINITY, s = 0.0;
  int32_t v;
  for (v = 0; v < V; ++v) {
    double z = load_elem(logits, dtype, base + v) * inv_t;
    if (z > m) m = z;
  }
  for (v = 0; v < V; ++v) s += exp(load_elem(logits, dtype, base + v) * inv_t - m);
  return exp(load_elem(logits, dtype, base + x) * inv_t - m) / s;
}

int oracle_verify_sampled(const void* target_logits, const void* draft_logits,
                          int dtype, int64_t target_stride,
                          int64_t draft_stride, int32_t B, int32_t Kp,
                          int32_t V, const int32_t* tokens,
                          const float* u_accept, float temperature,
                          uint64_t seed, int32_t* accepted_len,
                          int32_t* bonus_token) {
  int32_t b, j, v;
  double inv_t;
  if (B < 0 || Kp < 0 || V < 1 || !(temperature > 0.0f)) return -1;
  if (B == 0) return 0;
  if (!target_logits || !accepted_len || !bonus_token) return -1;
  if (Kp > 0 && (!draft_logits || !tokens || !u_accept)) return -1;
  inv_t = 1.0 / (double)temperature;
  for (b = 0; b < B; ++b) {
    int32_t a = Kp, best = 0;
    double best_s = -INFINITY;
    int64_t trow, drow;
    for (j = 0; j < Kp; ++j) {
      int32_t x = tokens[(int64_t)b * (Kp + 1) + j + 1];
      double px, qx;
      trow = ((int64_t)b * (Kp + 1) + j) * target_stride;
      drow = ((int64_t)b * Kp + j) * draft_stride;
      if (x < 0 || x >= V) {
        a = j;
        break;
      }
      px = softmax_at(target_logits, dtype, trow, V, inv_t, x);
      qx = softmax_at(draft_logits, dtype, drow, V, inv_t, x);
      if (!((double)u_accept[(int64_t)b * Kp + j] * qx < px)) {
        a = j;
        break;
      }
    }
    trow = ((int64_t)b * (Kp + 1) + a) * target_stride;
    if (a < Kp) { /* draw from max(0, p - q) */
      double mt = -INFINITY, md = -INFINITY, st = 0.0, sd = 0.0;
      int any = 0;
      drow = ((int64_t)b * Kp + a) * draft_stride;
      for (v = 0; v < V; ++v) {
        double zt = load_elem(target_logits, dtype, trow + v) * inv_t;
        double zd = load_elem(draft_logits, dtype, drow + v) * inv_t;
        if (zt > mt) mt = zt;
        if (zd > md) md = zd;
      }
      for (v = 0; v < V; ++v) {
        st += exp(load_elem(target_logits, dtype, trow + v) * inv_t - mt);
        sd += exp(load_elem(draft_logits, dtype, drow + v) * inv_t - md);
      }
      for (v = 0; v < V; ++v) {
        double pv = exp(load_elem(target_logits, dtype, trow + v) * inv_t - mt) / st;
        double qv = exp(load_elem(draft_logits, dtype, drow + v) * inv_t - md) / sd;
        if (pv - qv > 0.0) {
          double sc = log(pv - qv) + gumbel(seed, (uint32_t)b, v);
          if (!any || sc > best_s) {
            best_s = sc;
            best = v;
          }
          any = 1;
        }
      }
      if (any) {
        accepted_len[b] = a;
        bonus_token[b] = best;
        continue;
      }
      /* p == q: the residual is empty, draw from p */
    }
    for (v = 0; v < V; ++v) { /* draw from softmax(row / temperature) */
      double sc = load_elem(target_logits, dtype, trow + v) * inv_t +
                  gumbel(seed, (uint32_t)b, v);
      if (v == 0 || sc > best_s) {
        best_s = sc;
        best = v;
      }
    }
    accepted_len[b] = a;
    bonus_token[b] = best;
  }
  return 0;
}

/* ---- a3..a5: draft-batch rebuild --------------------------------------- */

int oracle_build_draft_batch(int32_t B, int32_t Kp, int32_t K, int32_t mask_id,
                             const int32_t* in_offsets, const int32_t* in_tokens,
                             const int32_t* in_positions,
                             const int32_t* accepted_len,
                             const int32_t* bonus_token,
                             const int32_t* block_table, int32_t bt_width,
                             int32_t block_size, int32_t* out_offsets,
                             int32_t* out_tokens, int32_t* out_positions,
                             uint8_t* is_rejected, uint8_t* is_masked,
                             int32_t* hidden_map, int64_t* slot_mapping,
                             int32_t* sample_idx, uint32_t* err) {
  int32_t b, k;
  int32_t* io;
  int32_t* oo;
  if (B < 0 || Kp < 0 || K < 1 || block_size < 1 || bt_width < 0) return -1;
  if (!err) return -1;
  if (B == 0) {
    if (out_offsets) out_offsets[0] = 0;
    return 0;
  }
  if (!in_tokens || !in_positions || !bonus_token || !block_table ||
      !out_offsets || !out_tokens || !out_positions || !is_rejected ||
      !is_masked || !hidden_map || !slot_mapping)
    return -1;

  io = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B + 1));
  oo = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B + 1));
  if (!io || !oo) {
    free(io);
    free(oo);
    return -1;
  }

  /* input segments: given offsets, or fixed blocks of Kp+1 rows */
  for (b = 0; b <= B; ++b) io[b] = in_offsets ? in_offsets[b] : b * (Kp + 1);
  if (in_offsets) {
    int ok = (io[0] == 0);
    for (b = 0; b < B; ++b)
      if (io[b + 1] - io[b] < Kp + 1) ok = 0; /* need >= 1 row and Kp drafts */
    if (!ok) {
      *err |= ORC_ERR_OFFSETS; /* nothing is written */
      free(io);
      free(oo);
      return 0;
    }
  }

  /* a3: output offsets, exclusive scan of m_b = n_b + K - 1 */
  oo[0] = 0;
  for (b = 0; b < B; ++b) oo[b + 1] = oo[b] + (io[b + 1] - io[b]) + (K - 1);
  for (b = 0; b <= B; ++b) out_offsets[b] = oo[b];

  for (b = 0; b < B; ++b) {
    int32_t n = io[b + 1] - io[b];
    int32_t m = n + K - 1;
    int32_t a = accepted_len ? accepted_len[b] : 0;
    int32_t s;
    int32_t bonus = bonus_token[b];
    if (a < 0 || a > Kp) {
      *err |= ORC_ERR_SLOT_RANGE;
      a = 0;
    }
    /* bonus slot: a_b among the Kp+1 verified rows, which are the last
       Kp+1 rows of the segment (decode: all n = Kp+1; prefill: the last) */
    s = n - 1 - Kp + a;

    for (k = 0; k < m; ++k) {
      int32_t t = oo[b] + k;
      int32_t tok, pos;
      uint8_t rej = 0, msk = 0;
      if (k < s) { /* accepted / prompt slot: token shifted by one */
        tok = in_tokens[io[b] + k + 1];
        pos = in_positions[io[b] + k];
      } else if (k == s) { /* next-token-prediction slot */
        tok = bonus;
        pos = in_positions[io[b] + s];
      } else if (k < n) { /* rejected draft slot */
        rej = 1;
        tok = (k < n - 1) ? in_tokens[io[b] + k + 1] : mask_id;
        pos = in_positions[io[b] + k];
      } else { /* MASK slot i = k - n + 1, i in 1..K-1 */
        msk = 1;
        tok = mask_id;
        pos = in_positions[io[b] + s] + (k - n + 1);
      }
      out_tokens[t] = tok;
      out_positions[t] = pos;
      is_rejected[t] = rej;
      is_masked[t] = msk;
      /* a5: paged-KV slot, rejected slots padded with -1 */
      if (rej) {
        slot_mapping[t] = -1;
      } else if (pos < 0 || pos / block_size >= bt_width) {
        *err |= ORC_ERR_BLOCK_RANGE;
        slot_mapping[t] = -1;
      } else {
        int64_t blk = block_table[(int64_t)b * bt_width + pos / block_size];
        slot_mapping[t] = blk * block_size + (pos % block_size);
      }
    }
    /* hidden-state mapping: target row io_b+k moves to output slot oo_b+k */
    for (k = 0; k < n; ++k) hidden_map[io[b] + k] = oo[b] + k;
    /* the K rows whose drafter outputs become t_1..t_K */
    if (sample_idx) {
      sample_idx[(int64_t)b * K] = oo[b] + s;
      for (k = 1; k < K; ++k) sample_idx[(int64_t)b * K + k] = oo[b] + n + k - 1;
    }
  }
  free(io);
  free(oo);
  return 0;
}

/* ---- a6, a7: drafter input assembly ----------------------------------- */

int oracle_assemble_draft_inputs(int32_t elt, int32_t H, int32_t V, int32_t T,
                                 int32_t R, const void* emb,
                                 const void* target_hidden,
                                 const void* h_shared,
                                 const int32_t* out_tokens,
                                 const int32_t* hidden_map,
                                 const uint8_t* is_masked, void* X,
                                 uint32_t* err) {
  int32_t t, i;
  size_t half;
  char* x = (char*)X;
  if ((elt != 2 && elt != 4) || H < 1 || V < 1 || T < 0 || R < 0) return -1;
  if (!err) return -1;
  if (T == 0 && R == 0) return 0;
  if (!emb || !target_hidden || !h_shared || !out_tokens || !hidden_map ||
      !is_masked || !X)
    return -1;
  half = (size_t)H * (size_t)elt;

  /* embedding half: emb(token) of every output slot */
  for (t = 0; t < T; ++t) {
    int32_t tok = out_tokens[t];
    char* dst = x + (size_t)t * 2 * half;
    if (tok < 0 || tok >= V) {
      *err |= ORC_ERR_TOKEN_RANGE;
      memset(dst, 0, half);
    } else {
      memcpy(dst, (const char*)emb + (size_t)tok * half, half);
    }
  }
  /* hidden half, step 1: target rows copied to their new positions */
  for (i = 0; i < R; ++i) {
    int32_t dst_row = hidden_map[i];
    if (dst_row < 0 || dst_row >= T) {
      *err |= ORC_ERR_MAP_RANGE;
      continue;
    }
    memcpy(x + (size_t)dst_row * 2 * half + half,
           (const char*)target_hidden + (size_t)i * half, half);
  }
  /* hidden half, step 2: masked slots take the shared hidden state */
  for (t = 0; t < T; ++t)
    if (is_masked[t]) memcpy(x + (size_t)t * 2 * half + half, h_shared, half);
  return 0;
}

/* ---- the whole step ----------------------------------------------------- */

int oracle_step(int logits_dtype, int x_dtype, int32_t B, int32_t Kp, int32_t K,
                int32_t V, int32_t H, int32_t mask_id, const void* logits,
                int64_t row_stride, const int32_t* in_offsets,
                const int32_t* in_tokens, const int32_t* in_positions,
                const int32_t* block_table, int32_t bt_width,
                int32_t block_size, const void* emb, const void* target_hidden,
                const void* h_shared, int32_t* accepted_len,
                int32_t* bonus_token, int32_t* target_argmax,
                int32_t* out_offsets, int32_t* out_tokens,
                int32_t* out_positions, uint8_t* is_rejected,
                uint8_t* is_masked, int32_t* hidden_map,
                int64_t* slot_mapping, int32_t* sample_idx, void* X,
                uint32_t* err) {
  int32_t R, T, b;
  int rc;
  if (B < 0 || Kp < 0 || K < 1 || !err) return -1;
  if ((Kp >= 1) != (in_offsets == NULL)) return -1;
  if (mask_id < 0 || mask_id >= V) return -1;
  if (B == 0) {
    if (out_offsets) out_offsets[0] = 0;
    return 0;
  }
  if (Kp == 0) { /* prefill: offsets must partition the rows first */
    int ok = (in_offsets[0] == 0);
    for (b = 0; b < B; ++b)
      if (in_offsets[b + 1] - in_offsets[b] < 1) ok = 0;
    if (!ok) {
      *err |= ORC_ERR_OFFSETS;
      return 0;
    }
  }
  /* verification: logits hold Kp+1 rows per request (prefill: one, the
     last prompt row, whose argmax is the new token) */
  rc = oracle_verify_greedy(logits, logits_dtype, row_stride, B, Kp, V,
                            in_tokens, accepted_len, bonus_token, target_argmax);
  if (rc) return rc;
  rc = oracle_build_draft_batch(B, Kp, K, mask_id, in_offsets, in_tokens,
                                in_positions, accepted_len, bonus_token,
                                block_table, bt_width, block_size, out_offsets,
                                out_tokens, out_positions, is_rejected,
                                is_masked, hidden_map, slot_mapping, sample_idx,
                                err);
  if (rc) return rc;
  R = in_offsets ? in_offsets[B] : B * (Kp + 1);
  T = R + B * (K - 1);
  return oracle_assemble_draft_inputs(elt_of(x_dtype), H, V, T, R, emb,
                                      target_hidden, h_shared, out_tokens,
                                      hidden_map, is_masked, X, err);
}
