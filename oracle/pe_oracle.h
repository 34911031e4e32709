/*
 * CPU oracle for the P-EAGLE parallel-drafting step (verify -> rebuild ->
 * assemble).  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product path never does.  It
 * shares no code, header or constant with the CUDA library.
 *
 * Every function is the plain definition, one element at a time, single
 * threaded.  Floating point enters only through the argmax, which compares
 * values widened to double (exact for fp32 and bf16 inputs).
 */
#ifndef PE_ORACLE_H
#define PE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of logits and of the embedding / hidden / X tensors */
#define ORC_F32 0
#define ORC_BF16 1

/* error-word bits the oracle raises (same meanings as the library's) */
#define ORC_ERR_TOKEN_RANGE 1u /* a gathered token id is outside [0, V)      */
#define ORC_ERR_BLOCK_RANGE 2u /* position < 0 or position/bs >= table width */
#define ORC_ERR_SLOT_RANGE 4u  /* accepted length outside [0, K']            */
#define ORC_ERR_OFFSETS 8u     /* segment offsets are not a valid partition  */
#define ORC_ERR_MAP_RANGE 16u  /* hidden-state mapping outside [0, T)        */
#define ORC_ERR_ROW_RANGE 64u  /* readout row index outside [0, rows)        */

/* Row argmax, lowest index on ties, -0.0 == +0.0.  out[rows]. */
int oracle_argmax_rows(const void* logits, int dtype, int64_t row_stride,
                       int32_t rows, int32_t V, int32_t* out);

/* Greedy drafter readout: out[i] = argmax of logits row sample_idx[i]
 * (row i when sample_idx is NULL), lowest index on ties; an index outside
 * [0, rows) gives -1 and raises ORC_ERR_ROW_RANGE. */
int oracle_draft_readout(const void* logits, int dtype, int64_t row_stride,
                         int32_t rows, int32_t V, const int32_t* sample_idx,
                         int32_t n, int32_t* out, uint32_t* err);

/* Greedy verification over logits[B*(Kp+1), V] (row r of request b is
 * b*(Kp+1)+j).  tokens[B*(Kp+1)]: row j+1 of request b holds draft d_{j+1}.
 * tokens may be NULL when Kp == 0.  target_argmax may be NULL. */
int oracle_verify_greedy(const void* logits, int dtype, int64_t row_stride,
                         int32_t B, int32_t Kp, int32_t V,
                         const int32_t* tokens, int32_t* accepted_len,
                         int32_t* bonus_token, int32_t* target_argmax);

/* Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): out = the counter
 * after ten rounds under the key. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]);

/* Rejection-sampling verification (the acceptance rule of speculative
 * sampling).  For request b and draft j (0 <= j < Kp), with
 * p = softmax(target row b(Kp+1)+j / temperature), q = softmax(draft row
 * b*Kp+j / temperature) and x = tokens[b(Kp+1)+j+1]: the draft is accepted
 * when u_accept[b*Kp+j] * q(x) < p(x).  At the first rejection a_b = j and
 * the bonus is drawn from max(0, p - q) (from p when that is all zero);
 * when every draft is accepted a_b = Kp and the bonus is drawn from
 * softmax(target row b(Kp+1)+Kp / temperature).  Draws use the Gumbel-max
 * rule with noise -log(-log(U)), U = ((w >> 9) + 0.5) / 2^23, w = word (i mod 4)
 * of Philox4x32-10(counter = (i / 4, b, 0, 0), key = (seed lo, seed hi)).
 * A draft token outside [0, V) is rejected. */
int oracle_verify_sampled(const void* target_logits, const void* draft_logits,
                          int dtype, int64_t target_stride,
                          int64_t draft_stride, int32_t B, int32_t Kp,
                          int32_t V, const int32_t* tokens,
                          const float* u_accept, float temperature,
                          uint64_t seed, int32_t* accepted_len,
                          int32_t* bonus_token);

/* Draft-batch rebuild.  in_offsets[B+1] (NULL: fixed segments of Kp+1
 * rows); accepted_len[B] (NULL: all zero).  Outputs sized from
 * R = in_offsets[B] and T = R + B*(K-1).  sample_idx[B*K] may be NULL. */
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
                             int32_t* sample_idx, uint32_t* err);

/* Drafter input X[T, 2H] = emb(out_tokens[t]) (+) hidden, hidden half by
 * scatter of target rows through hidden_map, then h_shared in masked slots.
 * elt = bytes per element (4 or 2).  Rows neither mapped nor masked keep
 * their previous hidden half. */
int oracle_assemble_draft_inputs(int32_t elt, int32_t H, int32_t V, int32_t T,
                                 int32_t R, const void* emb,
                                 const void* target_hidden,
                                 const void* h_shared,
                                 const int32_t* out_tokens,
                                 const int32_t* hidden_map,
                                 const uint8_t* is_masked, void* X,
                                 uint32_t* err);

/* Full step: verify (logits rows B*(Kp+1)), rebuild, assemble.
 * Kp >= 1: decode, in_offsets must be NULL.  Kp == 0: prefill, in_offsets
 * required and logits hold one row per request (its last prompt row). */
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
                uint32_t* err);

#ifdef __cplusplus
}
#endif
#endif
