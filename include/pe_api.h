/*
 * pe_api.h -- C ABI of libpe.so: the per-step data path of P-EAGLE parallel
 * drafting on one GB300 (sm_103a): greedy verification, the fused
 * draft-batch rebuild and the drafter input assembly.
 *
 * Sources (page title -- section):
 *  [P1] "P-EAGLE: Faster LLM Inference with Parallel Speculative Decoding in
 *       vLLM" -- quick-read section (equation Input_i; acceptance length;
 *       rejected tokens mapped to -1) and the vLLM engineering listing
 *       (target hidden rows scattered to new slots, then MASK slots
 *       overwritten with the learned hidden state).
 *  [P2] "P-EAGLE: Parallel Speculative Decoding in vLLM" -- Step 2: Parallel
 *       Drafting; Fused Triton Kernel; Hidden State Management; KV Cache and
 *       CUDA Graphs.
 *  [P3] "并行草稿机制解析：从P-EAGLE到DSpark的投机采样加速" -- §1.2 (the
 *       target checks the drafts against its own distribution, accepts the
 *       ones that agree and replaces from the first disagreement, keeping
 *       its own output distribution).
 *
 * Notation.  Request b in [0,B).  Its target (verification) segment holds
 * n_b rows starting at input offset io_b; decode has n_b = K'+1 (the last
 * committed token, then drafts d_1..d_K'), the first step after prefill has
 * K' = 0 and n_b = prompt length.  Its output segment holds m_b = n_b+K-1
 * rows at output offset oo_b.  R = sum n_b, T = sum m_b = R + B(K-1).
 * The Kp+1 "verified rows" of a segment are its last Kp+1 rows; logits hold
 * exactly those rows, request-major: logits row b(Kp+1)+j.
 *
 * Conventions shared by every entry point:
 *  - All pointers not marked "host" are device pointers.  The caller owns
 *    every buffer; the library never allocates, frees or synchronises, and
 *    enqueues its work on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  Outputs are valid once the stream reaches that point.
 *  - The return value reports host-checkable argument errors only
 *    (pe_status); nothing is enqueued when it is not PE_OK.
 *  - Data errors found on the device never trap: the kernel ORs a PE_ERR_*
 *    bit into *err (a device word the caller zeroes and reads when it wants
 *    to) and writes the defined value stated for that case.
 *  - Integer outputs are exact.  Floating point only enters the argmax:
 *    values are compared numerically (-0.0 == +0.0), the lowest column wins
 *    ties; logits must not hold NaN.  (pe_verify_sampled is the exception:
 *    it decides in fp32 arithmetic, see there.)
 *  - Element types: PE_F32 (4 bytes) or PE_BF16 (2 bytes).  Embedding table,
 *    target hidden rows, h_shared and X share one element type.
 *  - Alignment: logits base, emb, target_hidden, h_shared and X must be
 *    16-byte aligned, the logits row stride (in bytes) and H*elt a multiple
 *    of 16 bytes; otherwise PE_EALIGN.
 */
#ifndef PE_API_H
#define PE_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pe_status {
  PE_OK = 0,
  PE_EINVAL = -1, /* NULL pointer, size out of range, inconsistent sizes */
  PE_EDTYPE = -2, /* element type is neither PE_F32 nor PE_BF16 */
  PE_EALIGN = -3, /* pointer / stride / row size not 16-byte aligned */
  PE_ECUDA = -4   /* the CUDA runtime reported an error at launch */
} pe_status;

typedef enum pe_dtype { PE_F32 = 0, PE_BF16 = 1 } pe_dtype;

/* Bits of the device error word. */
#define PE_ERR_TOKEN_RANGE 1u /* gathered token id outside [0,V): zero row   */
#define PE_ERR_BLOCK_RANGE 2u /* pos < 0 or pos/block_size >= bt_width: -1  */
#define PE_ERR_SLOT_RANGE 4u  /* accepted_len outside [0,Kp]: taken as 0    */
#define PE_ERR_OFFSETS 8u     /* in_offsets invalid: nothing is written     */
#define PE_ERR_MAP_RANGE 16u  /* hidden_map entry outside [0,T): skipped    */
#define PE_ERR_ROW_RANGE 64u  /* readout row index outside [0,rows): -1     */
#define PE_ERR_TIMEOUT 32u    /* a bounded wait gave up (a bulk-copy tile
                                 waiting for its own loads, the single
                                 pass's collection of its chunk keys, the
                                 sampled stats merge); outputs incomplete;
                                 never expected with a zeroed workspace    */
/* Raised only by the checked build (libpe_checked.so: the same entry points
 * compiled with PE_CHECKED, for debugging; slower).  Neither traps. */
#define PE_ERR_NAN 128u       /* a logits row read by the greedy argmax
                                 (pe_step, pe_step_early_exit,
                                 pe_verify_greedy, pe_draft_readout) holds a
                                 NaN; the outputs are then undefined        */
#define PE_ERR_INTERNAL 256u  /* an internal index invariant of the fused
                                 step failed; the access was skipped (never
                                 expected: a library bug)                  */
/* Raised by every build. */
#define PE_ERR_WORKSPACE 512u /* a workspace counter or hand-off word held a
                                 value outside its legal range: the
                                 workspace was not zero when the call
                                 started (never zero-filled, shared by
                                 calls that overlap on the GPU, or left
                                 dirty by an earlier call that raised
                                 PE_ERR_TIMEOUT or PE_ERR_WORKSPACE).  The
                                 call skipped the work the bad value
                                 governs: outputs are incomplete, and the
                                 workspace must be zero-filled again before
                                 its next use.  Detection is by range: a
                                 corruption that keeps every value inside
                                 its legal range goes unseen.              */

/* Limits checked on the host. */
#define PE_MAX_KP 255 /* previous draft depth K'  */
#define PE_MAX_K 256  /* new draft depth K        */

/* Bytes of scratch that pe_verify_greedy, pe_draft_readout (with
 * logits_rows = B = n), pe_step and pe_step_early_exit need for a batch with
 * `logits_rows` = B*(Kp+1) logits rows and B requests.  The caller
 * allocates it once, zero-filled, and may reuse it for every later call of
 * any size up to those; each call leaves it zeroed again on completion,
 * unless it raised PE_ERR_TIMEOUT or PE_ERR_WORKSPACE: after either bit the
 * caller zero-fills the workspace again (a caller that does not tell the
 * bits apart may simply do so after any bit).  Calls that may run
 * concurrently need separate workspaces. */
size_t pe_workspace_bytes(int32_t logits_rows, int32_t B);

/* Greedy verification [P1 quick-read: acceptance length].
 *  logits      [B*(Kp+1), V] of `dtype`, row stride `row_stride` elements.
 *  in_tokens   [B*(Kp+1)] int32: row b(Kp+1)+j+1 holds draft d_{j+1} of
 *              request b (row b(Kp+1) holds the last committed token and is
 *              not read).  May be NULL when Kp == 0.
 *  accepted_len[B] out: a_b = first j < Kp with argmax(row j) != d_{j+1},
 *              or Kp when every draft matches.
 *  bonus_token [B] out: argmax of row a_b (the target's own next token).
 *  target_argmax [B*(Kp+1)] out, or NULL: every row's argmax.
 *  workspace   pe_workspace_bytes(B*(Kp+1), B) bytes, zeroed (see above).
 *  err         device error word: PE_ERR_WORKSPACE; PE_ERR_TIMEOUT (the
 *              single pass's bounded wait, never expected); PE_ERR_NAN in
 *              the checked build.
 * B == 0 enqueues nothing. */
int pe_verify_greedy(const void* logits, int dtype, int64_t row_stride,
                     int32_t B, int32_t Kp, int32_t V, const int32_t* in_tokens,
                     int32_t* accepted_len, int32_t* bonus_token,
                     int32_t* target_argmax, void* workspace, uint32_t* err,
                     void* stream);

/* Drafter readout [P2 Step 2: all positions pass through the drafter's N
 * layers and LM head, which predicts t_1..t_K]: greedy draft tokens.
 *   out_tokens[i] = argmax over the first V columns of logits row
 *                   sample_idx[i] (row i when sample_idx is NULL), lowest
 *                   column on ties
 *  logits      [rows, V'] of `dtype`, row stride `row_stride` elements:
 *              either the drafter's logits for every output slot ([T, V],
 *              read through sample_idx from pe_build_draft_batch) or only for
 *              the sampled rows ([B*K, V], sample_idx NULL).
 *  sample_idx  [n] int32 or NULL (then n <= rows).  An index outside
 *              [0, rows) gives out_tokens[i] = -1 and PE_ERR_ROW_RANGE.
 *  workspace   pe_workspace_bytes(n, n) bytes, zeroed (as for pe_step).
 * n == 0 enqueues nothing. */
int pe_draft_readout(const void* logits, int dtype, int64_t row_stride,
                     int32_t rows, int32_t V, const int32_t* sample_idx,
                     int32_t n, int32_t* out_tokens, void* workspace,
                     uint32_t* err, void* stream);

/* Bytes of scratch that pe_verify_sampled needs for B requests of depth Kp
 * (any V).  Allocated once, zero-filled; every call leaves it zeroed again
 * (except after PE_ERR_TIMEOUT or PE_ERR_WORKSPACE, as above), so it serves
 * every later call with B and Kp up to those. */
size_t pe_workspace_bytes_sampled(int32_t B, int32_t Kp);

/* Rejection-sampling verification [P3 §1.2], read as the acceptance rule of
 * speculative sampling, for callers that sample rather than take argmax.
 * With T = temperature, for request b and draft j < Kp:
 *   p_j = softmax(target row b(Kp+1)+j / T),  q_j = softmax(draft row
 *   b*Kp+j / T),  x = in_tokens[b(Kp+1)+j+1]  (the draft d_{j+1});
 *   draft j is accepted when u_accept[b*Kp+j] * q_j(x) < p_j(x)
 *   (probability min(1, p/q) for u uniform in [0,1)); a token outside
 *   [0,V) is rejected.
 *   accepted_len[b] = a_b = the first rejected j, or Kp.
 *   bonus_token[b] = a draw from max(0, p_a - q_a) normalised when a_b < Kp
 *   (from p_a when that residual is zero everywhere), from p_Kp (target
 *   row b(Kp+1)+Kp) when a_b = Kp.
 * Draws are Gumbel-max: the column maximising s(v) + G_b(v), s(v) = log of
 * the (unnormalised) weight of column v, G_b(v) = -log(-log(U)),
 * U = ((w >> 9) + 0.5) / 2^23 (exact in fp32) and w = word (v mod 4) of Philox4x32-10
 * (Salmon et al., SC'11) at counter (v/4, b, 0, 0) under the key (low,
 * high word of `seed`).  Only the accept/reject coins come from the caller.
 *  target_logits [B*(Kp+1), V], row stride target_stride elements.
 *  draft_logits  [B*Kp, V], row stride draft_stride (the drafter's logits
 *                at the drafted positions); NULL allowed when Kp == 0.
 *  in_tokens     [B*(Kp+1)] int32 as for pe_verify_greedy; u_accept
 *                [B*Kp] fp32 in [0,1).  Both may be NULL when Kp == 0.
 *  temperature   > 0 (PE_EINVAL otherwise); logits must be finite.
 *  workspace     pe_workspace_bytes_sampled(B, Kp) bytes, zeroed.
 *  err           device error word: PE_ERR_TIMEOUT when a bounded wait of
 *                the statistics merge gave up (never expected with a zeroed
 *                workspace); PE_ERR_WORKSPACE as above.
 * Arithmetic is fp32 in the log2 domain (the hardware's approximate ex2 and
 * lg2 instructions; near U = 1 the noise uses a short series of
 * -log2(1 - t) instead): accept decisions and draws agree with
 * an exact evaluation except where p(x) - u q(x), or the gap between the
 * two best Gumbel scores, is within rounding of zero.  Two kernel launches;
 * B == 0 enqueues nothing. */
int pe_verify_sampled(const void* target_logits, const void* draft_logits,
                      int dtype, int64_t target_stride, int64_t draft_stride,
                      int32_t B, int32_t Kp, int32_t V,
                      const int32_t* in_tokens, const float* u_accept,
                      float temperature, uint64_t seed, int32_t* accepted_len,
                      int32_t* bonus_token, void* workspace, uint32_t* err,
                      void* stream);

/* Draft-batch rebuild [P2 Fused Triton Kernel; KV Cache and CUDA Graphs].
 * For request b with bonus slot s_b = n_b-1-Kp+a_b and slot k of its output
 * segment (t = oo_b + k):
 *   k <  s_b        token in[io_b+k+1] (shift by one), position pos[io_b+k]
 *   k == s_b        token bonus_b (next-token prediction), position pos[io_b+s_b]
 *   s_b < k < n_b   rejected: is_rejected=1, position pos[io_b+k], token
 *                   in[io_b+k+1] for k < n_b-1 and mask_id for k = n_b-1
 *   n_b <= k < m_b  MASK: is_masked=1, token mask_id,
 *                   position pos[io_b+s_b] + (k-n_b+1)
 *   slot_mapping[t] = -1 when rejected, else
 *     block_table[b*bt_width + pos/block_size]*block_size + pos%block_size
 *     (-1 and PE_ERR_BLOCK_RANGE when pos < 0 or pos/block_size >= bt_width)
 *   hidden_map[io_b+k] = oo_b+k for k < n_b
 *   sample_idx[b*K + 0] = oo_b+s_b, sample_idx[b*K + i] = oo_b+n_b+i-1
 *   out_offsets[b] = oo_b (exclusive scan of m_b), out_offsets[B] = T
 *  in_offsets  [B+1] int32, or NULL for fixed segments n_b = Kp+1 (decode).
 *              When given: in_offsets[0] = 0, in_offsets[B] = R and every
 *              n_b >= Kp+1, else PE_ERR_OFFSETS and nothing is written.
 *  R           total input rows (host): B*(Kp+1) when in_offsets is NULL.
 *  in_tokens, in_positions [R] int32.
 *  accepted_len [B] int32 (NULL: all 0); values outside [0,Kp] count as 0
 *              and raise PE_ERR_SLOT_RANGE.
 *  bonus_token [B] int32.
 *  block_table [B, bt_width] int32 physical block ids.
 *  outputs: out_offsets[B+1], out_tokens[T], out_positions[T] int32;
 *           is_rejected[T], is_masked[T] uint8; hidden_map[R] int32;
 *           slot_mapping[T] int64; sample_idx[B*K] int32 or NULL. */
int pe_build_draft_batch(int32_t B, int32_t Kp, int32_t K, int32_t mask_id,
                         int32_t R, const int32_t* in_offsets,
                         const int32_t* in_tokens, const int32_t* in_positions,
                         const int32_t* accepted_len, const int32_t* bonus_token,
                         const int32_t* block_table, int32_t bt_width,
                         int32_t block_size, int32_t* out_offsets,
                         int32_t* out_tokens, int32_t* out_positions,
                         uint8_t* is_rejected, uint8_t* is_masked,
                         int32_t* hidden_map, int64_t* slot_mapping,
                         int32_t* sample_idx, uint32_t* err, void* stream);

/* Drafter input assembly [P1 equation Input_i and the engineering listing;
 * P2 Hidden State Management].
 *   X[t, 0:H]  = emb[out_tokens[t]]   (zeros + PE_ERR_TOKEN_RANGE when the
 *                token is outside [0,V))
 *   X[t, H:2H] = h_shared                         when is_masked[t]
 *              = target_hidden[i] with hidden_map[i] == t   otherwise
 * i.e. the target rows are scattered through hidden_map and the masked slots
 * then take h_shared.  hidden_map must not repeat a slot; entries outside
 * [0,T) are skipped with PE_ERR_MAP_RANGE; an unmasked slot that no entry
 * names keeps its previous hidden half.
 *  emb [V,H], target_hidden [R,H], h_shared [H], X [T,2H] of `dtype`;
 *  out_tokens[T], hidden_map[R] int32; is_masked[T] uint8. */
int pe_assemble_draft_inputs(int dtype, int32_t H, int32_t V, int32_t T,
                             int32_t R, const void* emb,
                             const void* target_hidden, const void* h_shared,
                             const int32_t* out_tokens,
                             const int32_t* hidden_map,
                             const uint8_t* is_masked, void* X, uint32_t* err,
                             void* stream);

/* The whole step in one launch: pe_verify_greedy, then pe_build_draft_batch
 * on its result, then pe_assemble_draft_inputs, with identical outputs.
 * Kp >= 1: decode; in_offsets must be NULL, R = B*(Kp+1).
 * Kp == 0: first drafting step after prefill; in_offsets [B+1] required,
 * logits hold one row per request (its last prompt row), whose argmax is
 * the new token placed at the next-token-prediction slot.
 * Optional outputs (may be NULL): target_argmax, sample_idx. */
typedef struct pe_step_args {
  int32_t B, Kp, K, V, H, R;
  int32_t mask_id, bt_width, block_size;
  int32_t logits_dtype, x_dtype;
  int64_t logits_row_stride; /* elements */
  /* inputs */
  const void* logits;
  const int32_t* in_offsets;
  const int32_t* in_tokens;
  const int32_t* in_positions;
  const int32_t* block_table;
  const void* emb;
  const void* target_hidden;
  const void* h_shared;
  /* outputs */
  int32_t* accepted_len;
  int32_t* bonus_token;
  int32_t* target_argmax;
  int32_t* out_offsets;
  int32_t* out_tokens;
  int32_t* out_positions;
  uint8_t* is_rejected;
  uint8_t* is_masked;
  int32_t* hidden_map;
  int64_t* slot_mapping;
  int32_t* sample_idx;
  void* X;
  /* scratch and error word */
  void* workspace; /* pe_workspace_bytes(B*(Kp+1), B), zeroed */
  uint32_t* err;
} pe_step_args;

int pe_step(const pe_step_args* args /* host */, void* stream);

/* The whole step with early exit [P1 quick-read: acceptance length]: the
 * verified rows of a request are read in order and the rows after its
 * first mismatch are not read at all (rows of every request are streamed
 * row 0 first, then row 1, ...; a chunk whose request already has a known
 * earlier mismatch is skipped).  Every output equals pe_step's, except
 * target_argmax, which holds each request's rows 0..a_b and -1 for the rows
 * after a_b.  Same arguments and workspace as pe_step; Kp <= 31 (one bit per
 * verified row), else PE_EINVAL.  It pays off when many requests share the
 * step (their rows interleave); with few requests the rows of a request
 * serialise, so when the logits take at most pe_tuning.early_full_read_mb
 * MiB (default 128) this call reads every row instead, with the same
 * outputs (target_argmax still -1 after a_b).  The early-exit reading runs
 * the register-streaming kernel (pe_tuning.variant does not apply); the
 * full read follows pe_tuning.variant. */
int pe_step_early_exit(const pe_step_args* args /* host */, void* stream);

/* pe_step for callers that cannot allocate device memory at all, not even
 * the small scratch above: code running under a memory manager that owns
 * the whole device, plug-ins that only receive the tensors they work on,
 * loops that must not hit the device-wide synchronisation of cudaMalloc /
 * cudaFree.  The pages have no counterpart of this entry point.
 * Outputs are identical to pe_step's; args->workspace is ignored (may be
 * NULL).  The scratch is a fixed array of PE_NOALLOC_WS_BYTES bytes inside
 * the library, held by every GPU that loads it until the process exits.
 *  - The first call on a device looks up the array's device address (and
 *    may load the library's GPU code there).  The address is kept for the
 *    life of the process;
 *    a program that resets a device (cudaDeviceReset) must not call this
 *    entry point on that device afterwards (the kept address would no
 *    longer be the array's).
 *  - Each call enqueues a memset clearing the scratch it needs, then the
 *    step; if pe_step then rejects the arguments, the memset has still been
 *    enqueued (it touches only the library's own array).
 *  - A batch that needs more than PE_NOALLOC_WS_BYTES of scratch
 *    (pe_workspace_bytes(B*(Kp+1), B)) is rejected with PE_EINVAL.
 *  - Every call shares the array: calls whose work overlaps on the GPU
 *    race on it, so order them (one stream, or events between streams).
 *  - Nothing is allocated or freed. */
#define PE_NOALLOC_WS_BYTES 65536
int pe_step_noalloc(const pe_step_args* args /* host */, void* stream);

/* Launch-shape knobs of the fused step (process-wide; defaults chosen by
 * measurement).  Zero fields keep the current value. */
typedef struct pe_tuning {
  int32_t ctas_per_sm;     /* resident CTAs per SM for the persistent grid */
  int32_t chunk_batches;   /* max 32 KiB load batches per argmax unit      */
  int32_t rows_per_unit;   /* X rows per copy unit                         */
  int32_t variant;         /* how copy tiles move X's half rows (the argmax
                              streams through registers either way):
                              1: 16-byte loads and stores through registers
                              (default); 2: bulk asynchronous copies
                              (cp.async.bulk) global -> shared -> global,
                              one thread issuing them, with as many rows
                              per tile as a 48 KiB staging buffer holds
                              (register copies when not even one fits) */
  int32_t queue_order;     /* 2: argmax chunks first, every copy tile after
                              (default: the tiles fill the drain, and a
                              request's last verified-row tile, not its
                              verdict, usually writes the bonus row);
                              1: copy tiles of the verified rows first, then
                              the argmax chunks, then the other copy tiles
                              (same outputs; the verdict usually writes the
                              bonus row) */
  int32_t early_full_read_mb; /* pe_step_early_exit reads every row (the
                              full-read kernel, outputs unchanged) when the
                              logits take at most this many MiB: with few
                              requests the serial row waves cost more than
                              the extra bytes.  Default 128; -1 sets 0
                              (always the early-exit kernel) */
  int32_t single_pass;     /* 1 (default): a step whose work units fit one
                              per co-resident CTA (few requests) runs as a
                              cooperative launch in which every CTA does one
                              unit and leaves: chunk keys go to slots in the
                              workspace, and the CTA of a request's last
                              chunk collects them (a bounded wait on the
                              other CTAs, all resident by construction)
                              instead of merging and counting through
                              atomics; same outputs.  -1: never */
} pe_tuning;
int pe_get_tuning(pe_tuning* out /* host */);
int pe_set_tuning(const pe_tuning* in /* host */);

/* Launch-latency reference (no counterpart on the pages: a measuring aid).
 * Launches `ctas` CTAs of 256 threads on `stream` that do no work, except
 * that thread 0 of CTA 0 follows `hops` dependent 4-byte loads through
 * `chain` [n] int32 (entry i holds the index of the next entry; an index
 * outside [0, n) continues from entry 0) and stores the last index to
 * *out.  hops = 0: an empty launch (chain and out may be NULL).  At small
 * batch the fused step is a chain of dependent round trips, and this is the
 * floor it is measured against: an empty launch of the step's grid, plus
 * one round trip to global memory. */
int pe_latency_floor(int32_t ctas, int32_t hops, const int32_t* chain, int32_t n,
                     int32_t* out, void* stream);

/* Human-readable name of a pe_status value. */
const char* pe_status_str(int status);

#ifdef __cplusplus
}
#endif
#endif /* PE_API_H */
