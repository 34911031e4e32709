// Fused P-EAGLE drafting step on one GPU: greedy verification, draft-batch
// rebuild and drafter input assembly in a single persistent launch
// (pe_step); the same with early exit (pe_step_early_exit); verification
// alone (pe_verify_greedy); the drafter readout (pe_draft_readout).
//
// Sources (page title -- section):
//  "P-EAGLE: Parallel Speculative Decoding in vLLM" -- Fused Triton Kernel
//    (copy token ids / positions, insert the bonus token, fill MASK slots,
//    emit rejected / masked masks and the hidden-state mapping in one pass);
//    Hidden State Management (target rows to their new slots, learned hidden
//    state broadcast into MASK slots); KV Cache and CUDA Graphs (rejected
//    slots -> -1).
//  "P-EAGLE: Faster LLM Inference with Parallel Speculative Decoding in
//    vLLM" -- quick-read section: Input_1 = emb(new) (+) h_context,
//    Input_i = emb(mask) (+) h_shared for 2 <= i <= K; acceptance length.
//
// Design (one launch, no grid-wide barrier, no CTA ever waits for another):
//  * A persistent grid pulls work units from a counter in the workspace.
//    Units [0, n_arg) are argmax chunks (row r, chunk c) of the logits, in
//    row order; units [n_arg, n_units) copy tiles of X rows, first those of
//    the verified rows, then those of the prompt and MASK rows (unit_at
//    gives the order in which they are handed out).
//  * Argmax chunk: 256 threads stream 32 KiB batches with 16-byte loads
//    (eight per thread in flight), keep the thread's running maximum and the
//    column where it first appears, reduce (value, column) keys with warp
//    shuffles, and merge into the row's key with one 64-bit atomicMax.
//  * The CTA whose chunk completes a request (per-request counter) runs
//    that request's epilogue, the verdict: accepted length, bonus token and
//    the rebuild metadata of its verified and MASK slots.  It copies no
//    embedding rows.
//  * Copy tiles write all of X: the hidden half of every row, MASK rows
//    whole (emb(mask) (+) h_shared), prompt rows whole (prefill) with their
//    metadata, and the embedding half of every verified slot with the token
//    it has unless it is the bonus slot.  The bonus row alone depends on the
//    verdict: whichever of the verdict and the request's last verified-row
//    tile comes second (one atomic each on the request's hand-off word)
//    writes E[bonus] over the tile's default.  Every other byte of X has one
//    writer.
//  * Each CTA takes one index past the end of the queue and leaves; the
//    claim that returns the last index resets the counter for the next call.
//  * Copy tiles move their half rows through registers (16-byte loads and
//    stores), or, with pe_tuning.variant = 2, through shared memory with
//    bulk asynchronous copies (one thread issues a load per half row into a
//    staging buffer, waits on the CTA's barrier, and issues the bulk stores
//    into X).
//  * Workspace words are checked against their legal ranges as they are
//    used (a unit index past the queue, a count past its total, a hand-off
//    word or state word with bits no call sets, a row key whose column is
//    outside the vocabulary); a bad value raises PE_ERR_WORKSPACE and the
//    work it governs is skipped, so a dirty workspace never sends an access
//    out of bounds.
//  * Early exit reads a request's rows in order and skips the rows after a
//    known mismatch (step_kernel_early); with a small logits footprint the
//    host serves it with the full read instead, the epilogue writing -1 to
//    target_argmax after a_b.
#include "pe_argmax.cuh"
#include "pe_internal.cuh"
#include "pe_tma.cuh"
#include "pe_workspace.cuh"

namespace pe {

struct StepParams {
  int B, Kp, K, V, H, R, T, mask_id, bt_width, block_size;
  int full;               // 1: rebuild + assemble too; 0: verification only
  int nvh;                // 16-byte vectors per half row of X
  int bulk_rows;          // bulk-copy tiles: X rows the staging buffer holds
  long long row_bytes;    // logits row stride in bytes
  int nvec, tail;         // whole 16-byte vectors per logits row, leftover elements
  int chunk_vecs, C, Rl;  // argmax chunking: vectors per chunk, chunks per row, rows
  int n_arg_units, rows_per_unit, n_copy_units, n_units;
  int rv, n_vtile;        // verified rows B(K'+1); copy tiles over them
  int mask_unread;        // target_argmax -1 after a_b (early exit served by a full read)
  int vfirst;             // 1: those tiles are handed out before the argmax chunks
  const void* logits;
  const int32_t* row_index;  // logits row of argmax row r (NULL: r itself)
  int rows_total;            // logits rows addressable through row_index
  const int32_t* in_offsets;
  const int32_t* in_tokens;
  const int32_t* in_positions;
  const int32_t* block_table;
  const uint4* emb;
  const uint4* hidden;
  const uint4* h_shared;
  int32_t* accepted_len;
  int32_t* bonus_token;
  int32_t* target_argmax;
  int32_t* out_offsets;
  int32_t* out_tokens;
  int32_t* out_positions;
  uint8_t* is_rejected;
  uint8_t* is_masked;
  int32_t* hidden_map;
  long long* slot_mapping;
  int32_t* sample_idx;
  uint4* X;
  uint32_t* sched;
  uint32_t* count;
  unsigned long long* keys;
  unsigned long long* state;  // early exit: per-request done / match bits
  unsigned long long* xfer;   // per-request bonus-row hand-off word
  uint32_t* rcount;           // early exit: finished chunks per row
  int32_t* amax_ws;           // early exit: argmax of each completed row
  unsigned long long* slots;  // single pass: chunk key of each argmax unit
  uint32_t* err;
};

enum SegMode { kSkip = 0, kCopy = 1, kZero = 2 };

struct SharedState {
  unsigned long long red[kWarps];
  unsigned long long rowkey[PE_MAX_KP + 1];  // single pass: the rows' keys
  uint64_t bar;                // bulk-copy tiles: completion of the tile's loads
  int unit;
  int last;
  int first;
  int amax[PE_MAX_KP + 1];
  int tok[PE_MAX_KP + 1];
  int pos[PE_MAX_KP + 1];
  const uint4* src[2 * kMaxRowsPerUnit];
  uint4* dst[2 * kMaxRowsPerUnit];
  int mode[2 * kMaxRowsPerUnit];
  int vreq[kMaxRowsPerUnit];   // copy tile: request of each verified row
  int vrow0[kMaxRowsPerUnit];  // ... and the X row of its verified slot 0
  int nbonus;                  // bonus rows this tile writes
  int brow[kMaxRowsPerUnit];
  int btok[kMaxRowsPerUnit];
  int xwrite;                  // epilogue: this verdict writes the bonus row
};

// Hand-off word of a request (workspace xfer[b]): verified rows whose
// default embedding half a copy tile has written (bits 0-15), verdict taken
// (bit 16), accepted length (bits 17-24), bonus token (bits 32-63).
constexpr unsigned long long kXferCount = 0xffffull;
constexpr unsigned long long kXferVerdict = 1ull << 16;

// A hand-off word as a legal call can leave it for the side that updates it
// next: the tiles' count below K'+1 (a tile adding its rows) or at most K'+1
// (the verdict), bits 25-31 clear, and either no verdict yet (nothing above
// the count) or, for a tile, a verdict with a <= K'.  Anything else means the
// workspace was not zero when the call started.
__device__ __forceinline__ bool xfer_legal(unsigned long long w, int Kp, bool tile_side) {
  const unsigned long long cnt = w & kXferCount;
  if (tile_side ? cnt >= (unsigned long long)(Kp + 1) : cnt > (unsigned long long)(Kp + 1))
    return false;
  if (w & 0xfe000000ull) return false;
  if (!(w & kXferVerdict)) return (w >> 17) == 0ull;
  return tile_side && ((w >> 17) & 0xffull) <= (unsigned long long)Kp;
}

// Unit handed out at position q of the queue.  vfirst: the copy tiles of
// the verified rows first, then the argmax chunks, then the other copy tiles
// (prompt and MASK rows), so that a verified row's default embedding half is
// normally written before its request's verdict.  Otherwise (the default,
// measured faster): the argmax chunks, then every copy tile, which fill the
// drain at the end of the step.
__device__ __forceinline__ int unit_at(const StepParams& p, int q) {
  if (!p.vfirst) return q;  // argmax chunks, then every copy tile
  if (q < p.n_vtile) return p.n_arg_units + q;
  if (q < p.n_vtile + p.n_arg_units) return q - p.n_vtile;
  return q;
}

// Logits row read for argmax row r, or nullptr when an index given through
// row_index is outside [0, rows_total).
__device__ __forceinline__ const char* logits_row(const StepParams& p, int r) {
  const int pr = p.row_index ? __ldg(p.row_index + r) : r;
  if (pr < 0 || pr >= p.rows_total) return nullptr;
  return static_cast<const char*>(p.logits) + (long long)pr * p.row_bytes;
}

__device__ __forceinline__ int seg_begin(const StepParams& p, int b) {
  return p.in_offsets ? __ldg(p.in_offsets + b) : b * (p.Kp + 1);
}

// ------------------------------------------------------------------ epilogue
// Runs in the CTA that finished the last argmax chunk of request b.  Its
// global traffic is two dependent round trips: (1) the row keys (exchanged
// with 0, leaving the workspace clean), the drafts and the positions of the
// verified rows, all at once; (2) after the verdict, the hand-off atomic and
// the block-table entries of the kept slots with the metadata stores; then,
// only when the request's verified-row tiles are already done, the bonus
// row's embedding half.
// Where the row results come from:
//  kKeysInWorkspace: the rows' merged keys in the workspace (exchanged with
//    0) and the request's unit count (reset);
//  kRowsSettled: early exit -- the accepted length `a_known` is already
//    settled; rows 0..a_known are read from the completed-row results and
//    later rows, which may never have been read, report -1;
//  kKeysInShared: single pass -- the collecting CTA left the rows' keys in
//    sh.rowkey and the drafts and positions in sh.tok / sh.pos.
enum KeySource { kKeysInWorkspace = 0, kRowsSettled = 1, kKeysInShared = 2 };

template <int SRC = kKeysInWorkspace>
__device__ __forceinline__ void request_epilogue(const StepParams& p, SharedState& sh,
                                                 int b, int a_known = -1) {
  constexpr bool EARLY = SRC == kRowsSettled;
  const int tid = threadIdx.x;
  const int Kp = p.Kp;
  const int nr = Kp + 1;  // verified rows (<= 256 = threads)
  const int io = seg_begin(p, b);
  const int n = seg_begin(p, b + 1) - io;
  const int vb = n - 1 - Kp;  // segment row of the first verified row
  if (tid < nr) {
    if (SRC == kRowsSettled) {
      sh.amax[tid] = tid <= a_known ? __ldcg(p.amax_ws + (long long)b * nr + tid) : -1;
    } else if (SRC == kKeysInWorkspace) {
      const unsigned long long k = atomicExch(p.keys + (long long)b * nr + tid, 0ull);
      const uint32_t col = key_col(k);
      // a merged key names a column of the row (0: a readout row outside the
      // logits, which holds no element)
      if (k != 0ull && col >= (uint32_t)p.V) atomicOr(p.err, PE_ERR_WORKSPACE);
      sh.amax[tid] = (int)col;
    } else {
      sh.amax[tid] = (int)key_col(sh.rowkey[tid]);
    }
    if (SRC != kKeysInShared) {
      if (tid < Kp) sh.tok[tid] = __ldg(p.in_tokens + io + vb + tid + 1);  // draft d_{tid+1}
      if (p.full) sh.pos[tid] = __ldg(p.in_positions + io + vb + tid);
    }
  }
  if (tid == 0) {
    sh.first = EARLY ? a_known : Kp;
    if (SRC == kKeysInWorkspace) atomicExch(p.count + b, 0u);
  }
  __syncthreads();
  // accepted length: first draft that differs from the target's choice
  if (!EARLY && tid < Kp && sh.amax[tid] != sh.tok[tid]) atomicMin(&sh.first, tid);
  __syncthreads();
  const int a = sh.first;
  if (p.target_argmax && tid < nr)
    p.target_argmax[(long long)b * nr + tid] = p.mask_unread && tid > a ? -1 : sh.amax[tid];
  const int bonus = sh.amax[a];
  if (!p.full) {
    if (tid == 0) {
      if (p.accepted_len) p.accepted_len[b] = a;
      p.bonus_token[b] = bonus;
    }
    return;
  }
  const int oo = io + b * (p.K - 1);
  const int s = vb + a;        // next-token-prediction slot
  const int pos_s = sh.pos[a];
  if (tid == 0) {
    p.accepted_len[b] = a;
    p.bonus_token[b] = bonus;
    p.out_offsets[b] = oo;
    if (b == p.B - 1) p.out_offsets[p.B] = p.T;
  }
  // Token of verified slot j (segment row vb + j): the bonus at j == a, the
  // shifted draft d_{j+1} elsewhere, and the MASK id in the last row when it
  // is rejected.
  auto slot_token = [&](int j) { return j == a ? bonus : (j < Kp ? sh.tok[j] : p.mask_id); };
  // Embedding halves of the verified rows: the copy tiles write each one
  // with the token it has unless it is the bonus slot; only the bonus row
  // depends on the verdict, and whichever of this verdict and the request's
  // last verified-row tile comes second writes it (one atomic each on the
  // request's hand-off word).  Tokens outside the table give zero halves
  // (written by the tiles) and an error bit (raised here).
  // The hand-off atomic, the block-table loads of the metadata and (when
  // this verdict writes it) the bonus row's loads are independent, so they
  // share round trips.
  if (tid < nr) {
    const int tok = slot_token(tid);
    if (tok < 0 || tok >= p.V) atomicOr(p.err, PE_ERR_TOKEN_RANGE);
  }
  unsigned long long old = 0ull;
  if (tid == 0)
    old = atom_or_acquire(p.xfer + b, kXferVerdict | ((unsigned long long)a << 17) |
                                          ((unsigned long long)(uint32_t)bonus << 32));
  // the bonus row's first 2*kThreads vectors, read now in case this verdict
  // is the one to write it (the embedding table never changes)
  const bool bok = bonus >= 0 && bonus < p.V;
  const uint4* bsrc = p.emb + (long long)bonus * p.nvh;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint4 x1 = bok && tid < p.nvh ? __ldg(bsrc + tid) : zero;
  const uint4 x2 = bok && kThreads + tid < p.nvh ? __ldg(bsrc + kThreads + tid) : zero;
  // rebuild metadata of the verified rows (j <= Kp) and MASK rows (j > Kp)
  for (int j = tid; j < Kp + p.K; j += kThreads) {
    const int k = vb + j;
    const int t = oo + k;
    if (!PE_INVARIANT(p.err, t >= 0 && t < p.T && (j > Kp || (io + k >= 0 && io + k < p.R))))
      continue;
    int tok, pos, rej = 0, msk = 0;
    if (j <= Kp) {
      tok = slot_token(j);
      pos = sh.pos[j];
      rej = j > a;
    } else {
      msk = 1;
      tok = p.mask_id;
      pos = pos_s + (j - Kp);
    }
    p.out_tokens[t] = tok;
    p.out_positions[t] = pos;
    p.is_rejected[t] = (uint8_t)rej;
    p.is_masked[t] = (uint8_t)msk;
    p.slot_mapping[t] =
        rej ? -1 : kv_slot(p.block_table, p.bt_width, p.block_size, b, pos, p.err);
    if (j <= Kp) p.hidden_map[io + k] = t;
    if (p.sample_idx) {
      if (k == s) p.sample_idx[(long long)b * p.K] = t;
      if (j > Kp) p.sample_idx[(long long)b * p.K + (j - Kp)] = t;
    }
  }
  if (tid == 0) {
    const bool legal = xfer_legal(old, Kp, false);
    if (!legal) atomicOr(p.err, PE_ERR_WORKSPACE);
    const bool mine = legal && (old & kXferCount) == (unsigned long long)nr;
    // both sides are done: clear for the next call (the acquire above
    // already orders the tiles' writes of the row before ours)
    if (mine) st_relaxed(p.xfer + b, 0ull);
    sh.xwrite = mine ? 1 : 0;
  }
  __syncthreads();
  if (sh.xwrite && PE_INVARIANT(p.err, oo + s >= 0 && oo + s < p.T)) {
    uint4* dst = p.X + (long long)(oo + s) * 2 * p.nvh;
    if (tid < p.nvh) dst[tid] = x1;
    if (kThreads + tid < p.nvh) dst[kThreads + tid] = x2;
    for (int v = 2 * kThreads + tid; v < p.nvh; v += kThreads)
      dst[v] = bok ? __ldg(bsrc + v) : zero;
  }
}

// ------------------------------------------------------------ key slots
// In the single pass (below) chunk keys travel through slots instead of
// per-row atomic maxima: each argmax unit u stores its chunk key into slot u
// (one relaxed 64-bit store; a chunk without an element would store 1, which
// no key equals), and the CTA of the request's last chunk collects them.
// The slot is its own message, so the store needs no fence.
constexpr unsigned long long kEmptyChunk = 1ull;
constexpr unsigned long long kSlotWaitNs = 20000000ull;  // 20 ms: never expected

__device__ __forceinline__ unsigned long long slot_value(unsigned long long key) {
  return key ? key : kEmptyChunk;
}

// The collecting CTA of request b: the drafts and positions into sh.tok /
// sh.pos, then every chunk slot of the request (waiting, bounded, for those
// still in flight), each row's maximum into sh.rowkey; the slots are left
// zero for the next call.
__device__ __forceinline__ void collect_request_keys(const StepParams& p, SharedState& sh,
                                                     int b) {
  const int tid = threadIdx.x;
  const int nr = p.Kp + 1;
  const int io = seg_begin(p, b);
  const int vb = seg_begin(p, b + 1) - io - 1 - p.Kp;
  if (tid < nr) {
    sh.rowkey[tid] = 0ull;
    if (tid < p.Kp) sh.tok[tid] = __ldg(p.in_tokens + io + vb + tid + 1);
    if (p.full) sh.pos[tid] = __ldg(p.in_positions + io + vb + tid);
  }
  __syncthreads();
  const int n = nr * p.C;
  unsigned long long* slot = p.slots + (long long)b * n;
  bool late = false;
  for (int i = tid; i < n; i += kThreads) {
    unsigned long long v = ld_relaxed(slot + i);
    if (v == 0ull) {
      const unsigned long long t0 = global_ns();
      while (v == 0ull && global_ns() - t0 < kSlotWaitNs) v = ld_relaxed(slot + i);
    }
    if (v == 0ull) {
      late = true;
    } else if (v != kEmptyChunk) {
      if (key_col(v) >= (uint32_t)p.V) atomicOr(p.err, PE_ERR_WORKSPACE);  // not a key of this call
      atomicMax(&sh.rowkey[i / p.C], v);
    }
    slot[i] = 0ull;  // clear for the next call
  }
  if (late) atomicOr(p.err, PE_ERR_TIMEOUT);
  __syncthreads();
}

// ------------------------------------------------------------- argmax chunk
template <int DT>
__device__ __forceinline__ void finish_argmax_unit(const StepParams& p, SharedState& sh, int r,
                                                   int c, const char* rowp,
                                                   unsigned long long key);

template <int DT>
__device__ __forceinline__ void argmax_unit(const StepParams& p, SharedState& sh, int u) {
  const int tid = threadIdx.x;
  const int r = u / p.C;
  const int c = u - r * p.C;
  const char* rowp = logits_row(p, r);
  const int v_lo = c * p.chunk_vecs;
  const int v_hi = rowp ? min(v_lo + p.chunk_vecs, p.nvec) : v_lo;  // bad index: nothing
  if (!rowp && c == 0 && tid == 0) atomicOr(p.err, PE_ERR_ROW_RANGE);
  const unsigned long long key =
      thread_key<DT, kThreads>(reinterpret_cast<const uint4*>(rowp), v_lo, v_hi, p.err);
  finish_argmax_unit<DT>(p, sh, r, c, rowp, key);
}

// End of an argmax unit: fold in the leftover elements, reduce the threads'
// keys, merge into the row's key, and run the request's epilogue in the CTA
// whose unit completes the request.
template <int DT>
__device__ __forceinline__ void finish_argmax_unit(const StepParams& p, SharedState& sh, int r,
                                                   int c, const char* rowp,
                                                   unsigned long long key) {
  const int tid = threadIdx.x;
  // leftover elements past the last whole vector (last chunk, one thread)
  if (p.tail && rowp && c == p.C - 1 && tid == 0) {
    const unsigned long long tk = tail_key<DT>(rowp, p.nvec, p.tail, p.err);
    key = tk > key ? tk : key;
  }

  key = warp_max_key(key);
  if ((tid & 31) == 0) sh.red[tid >> 5] = key;
  __syncthreads();
  if (tid < 32) {
    unsigned long long k = tid < kWarps ? sh.red[tid] : 0ull;
    k = warp_max_key(k);
    if (tid == 0) {
      atomicMax(p.keys + r, k);
      const int b = r / (p.Kp + 1);
      const unsigned total = (unsigned)((p.Kp + 1) * p.C);
      // release: the key merge above before the count; acquire (for the
      // last arrival): every other chunk's merge
      const unsigned done = atom_add_acq_rel_u32(p.count + b, 1u);
      if (done >= total) atomicOr(p.err, PE_ERR_WORKSPACE);  // did not start at zero
      const bool last = done == total - 1u;
      sh.last = last ? b : -1;
    }
  }
  __syncthreads();
  const int last = sh.last;
  if (last >= 0) request_epilogue<kKeysInWorkspace>(p, sh, last);
}

// ------------------------------------------------------- early-exit units
// Early exit reads a request's rows in order and stops after the first
// mismatch.  Units run row-major over (row j, request b, chunk c), so every
// request's row 0 streams first, then row 1, ...; a unit whose request is
// already known to mismatch at an earlier row is skipped before it reads
// anything (skip_moot).  The CTA that completes a row records its argmax and
// ORs two bits into the request's state word (row done; row's argmax equals
// the draft).  The OR after which the rows 0..a are all done, 0..a-1 all
// match and a mismatches (or a = K') settles the request: exactly one CTA
// sees that change, and it runs the epilogue.  A chunk that ends before its
// row completes ORs bit j into the request's count word when its key beats
// the draft's own key (the row's argmax cannot be the draft), so the later
// rows turn moot without waiting for the whole row (B=256 61.1 us against
// 62.5, B=64 37.5 against 39.1).  Nothing ever waits for another CTA.

// Accepted length settled by a state word, or -1 while it is still open.
__device__ __forceinline__ int settled(unsigned long long st, int Kp) {
  for (int j = 0; j <= Kp; ++j) {
    if (!((st >> j) & 1ull)) return -1;               // row j not done yet
    if (j == Kp || !((st >> (32 + j)) & 1ull)) return j;  // bonus row / mismatch
  }
  return -1;
}

template <int DT>
__device__ __forceinline__ void argmax_unit_early(const StepParams& p, SharedState& sh, int u) {
  const int tid = threadIdx.x;
  const int per_row = p.B * p.C;
  const int j = u / per_row;
  const int rem = u - j * per_row;
  const int b = rem / p.C;
  const int c = rem - b * p.C;
  const int r = b * (p.Kp + 1) + j;  // (moot units were skipped by the scheduler)
  const char* rowp = logits_row(p, r);
  const int v_lo = c * p.chunk_vecs;
  const int v_hi = min(v_lo + p.chunk_vecs, p.nvec);
  int d = -1;  // the draft this row is compared with (thread 0; loaded while the chunk streams)
  if (tid == 0 && j < p.Kp) {
    const int io = seg_begin(p, b);
    const int vb = seg_begin(p, b + 1) - io - 1 - p.Kp;
    d = __ldg(p.in_tokens + io + vb + j + 1);
  }
  unsigned long long key =
      thread_key<DT, kThreads>(reinterpret_cast<const uint4*>(rowp), v_lo, v_hi, p.err);
  float xd = 0.f;  // the draft's own logit
  if (tid == 0 && d >= 0 && d < p.V) xd = Elem<DT>::scalar(rowp, d);
  if (p.tail && c == p.C - 1 && tid == 0) {  // leftover elements past the last vector
    const unsigned long long tk = tail_key<DT>(rowp, p.nvec, p.tail, p.err);
    key = tk > key ? tk : key;
  }
  key = warp_max_key(key);
  if ((tid & 31) == 0) sh.red[tid >> 5] = key;
  __syncthreads();
  if (tid < 32) {
    unsigned long long k = tid < kWarps ? sh.red[tid] : 0ull;
    k = warp_max_key(k);
    if (tid == 0) {
      int due = -1, a = -1;
      atomicMax(p.keys + r, k);
      // release / acquire as for the fused step's request count
      const unsigned rc = atom_add_acq_rel_u32(p.rcount + r, 1u);
      if (rc >= (unsigned)p.C) atomicOr(p.err, PE_ERR_WORKSPACE);  // did not start at zero
      // A chunk whose key beats the draft's own key proves the row's argmax
      // is not the draft: the request mismatches at row j at the latest, so
      // its later rows are moot before the row completes.
      if (j < p.Kp && rc < (unsigned)(p.C - 1) &&
          (d < 0 || d >= p.V || k > make_key(xd, (uint32_t)d)))
        atomicOr(p.count + b, 1u << j);
      if (rc == (unsigned)(p.C - 1)) {  // row r complete
        const unsigned long long kk = atomicExch(p.keys + r, 0ull);
        atomicExch(p.rcount + r, 0u);
        const uint32_t col = key_col(kk);
        if (kk == 0ull || col >= (uint32_t)p.V) atomicOr(p.err, PE_ERR_WORKSPACE);
        const int am = (int)col;
        p.amax_ws[r] = am;
        const int io = seg_begin(p, b);
        const int vb = seg_begin(p, b + 1) - io - 1 - p.Kp;
        const bool match = j < p.Kp && am == __ldg(p.in_tokens + io + vb + j + 1);
        const unsigned long long bits = (1ull << j) | (match ? (1ull << (32 + j)) : 0ull);
        // release: the row's argmax before its done bit; acquire (for the
        // CTA that settles the request): the argmax of every row it settles on
        const unsigned long long old = atom_or_acq_rel(p.state + b, bits);
        // before this OR: done bits of other rows < K'+1 only, match bits of
        // rows < K' only, and not this row's done bit
        const unsigned long long legal =
            (p.Kp == 31 ? 0xffffffffull : (1ull << (p.Kp + 1)) - 1ull) |
            (((1ull << p.Kp) - 1ull) << 32);
        if ((old & ~legal) || ((old >> j) & 1ull)) atomicOr(p.err, PE_ERR_WORKSPACE);
        const int a_new = settled(old | bits, p.Kp);
        if (settled(old, p.Kp) < 0 && a_new >= 0) {
          due = b;
          a = a_new;
        }
      }
      sh.last = due;
      sh.first = a;
    }
  }
  __syncthreads();
  const int due = sh.last;
  const int a = sh.first;
  if (due >= 0) request_epilogue<kRowsSettled>(p, sh, due, a);
}

// ------------------------------------------------------------------ X tiles
// Rows whose content verification cannot change: hidden half of every row,
// MASK rows entirely, prompt rows (prefill) entirely plus their metadata.
// X row t (request b, segment io / n) of row i of the verified rows, which
// are listed request by request, K'+1 each.
__device__ __forceinline__ void verified_row(const StepParams& p, int i, int& t, int& b,
                                             int& io, int& n) {
  const int nr = p.Kp + 1;
  b = i / nr;
  io = seg_begin(p, b);
  n = seg_begin(p, b + 1) - io;
  t = io + b * (p.K - 1) + (n - nr) + (i - b * nr);
}

// X row t of row i of the other rows: each request's prompt rows, then its
// K-1 MASK rows, request by request; request b holds n_b - (K'+1) + K - 1
// of them, starting at oo_b - b(K'+1).
__device__ __forceinline__ void other_row(const StepParams& p, int i, int& t, int& b, int& io,
                                          int& n) {
  const int nr = p.Kp + 1;
  if (!p.in_offsets) {  // decode: MASK rows only (K > 1 when there are any)
    b = i / (p.K - 1);
    io = b * nr;
    n = nr;
    t = io + b * (p.K - 1) + nr + (i - b * (p.K - 1));
    return;
  }
  int lo = 0, hi = p.B - 1;  // largest b whose first such row is at or before i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.in_offsets + mid) + mid * (p.K - 1 - nr) <= i)
      lo = mid;
    else
      hi = mid - 1;
  }
  b = lo;
  io = __ldg(p.in_offsets + b);
  n = __ldg(p.in_offsets + b + 1) - io;
  const int l = i - (io + b * (p.K - 1 - nr));
  t = io + b * (p.K - 1) + (l < n - nr ? l : l + nr);
}

// Setup of a copy tile: thread i < nrows works out row i's two half rows
// (source, destination, mode), writes a prompt row's metadata, and notes a
// verified row's request for the hand-off.  Returns the tile's row count.
__device__ __forceinline__ int copy_setup(const StepParams& p, SharedState& sh, int u,
                                          bool& vtile_out) {
  const int tid = threadIdx.x;
  const bool vtile = u < p.n_vtile;  // a tile of verified rows
  const int i0 = (vtile ? u : u - p.n_vtile) * p.rows_per_unit;
  const int nrows = min(p.rows_per_unit, (vtile ? p.rv : p.T - p.rv) - i0);
  if (tid < nrows) {
    int t, b, io, n;
    if (vtile)
      verified_row(p, i0 + tid, t, b, io, n);
    else
      other_row(p, i0 + tid, t, b, io, n);
    const int oo = io + b * (p.K - 1);
    const int k = t - oo;
    const int vb = n - 1 - p.Kp;
    uint4* xr = p.X + (long long)t * 2 * p.nvh;
    int me;
    const uint4* se = nullptr;
    const uint4* sh_src;
    sh.vreq[tid] = -1;
    if (!PE_INVARIANT(p.err, t >= 0 && t < p.T && b >= 0 && b < p.B && k >= 0 && k < n + p.K - 1)) {
      me = kSkip;  // (checked build only) leave the row alone
      sh_src = nullptr;
      xr = nullptr;
    } else if (k < vb) {  // prompt row: shifted token, own hidden row
      const int tok = __ldg(p.in_tokens + io + k + 1);
      const int pos = __ldg(p.in_positions + io + k);
      p.out_tokens[t] = tok;
      p.out_positions[t] = pos;
      p.is_rejected[t] = 0;
      p.is_masked[t] = 0;
      p.slot_mapping[t] = kv_slot(p.block_table, p.bt_width, p.block_size, b, pos, p.err);
      p.hidden_map[io + k] = t;
      if (tok >= 0 && tok < p.V) {
        me = kCopy;
        se = p.emb + (long long)tok * p.nvh;
      } else {
        me = kZero;
        atomicOr(p.err, PE_ERR_TOKEN_RANGE);
      }
      sh_src = p.hidden + (long long)(io + k) * p.nvh;
    } else if (k < n) {
      // verified slot j: the token it has unless it is the bonus slot (the
      // shifted draft d_{j+1}, or the MASK id in the last row); the bonus
      // row is rewritten through the request's hand-off word.  A token
      // outside the table gives a zero half here; the verdict raises the
      // error bit for the slots that keep it.
      const int j = k - vb;
      const int tok = j < p.Kp ? __ldg(p.in_tokens + io + k + 1) : p.mask_id;
      if (tok >= 0 && tok < p.V) {
        me = kCopy;
        se = p.emb + (long long)tok * p.nvh;
      } else {
        me = kZero;
      }
      sh_src = p.hidden + (long long)(io + k) * p.nvh;
      sh.vreq[tid] = b;
      sh.vrow0[tid] = oo + vb;
    } else {  // MASK row: emb(mask) (+) h_shared
      me = kCopy;
      se = p.emb + (long long)p.mask_id * p.nvh;
      sh_src = p.h_shared;
    }
    sh.mode[2 * tid] = me;
    sh.src[2 * tid] = se;
    sh.dst[2 * tid] = xr;
    sh.mode[2 * tid + 1] = xr ? kCopy : kSkip;
    sh.src[2 * tid + 1] = sh_src;
    sh.dst[2 * tid + 1] = xr ? xr + p.nvh : nullptr;
  }
  if (tid == 0) sh.nbonus = 0;
  vtile_out = vtile;
  return nrows;
}

// Copy body, register path: kSeg half rows x kCols vectors per thread in
// flight (eight 16-byte loads per thread).
template <int kSeg, int kCols>
__device__ __forceinline__ void copy_body_regs(const StepParams& p, const SharedState& sh,
                                               int nrows) {
  const int tid = threadIdx.x;
  const int nseg = 2 * nrows;  // kSeg half rows x kCols vectors per thread per batch
  for (int v0 = 0; v0 < p.nvh; v0 += kCols * kThreads) {
    for (int sg = 0; sg < nseg; sg += kSeg) {
      uint4 buf[kSeg][kCols];
#pragma unroll
      for (int s = 0; s < kSeg; ++s) {
        const int md = (sg + s < nseg) ? sh.mode[sg + s] : kSkip;
        const uint4* src = (sg + s < nseg) ? sh.src[sg + s] : nullptr;
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
          const int v = v0 + i * kThreads + tid;
          if (md == kCopy && v < p.nvh)
            buf[s][i] = __ldg(src + v);
          else
            buf[s][i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int s = 0; s < kSeg; ++s) {
        const int md = (sg + s < nseg) ? sh.mode[sg + s] : kSkip;
        uint4* dst = (sg + s < nseg) ? sh.dst[sg + s] : nullptr;
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
          const int v = v0 + i * kThreads + tid;
          if (md != kSkip && v < p.nvh) dst[v] = buf[s][i];
        }
      }
    }
  }
}

// Copy body, bulk path: one thread moves every half row of the tile through
// the CTA's staging buffer (2 * rows_per_unit half rows of nvh vectors):
// a bulk load per half row, completion on the CTA's barrier, then a bulk
// store per half row.  Half rows to be zeroed (a token outside the table)
// are written by all threads with plain stores.  `phase` is the parity of
// the barrier's next phase (thread 0's copy).  verified: the tile's rows
// take part in the bonus-row hand-off, so the stores must be complete and
// ordered before the thread's later accesses when this returns.
__device__ __forceinline__ void copy_body_bulk(const StepParams& p, SharedState& sh, int nrows,
                                               uint4* stage, uint32_t& phase, bool verified) {
  const int tid = threadIdx.x;
  const int nseg = 2 * nrows;
  const uint32_t seg_bytes = (uint32_t)p.nvh * 16u;
  if (tid == 0) {
    bulk_wait_read_all();  // the previous tile's stores have left the buffer
    uint32_t bytes = 0;
    for (int sg = 0; sg < nseg; ++sg)
      if (sh.mode[sg] == kCopy) bytes += seg_bytes;
    mbar_arrive_expect_tx(&sh.bar, bytes);
    for (int sg = 0; sg < nseg; ++sg)
      if (sh.mode[sg] == kCopy)
        bulk_load(stage + (long long)sg * p.nvh, sh.src[sg], seg_bytes, &sh.bar);
  }
  for (int sg = 0; sg < nseg; ++sg)
    if (sh.mode[sg] == kZero)
      for (int v = tid; v < p.nvh; v += kThreads) sh.dst[sg][v] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) {
    if (mbar_wait(&sh.bar, phase)) {
      for (int sg = 0; sg < nseg; ++sg)
        if (sh.mode[sg] == kCopy) bulk_store(sh.dst[sg], stage + (long long)sg * p.nvh, seg_bytes);
      bulk_commit();
    } else {
      atomicOr(p.err, PE_ERR_TIMEOUT);  // never expected: the loads did not land
    }
    phase ^= 1u;
    if (verified) bulk_wait_all_visible();
  }
}

// Hand-off of a verified-row tile: count this tile's verified rows into
// their requests' words, ordered after every thread's stores of the tile
// (the barrier gathers them, the counting thread's release fence publishes
// them).  The tile that completes a request's count after its verdict was
// taken writes the bonus row (its embedding half with the bonus token); if
// the verdict comes later, the verdict writes it.
__device__ __forceinline__ void copy_handoff(const StepParams& p, SharedState& sh, int nrows) {
  const int tid = threadIdx.x;
  __syncthreads();
  if (tid < nrows && sh.vreq[tid] >= 0) {
    const int b = sh.vreq[tid];
    const unsigned long long old = atom_add_acq_rel(p.xfer + b, 1ull);
    if (!xfer_legal(old, p.Kp, true)) {
      atomicOr(p.err, PE_ERR_WORKSPACE);
    } else if ((old & kXferCount) + 1 == (unsigned long long)(p.Kp + 1) &&
               (old & kXferVerdict)) {
      st_relaxed(p.xfer + b, 0ull);  // both sides are done: clear for the next call
      const int e = atomicAdd(&sh.nbonus, 1);
      sh.brow[e] = sh.vrow0[tid] + (int)((old >> 17) & 0xffull);
      sh.btok[e] = (int)(uint32_t)(old >> 32);
    }
  }
  __syncthreads();
  const int nb = sh.nbonus;
  for (int e = 0; e < nb; ++e) {
    const int tok = sh.btok[e];
    uint4* dst = p.X + (long long)sh.brow[e] * 2 * p.nvh;
    const bool ok = tok >= 0 && tok < p.V;
    for (int v = tid; v < p.nvh; v += kThreads)
      dst[v] = ok ? __ldg(p.emb + (long long)tok * p.nvh + v) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Copy tile u.  Register path: eight loads per thread in flight, eight half
// rows at a time when a half row is at most one vector per thread, else four
// half rows of two vectors.  Bulk path: see copy_body_bulk.
template <bool BULK>
__device__ __forceinline__ void copy_tile(const StepParams& p, SharedState& sh, int u,
                                          uint4* stage, uint32_t& phase) {
  bool vtile;
  const int nrows = copy_setup(p, sh, u, vtile);
  __syncthreads();
  if (BULK)
    copy_body_bulk(p, sh, nrows, stage, phase, vtile);
  else if (p.nvh <= kThreads)
    copy_body_regs<8, 1>(p, sh, nrows);
  else
    copy_body_regs<4, 2>(p, sh, nrows);
  if (vtile) copy_handoff(p, sh, nrows);
}

// ------------------------------------------------------------------- kernel
// BULK: copy tiles through the dynamic shared-memory staging buffer.
template <int DT, bool BULK>
__global__ void __launch_bounds__(kThreads, 4) step_kernel(const StepParams p) {
  extern __shared__ __align__(128) uint4 stage[];
  __shared__ SharedState sh;
  if (p.in_offsets && !offsets_valid(p.in_offsets, p.B, p.R, p.Kp + 1)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, PE_ERR_OFFSETS);
    return;  // every CTA sees the same offsets and leaves without writing
  }
  uint32_t phase = 0;  // bulk tiles: parity of the barrier's next phase (thread 0)
  if (BULK) {
    if (threadIdx.x == 0) {
      mbar_init(&sh.bar, 1);
      mbar_init_fence();
    }
    __syncthreads();
  }
  // The first unit of each CTA is its own index; later units come from the
  // counter, which therefore hands out gridDim.x + 0, 1, 2, ...  A CTA takes
  // its next unit only when it is free: a unit handed out is a unit being
  // read, so no request's last chunk waits behind another unit.
  int q = blockIdx.x;  // queue position; unit_at gives the unit
  while (q < p.n_units) {
    const int u = unit_at(p, q);
    if (u < p.n_arg_units)
      argmax_unit<DT>(p, sh, u);
    else
      copy_tile<BULK>(p, sh, u - p.n_arg_units, stage, phase);
    __syncthreads();
    if (threadIdx.x == 0) {
      // The counter hands out n_units - gridDim.x units, then one index past
      // the end to each CTA, after which that CTA never touches it again: the
      // CTA that receives the last index (n_units - 1) is the last to finish
      // and resets the counter for the next call.  A larger value means the
      // counter did not start at zero: the CTA leaves.
      const unsigned v = atomicAdd(p.sched, 1u);
      if (v == (unsigned)p.n_units - 1u) atomicExch(p.sched, 0u);
      unsigned next = gridDim.x + v;
      if (v > (unsigned)p.n_units - 1u) {
        atomicOr(p.err, PE_ERR_WORKSPACE);
        next = (unsigned)p.n_units;
      }
      sh.unit = (int)next;
    }
    __syncthreads();
    q = sh.unit;
  }
  if (BULK && threadIdx.x == 0) bulk_wait_all_visible();  // stores done before the CTA ends
}

// ------------------------------------------------------------ single pass
// When every unit of a step fits one per co-resident CTA (few requests),
// the launch is cooperative (all CTAs resident at once) and CTA u does unit
// u and leaves: no work counter, no unit counts.  An argmax unit stores its
// chunk key into its slot; the CTA of a request's last chunk then waits,
// bounded, for the request's other slots (their CTAs are resident and never
// wait on anything), keeps each row's maximum, clears the slots and takes
// the verdict.  Each chunk pays one store instead of a key merge, a
// device-scope fence and a counting atomic in series, and the verdict reads
// its keys from shared memory.
template <int DT>
__device__ __forceinline__ void single_pass_argmax_unit(const StepParams& p, SharedState& sh,
                                                        int u) {
  const int tid = threadIdx.x;
  const int r = u / p.C;
  const int c = u - r * p.C;
  const char* rowp = logits_row(p, r);
  const int v_lo = c * p.chunk_vecs;
  const int v_hi = rowp ? min(v_lo + p.chunk_vecs, p.nvec) : v_lo;  // bad index: nothing
  if (!rowp && c == 0 && tid == 0) atomicOr(p.err, PE_ERR_ROW_RANGE);
  unsigned long long key =
      thread_key<DT, kThreads>(reinterpret_cast<const uint4*>(rowp), v_lo, v_hi, p.err);
  if (p.tail && rowp && c == p.C - 1 && tid == 0) {
    const unsigned long long tk = tail_key<DT>(rowp, p.nvec, p.tail, p.err);
    key = tk > key ? tk : key;
  }
  key = warp_max_key(key);
  if ((tid & 31) == 0) sh.red[tid >> 5] = key;
  __syncthreads();
  if (tid < 32) {
    unsigned long long k = tid < kWarps ? sh.red[tid] : 0ull;
    k = warp_max_key(k);
    if (tid == 0) st_relaxed(p.slots + u, slot_value(k));
  }
  const int nr = p.Kp + 1;
  const int b = r / nr;
  if (r - b * nr != p.Kp || c != p.C - 1) return;  // not the request's last chunk
  collect_request_keys(p, sh, b);
  request_epilogue<kKeysInShared>(p, sh, b);
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) step_kernel_single(const StepParams p) {
  __shared__ SharedState sh;
  if (p.in_offsets && !offsets_valid(p.in_offsets, p.B, p.R, p.Kp + 1)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, PE_ERR_OFFSETS);
    return;  // every CTA sees the same offsets and leaves without writing
  }
  uint32_t phase = 0;  // (register copy tiles: unused)
  const int u = blockIdx.x;  // one unit per CTA: argmax chunks, then copy tiles
  if (u < p.n_arg_units)
    single_pass_argmax_unit<DT>(p, sh, u);
  else
    copy_tile<false>(p, sh, u - p.n_arg_units, nullptr, phase);
}

// --------------------------------------------------- early-exit scheduling
// Units are handed out in order (argmax units row-major, then copy tiles).
// A CTA takes its next unit only when it is free (a unit handed out is a
// unit being read, so rows complete, and their requests' verdicts become
// known, as early as possible); thread 0 checks the unit's request and, if
// it is already known to mismatch at an earlier row, takes the next index
// instead, alone, without holding the CTA at a barrier per skipped unit.

// Next queue position (thread 0).  Every position below n_units is claimed
// once, then each CTA makes one claim past the end and leaves, so a value
// above n_units + gridDim.x - 1 means the counter did not start at zero.
__device__ __forceinline__ unsigned claim_early(const StepParams& p) {
  const unsigned v = atomicAdd(p.sched, 1u);
  if (v > (unsigned)p.n_units + gridDim.x - 1u) atomicOr(p.err, PE_ERR_WORKSPACE);
  return v;
}

// Unit at or after queue position q that is worth reading, or n_units when
// the queue is exhausted (thread 0 only).
__device__ __forceinline__ int skip_moot(const StepParams& p, unsigned q) {
  const int per_row = p.B * p.C;
  while (q < (unsigned)p.n_units) {
    const int u = unit_at(p, (int)q);
    if (u >= p.n_arg_units) return u;  // copy tile
    const int j = u / per_row;
    if (j == 0) return u;
    const int b = (u - j * per_row) / p.C;
    const unsigned long long st = __ldcg(p.state + b);
    const unsigned early = __ldcg(p.count + b);  // mismatches found before their row completed
    const unsigned done = (unsigned)st, match = (unsigned)(st >> 32);
    if (!(((done & ~match) | early) & ((1u << j) - 1u))) return u;  // no earlier mismatch known
    q = claim_early(p);                                 // moot: take the next one
  }
  return p.n_units;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) step_kernel_early(const StepParams p) {
  __shared__ SharedState sh;
  if (p.in_offsets && !offsets_valid(p.in_offsets, p.B, p.R, p.Kp + 1)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, PE_ERR_OFFSETS);
    return;  // every CTA sees the same offsets and leaves without writing
  }
  uint32_t phase = 0;  // (register copy tiles: unused)
  for (;;) {
    if (threadIdx.x == 0) sh.unit = skip_moot(p, claim_early(p));
    __syncthreads();
    const int u = sh.unit;
    if (u >= p.n_units) break;
    if (u < p.n_arg_units)
      argmax_unit_early<DT>(p, sh, u);
    else
      copy_tile<false>(p, sh, u - p.n_arg_units, nullptr, phase);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // release: this CTA's accesses before its departure; acquire (for the
    // last to leave): every other CTA's
    const unsigned done = atom_add_acq_rel_u32(p.sched + 1, 1u);
    if (done > gridDim.x - 1u) atomicOr(p.err, PE_ERR_WORKSPACE);  // did not start at zero
    sh.last = done == gridDim.x - 1;  // every other CTA has left
  }
  __syncthreads();
  if (sh.last) {  // the last CTA clears partly read rows, states and row results
    for (int i = threadIdx.x; i < p.Rl; i += kThreads) {
      p.keys[i] = 0ull;
      p.rcount[i] = 0u;
      p.amax_ws[i] = 0;
    }
    // every request has settled by now (its rows are read in order up to its
    // first mismatch); one that has not lost units to a dirty counter
    for (int i = threadIdx.x; i < p.B; i += kThreads) {
      if (settled(p.state[i], p.Kp) < 0) atomicOr(p.err, PE_ERR_WORKSPACE);
      if (p.Kp < 32 && (p.count[i] >> p.Kp)) atomicOr(p.err, PE_ERR_WORKSPACE);
      p.state[i] = 0ull;
      p.count[i] = 0u;
    }
    if (threadIdx.x == 0) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
}

}  // namespace pe

// ---------------------------------------------------------------- host side
#include <atomic>

namespace {

using pe_host::aligned16;
using pe_host::elt_size;

// Argmax chunking and grid size for `rows` logits rows of `V` elements.
// want_rows: the rows over which ~one unit per CTA is wanted (all rows, or
// for early exit half a row wave, so that each wave gives ~2 units per CTA).
void plan_argmax(pe::StepParams& p, int elt, int rows, int grid_max, int batches,
                 int want_rows = 0) {
  if (want_rows <= 0) want_rows = rows;
  const int epv = 16 / elt;
  p.Rl = rows;
  p.nvec = p.V / epv;
  p.tail = p.V % epv;
  if (p.nvec == 0) {
    p.C = 1;
    p.chunk_vecs = 0;
  } else {
    const long long cap = (long long)batches * pe::kBatchVecs;
    int c_min = (int)((p.nvec + cap - 1) / cap);
    int c_want = (grid_max + want_rows - 1) / want_rows;  // at least ~one unit per CTA
    int c_max = (p.nvec + pe::kThreads - 1) / pe::kThreads;
    int C = c_min > c_want ? c_min : c_want;
    if (C > c_max) C = c_max;
    if (C < 1) C = 1;
    // Chunks of whole batches (only a row's last chunk is ragged; measured
    // faster than equal chunks with a partial last batch each), or, below
    // one batch, of whole vectors per thread.
    int chunk = (p.nvec + C - 1) / C;
    const int grain = chunk > pe::kBatchVecs ? pe::kBatchVecs : pe::kThreads;
    chunk = (chunk + grain - 1) / grain * grain;
    p.chunk_vecs = chunk;
    p.C = (p.nvec + chunk - 1) / chunk;
  }
  // -1 when the units (plus one final claim per CTA) would not fit an int
  const long long units = (long long)rows * p.C;
  p.n_arg_units = units + grid_max > 0x7fffffffLL ? -1 : (int)units;
}

// Staging budget of a bulk-copy tile per CTA (four CTAs per SM share the
// SM's shared memory with their static state).
constexpr int kBulkStageBytes = 48 * 1024;

// X rows a bulk-copy tile can stage for half rows of `half_bytes` bytes (0:
// not even one, the register path is used).
int bulk_rows_for(long long half_bytes, int rows_per_unit) {
  const long long fit = kBulkStageBytes / (2 * half_bytes);
  return (int)(fit < rows_per_unit ? fit : rows_per_unit);
}

template <int DT>
int launch_full(const pe::StepParams& p, int grid, cudaStream_t stream) {
  if (p.bulk_rows > 0) {
    static std::atomic<unsigned long long> attr_done{0};
    const int smem = p.bulk_rows * 2 * p.nvh * 16;
    if (!pe_host::allow_smem(pe::step_kernel<DT, true>, kBulkStageBytes, attr_done))
      return PE_ECUDA;
    pe::step_kernel<DT, true><<<grid, pe::kThreads, smem, stream>>>(p);
  } else {
    pe::step_kernel<DT, false><<<grid, pe::kThreads, 0, stream>>>(p);
  }
  return pe_host::launch_status();
}

int launch(const pe::StepParams& p, int dtype, int grid, cudaStream_t stream) {
  return dtype == PE_BF16 ? launch_full<PE_BF16>(p, grid, stream)
                          : launch_full<PE_F32>(p, grid, stream);
}

int launch_early(const pe::StepParams& p, int dtype, int grid, cudaStream_t stream) {
  if (dtype == PE_BF16)
    pe::step_kernel_early<PE_BF16><<<grid, pe::kThreads, 0, stream>>>(p);
  else
    pe::step_kernel_early<PE_F32><<<grid, pe::kThreads, 0, stream>>>(p);
  return pe_host::launch_status();
}

void bind_workspace(pe::StepParams& p, void* ws, int rows, int B) {
  pe::WorkspaceLayout L(rows, B);
  char* base = static_cast<char*>(ws);
  p.sched = reinterpret_cast<uint32_t*>(base);
  p.count = reinterpret_cast<uint32_t*>(base + L.count_off);
  p.state = reinterpret_cast<unsigned long long*>(base + L.state_off);
  p.xfer = reinterpret_cast<unsigned long long*>(base + L.xfer_off);
  p.keys = reinterpret_cast<unsigned long long*>(base + L.key_off);
  p.rcount = reinterpret_cast<uint32_t*>(base + L.rcount_off);
  p.amax_ws = reinterpret_cast<int32_t*>(base + L.amax_off);
  p.slots = reinterpret_cast<unsigned long long*>(base + L.slot_off);
}

// Single-pass plan for `rows` logits rows and `cap` co-resident CTAs: copy
// tiles of 4, 8 or 16 X rows and argmax chunks such that every unit has a
// CTA of its own, choosing the tile size that leaves the most CTAs to the
// logits (so the most chunks per row; ties to the smaller tiles), with no
// chunk below half a load batch per thread.  Chunks are whole vectors per
// thread and as equal as that allows, since nothing rebalances a static
// assignment.  False when not even one chunk per row
// fits beside the tiles, or when chunks would exceed eight load batches:
// with that much work per CTA, SMs that hold one CTA more than others set
// the end (measured: B=64 decode, whole-row chunks, 46.1 us against 43.8
// on the persistent queue; B=48 even; B=32, two chunks a row, 22.7 against
// 23.7 inside a CUDA graph).
bool plan_single(pe::StepParams& p, int elt, int rows, long long cap) {
  if (rows <= 0) return false;
  int best_rpu = p.rows_per_unit;
  long long best_c = 0;
  if (!p.full) {  // verification or readout alone: argmax units only
    best_c = cap / rows;
  } else {
    for (int rpu : {p.rows_per_unit, 8, 16}) {
      if (rpu < p.rows_per_unit) continue;
      const long long n_copy = (p.rv + rpu - 1) / rpu + (p.T - p.rv + rpu - 1) / rpu;
      const long long c = (cap - n_copy) / rows;
      if (c > best_c) {
        best_c = c;
        best_rpu = rpu;
      }
    }
  }
  // Chunks of at least half a load batch per thread: measured faster than
  // more, thinner ones (B=1 decode, V=201088: 200 chunks of 4 vectors a
  // thread 10.7 us launched / 6.1 in a CUDA graph, against 400 chunks of 2
  // vectors 12.2 / 6.8; 104 chunks of 8 vectors 10.7 / 6.1).
  const long long nv = p.V / (16 / elt);
  const long long min_chunk = (long long)(pe::kVecPerThread / 2) * pe::kThreads;
  const long long c_cap = (nv + min_chunk - 1) / min_chunk;
  if (c_cap >= 1 && best_c > c_cap) best_c = c_cap;
  if (best_c < 1) return false;
  p.rows_per_unit = best_rpu;
  p.n_vtile = p.full ? (p.rv + best_rpu - 1) / best_rpu : 0;
  p.n_copy_units = p.full ? p.n_vtile + (p.T - p.rv + best_rpu - 1) / best_rpu : 0;
  const int epv = 16 / elt;
  p.Rl = rows;
  p.nvec = p.V / epv;
  p.tail = p.V % epv;
  if (p.nvec == 0) {
    p.C = 1;
    p.chunk_vecs = 0;
  } else {
    const long long per = (p.nvec + best_c - 1) / best_c;
    const long long chunk = (per + pe::kThreads - 1) / pe::kThreads * pe::kThreads;
    if (chunk > 8LL * pe::kBatchVecs) return false;
    p.chunk_vecs = (int)chunk;
    p.C = (int)((p.nvec + chunk - 1) / chunk);
  }
  p.n_arg_units = rows * p.C;
  return p.n_arg_units <= pe::kSinglePassSlots;
}

// CTAs of the single-pass kernel one SM holds at once (cached per device).
template <int DT>
int single_ctas_per_sm(int dev) {
  static std::atomic<int> cache[64];
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n) return n;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pe::step_kernel_single<DT>,
                                                    pe::kThreads, 0) != cudaSuccess || n < 1)
    n = -1;
  (void)cudaGetLastError();
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

constexpr int kNotTaken = 1;  // try_single: the step does not run as one pass

// Cooperative launch: the driver starts every CTA at once or refuses the
// launch (for instance while other work holds part of the GPU); a refusal
// leaves no error behind and returns kNotTaken, so the caller runs the
// persistent queue instead.
template <int DT>
int launch_single(const pe::StepParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeCooperative;
  attr.val.cooperative = 1;
  cfg.gridDim = dim3(p.n_units);
  cfg.blockDim = dim3(pe::kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, pe::step_kernel_single<DT>, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return kNotTaken;
  }
  return pe_host::launch_status();
}

// Few requests: plan, bind and launch the single pass when every unit fits
// one per co-resident CTA (register copy tiles only); kNotTaken otherwise
// (or when the cooperative launch is refused), with nothing enqueued.
// p holds the step's arguments, rows its logits rows (verified rows for
// pe_step; rv, T and rows_per_unit set when it copies).
int try_single(const pe::StepParams& p_in, int dtype, int elt, int rows, int B, void* ws,
               const pe_host::Tuning& tn, const pe_host::DeviceInfo& dev, void* stream) {
  if (tn.single_pass <= 0 || tn.variant == 2) return kNotTaken;
  int dev_id = 0;
  if (cudaGetDevice(&dev_id) != cudaSuccess || dev_id < 0 || dev_id >= 64) return PE_ECUDA;
  const int per_sm = dtype == PE_BF16 ? single_ctas_per_sm<PE_BF16>(dev_id)
                                      : single_ctas_per_sm<PE_F32>(dev_id);
  const long long cap = per_sm > 0 ? (long long)dev.sm_count * per_sm : 0;
  pe::StepParams q = p_in;
  if (!plan_single(q, elt, rows, cap)) return kNotTaken;
  q.n_units = q.n_arg_units + q.n_copy_units;
  bind_workspace(q, ws, rows, B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return dtype == PE_BF16 ? launch_single<PE_BF16>(q, st) : launch_single<PE_F32>(q, st);
}

}  // namespace

extern "C" {

int pe_verify_greedy(const void* logits, int dtype, int64_t row_stride, int32_t B,
                     int32_t Kp, int32_t V, const int32_t* in_tokens,
                     int32_t* accepted_len, int32_t* bonus_token,
                     int32_t* target_argmax, void* workspace, uint32_t* err,
                     void* stream) {
  const int elt = elt_size(dtype);
  if (!elt) return PE_EDTYPE;
  if (B < 0 || Kp < 0 || Kp > PE_MAX_KP || V < 1) return PE_EINVAL;
  if (B == 0) return PE_OK;
  if ((long long)B * (Kp + 1) > 0x7fffffffLL || row_stride < V) return PE_EINVAL;
  if (!logits || !accepted_len || !bonus_token || !workspace || !err) return PE_EINVAL;
  if (Kp > 0 && !in_tokens) return PE_EINVAL;
  if (!aligned16(logits) || !aligned16(workspace) || (row_stride * elt) % 16)
    return PE_EALIGN;
  pe_host::DeviceInfo dev;
  if (pe_host::device_info(&dev) != PE_OK) return PE_ECUDA;
  const pe_host::Tuning tn = pe_host::tuning();

  pe::StepParams p = {};
  p.B = B;
  p.Kp = Kp;
  p.K = 1;
  p.V = V;
  p.full = 0;
  p.row_bytes = row_stride * elt;
  p.logits = logits;
  p.rows_total = B * (Kp + 1);
  p.in_tokens = in_tokens;
  p.accepted_len = accepted_len;
  p.bonus_token = bonus_token;
  p.target_argmax = target_argmax;
  p.err = err;
  const int rows = B * (Kp + 1);
  const int single = try_single(p, dtype, elt, rows, B, workspace, tn, dev, stream);
  if (single != kNotTaken) return single;
  const int grid_max = dev.sm_count * tn.ctas_per_sm;
  plan_argmax(p, elt, rows, grid_max, tn.chunk_batches);
  p.n_units = p.n_arg_units;
  if (p.n_units < 0) return PE_EINVAL;  // more units than an int counts
  bind_workspace(p, workspace, rows, B);
  const int grid = p.n_units < grid_max ? p.n_units : grid_max;
  return launch(p, dtype, grid, static_cast<cudaStream_t>(stream));
}

int pe_draft_readout(const void* logits, int dtype, int64_t row_stride, int32_t rows,
                     int32_t V, const int32_t* sample_idx, int32_t n, int32_t* out_tokens,
                     void* workspace, uint32_t* err, void* stream) {
  const int elt = elt_size(dtype);
  if (!elt) return PE_EDTYPE;
  if (n < 0 || rows < 0 || V < 1 || row_stride < V) return PE_EINVAL;
  if (n == 0) return PE_OK;
  if (!sample_idx && n > rows) return PE_EINVAL;
  if (!logits || !out_tokens || !workspace || !err) return PE_EINVAL;
  if (!aligned16(logits) || !aligned16(workspace) || (row_stride * elt) % 16) return PE_EALIGN;
  pe_host::DeviceInfo dev;
  if (pe_host::device_info(&dev) != PE_OK) return PE_ECUDA;
  const pe_host::Tuning tn = pe_host::tuning();

  // each sampled row is a request of one verified row (K' = 0): its bonus
  // token is the row's argmax
  pe::StepParams p = {};
  p.B = n;
  p.Kp = 0;
  p.K = 1;
  p.V = V;
  p.full = 0;
  p.row_bytes = row_stride * elt;
  p.logits = logits;
  p.row_index = sample_idx;
  p.rows_total = rows;
  p.bonus_token = out_tokens;
  p.err = err;
  const int single = try_single(p, dtype, elt, n, n, workspace, tn, dev, stream);
  if (single != kNotTaken) return single;
  const int grid_max = dev.sm_count * tn.ctas_per_sm;
  plan_argmax(p, elt, n, grid_max, tn.chunk_batches);
  p.n_units = p.n_arg_units;
  if (p.n_units < 0) return PE_EINVAL;  // more units than an int counts
  bind_workspace(p, workspace, n, n);
  const int grid = p.n_units < grid_max ? p.n_units : grid_max;
  return launch(p, dtype, grid, static_cast<cudaStream_t>(stream));
}

namespace {
int step_common(const pe_step_args* a, void* stream, bool early);
}

int pe_step(const pe_step_args* a, void* stream) { return step_common(a, stream, false); }

int pe_step_early_exit(const pe_step_args* a, void* stream) {
  if (a && a->Kp > 31) return PE_EINVAL;  // one state bit per verified row
  return step_common(a, stream, true);
}

}  // extern "C"

namespace {
int step_common(const pe_step_args* a, void* stream, bool early) {
  if (!a) return PE_EINVAL;
  const int elt = elt_size(a->logits_dtype);
  const int xelt = elt_size(a->x_dtype);
  if (!elt || !xelt) return PE_EDTYPE;
  const int B = a->B, Kp = a->Kp, K = a->K;
  if (B < 0 || Kp < 0 || Kp > PE_MAX_KP || K < 1 || K > PE_MAX_K) return PE_EINVAL;
  if (a->V < 1 || a->H < 1 || a->mask_id < 0 || a->mask_id >= a->V) return PE_EINVAL;
  if (a->bt_width < 1 || a->block_size < 1 || a->logits_row_stride < a->V)
    return PE_EINVAL;
  if (B == 0) {
    if (!a->out_offsets) return PE_EINVAL;
    return cudaMemsetAsync(a->out_offsets, 0, sizeof(int32_t),
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PE_OK
               : PE_ECUDA;
  }
  if (Kp >= 1) {
    if (a->in_offsets || (long long)a->R != (long long)B * (Kp + 1)) return PE_EINVAL;
  } else {
    if (!a->in_offsets || a->R < B) return PE_EINVAL;
  }
  const long long T = (long long)a->R + (long long)B * (K - 1);
  if ((long long)B * (Kp + 1) > 0x7fffffffLL || T > 0x7fffffffLL) return PE_EINVAL;
  if (!a->logits || !a->in_tokens || !a->in_positions || !a->block_table || !a->emb ||
      !a->target_hidden || !a->h_shared || !a->accepted_len || !a->bonus_token ||
      !a->out_offsets || !a->out_tokens || !a->out_positions || !a->is_rejected ||
      !a->is_masked || !a->hidden_map || !a->slot_mapping || !a->X || !a->workspace ||
      !a->err)
    return PE_EINVAL;
  if (!aligned16(a->logits) || !aligned16(a->emb) || !aligned16(a->target_hidden) ||
      !aligned16(a->h_shared) || !aligned16(a->X) || !aligned16(a->workspace) ||
      (a->logits_row_stride * elt) % 16 || ((long long)a->H * xelt) % 16)
    return PE_EALIGN;
  pe_host::DeviceInfo dev;
  if (pe_host::device_info(&dev) != PE_OK) return PE_ECUDA;
  const pe_host::Tuning tn = pe_host::tuning();

  pe::StepParams p = {};
  p.B = B;
  p.Kp = Kp;
  p.K = K;
  p.V = a->V;
  p.H = a->H;
  p.R = a->R;
  p.T = (int)T;
  p.mask_id = a->mask_id;
  p.bt_width = a->bt_width;
  p.block_size = a->block_size;
  p.full = 1;
  p.nvh = (int)((long long)a->H * xelt / 16);
  p.row_bytes = a->logits_row_stride * elt;
  p.logits = a->logits;
  p.rows_total = B * (Kp + 1);
  p.in_offsets = a->in_offsets;
  p.in_tokens = a->in_tokens;
  p.in_positions = a->in_positions;
  p.block_table = a->block_table;
  p.emb = static_cast<const uint4*>(a->emb);
  p.hidden = static_cast<const uint4*>(a->target_hidden);
  p.h_shared = static_cast<const uint4*>(a->h_shared);
  p.accepted_len = a->accepted_len;
  p.bonus_token = a->bonus_token;
  p.target_argmax = a->target_argmax;
  p.out_offsets = a->out_offsets;
  p.out_tokens = a->out_tokens;
  p.out_positions = a->out_positions;
  p.is_rejected = a->is_rejected;
  p.is_masked = a->is_masked;
  p.hidden_map = a->hidden_map;
  p.slot_mapping = reinterpret_cast<long long*>(a->slot_mapping);
  p.sample_idx = a->sample_idx;
  p.X = static_cast<uint4*>(a->X);
  p.err = a->err;
  const int rows = B * (Kp + 1);
  // Early exit at a small logits footprint: reading every row is faster than
  // the serial row waves (measured crossover ~125 MB); the outputs stay the
  // early-exit ones (target_argmax -1 after a_b).
  if (early && (long long)rows * p.row_bytes <= (long long)tn.early_full_read_mb << 20) {
    early = false;
    p.mask_unread = 1;
  }

  const int grid_max = dev.sm_count * tn.ctas_per_sm;
  // Few requests: one unit per CTA in a single cooperative pass
  if (!early) {
    pe::StepParams q = p;
    q.rows_per_unit = tn.rows_per_unit;
    q.rv = rows;
    const int single = try_single(q, a->logits_dtype, elt, rows, B, a->workspace, tn, dev, stream);
    if (single != kNotTaken) return single;
  }
  plan_argmax(p, elt, rows, grid_max, tn.chunk_batches);
  // bulk-copy tiles (variant 2; the early-exit kernel copies through
  // registers): as many rows per tile as the staging buffer holds
  p.rows_per_unit = tn.rows_per_unit;
  if (tn.variant == 2 && !early) {
    p.bulk_rows = bulk_rows_for((long long)p.nvh * 16, tn.rows_per_unit);
    if (p.bulk_rows > 0) p.rows_per_unit = p.bulk_rows;
  }
  p.rv = rows;  // verified rows: tiles of their own
  p.n_vtile = (p.rv + p.rows_per_unit - 1) / p.rows_per_unit;
  p.vfirst = tn.queue_order != 2;
  p.n_copy_units = p.n_vtile + (p.T - p.rv + p.rows_per_unit - 1) / p.rows_per_unit;
  const long long n_units = (long long)p.n_arg_units + p.n_copy_units;
  if (p.n_arg_units < 0 || n_units + grid_max > 0x7fffffffLL) return PE_EINVAL;
  p.n_units = (int)n_units;
  bind_workspace(p, a->workspace, rows, B);
  const int grid = p.n_units < grid_max ? p.n_units : grid_max;
  if (early) return launch_early(p, a->logits_dtype, grid, static_cast<cudaStream_t>(stream));
  return launch(p, a->logits_dtype, grid, static_cast<cudaStream_t>(stream));
}
}  // namespace
