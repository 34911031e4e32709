// Draft-batch rebuild on its own (pe_build_draft_batch): the metadata half
// of the fused step, for callers that verify elsewhere.
//
// Source: "P-EAGLE: Parallel Speculative Decoding in vLLM" -- Fused Triton
// Kernel (copy previous token ids and positions, insert the bonus token,
// fill parallel-drafting slots with MASK ids, emit rejected-token mask,
// masked-token mask and hidden-state mapping in one pass) and KV Cache and
// CUDA Graphs (rejected tokens -> PADDING_SLOT_ID = -1).
//
// One CTA per request (grid-strided); threads walk the request's output
// slots.  Pure integer work.
#include "pe_internal.cuh"

namespace pe {

struct RebuildParams {
  int B, Kp, K, mask_id, R, T, bt_width, block_size;
  const int32_t* in_offsets;
  const int32_t* in_tokens;
  const int32_t* in_positions;
  const int32_t* accepted_len;
  const int32_t* bonus_token;
  const int32_t* block_table;
  int32_t* out_offsets;
  int32_t* out_tokens;
  int32_t* out_positions;
  uint8_t* is_rejected;
  uint8_t* is_masked;
  int32_t* hidden_map;
  long long* slot_mapping;
  int32_t* sample_idx;
  uint32_t* err;
};

__global__ void __launch_bounds__(kThreads) rebuild_kernel(const RebuildParams p) {
  if (p.in_offsets && !offsets_valid(p.in_offsets, p.B, p.R, p.Kp + 1)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, PE_ERR_OFFSETS);
    return;
  }
  const int tid = threadIdx.x;
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    const int io = p.in_offsets ? __ldg(p.in_offsets + b) : b * (p.Kp + 1);
    const int n = (p.in_offsets ? __ldg(p.in_offsets + b + 1) : io + p.Kp + 1) - io;
    const int oo = io + b * (p.K - 1);
    const int m = n + p.K - 1;
    int a = p.accepted_len ? __ldg(p.accepted_len + b) : 0;
    if (a < 0 || a > p.Kp) {
      if (tid == 0) atomicOr(p.err, PE_ERR_SLOT_RANGE);
      a = 0;
    }
    const int s = n - 1 - p.Kp + a;  // next-token-prediction slot
    const int bonus = __ldg(p.bonus_token + b);
    const int pos_s = __ldg(p.in_positions + io + s);
    if (tid == 0) {
      p.out_offsets[b] = oo;
      if (b == p.B - 1) p.out_offsets[p.B] = p.T;
    }
    for (int k = tid; k < m; k += kThreads) {
      const int t = oo + k;
      int tok, pos, rej = 0, msk = 0;
      if (k < s) {
        tok = __ldg(p.in_tokens + io + k + 1);
        pos = __ldg(p.in_positions + io + k);
      } else if (k == s) {
        tok = bonus;
        pos = pos_s;
      } else if (k < n) {
        rej = 1;
        tok = (k < n - 1) ? __ldg(p.in_tokens + io + k + 1) : p.mask_id;
        pos = __ldg(p.in_positions + io + k);
      } else {
        msk = 1;
        tok = p.mask_id;
        pos = pos_s + (k - n + 1);
      }
      p.out_tokens[t] = tok;
      p.out_positions[t] = pos;
      p.is_rejected[t] = (uint8_t)rej;
      p.is_masked[t] = (uint8_t)msk;
      p.slot_mapping[t] =
          rej ? -1 : kv_slot(p.block_table, p.bt_width, p.block_size, b, pos, p.err);
      if (k < n) p.hidden_map[io + k] = t;
      if (p.sample_idx) {
        if (k == s) p.sample_idx[(long long)b * p.K] = t;
        if (k >= n) p.sample_idx[(long long)b * p.K + (k - n + 1)] = t;
      }
    }
  }
}

}  // namespace pe

extern "C" int pe_build_draft_batch(
    int32_t B, int32_t Kp, int32_t K, int32_t mask_id, int32_t R,
    const int32_t* in_offsets, const int32_t* in_tokens, const int32_t* in_positions,
    const int32_t* accepted_len, const int32_t* bonus_token, const int32_t* block_table,
    int32_t bt_width, int32_t block_size, int32_t* out_offsets, int32_t* out_tokens,
    int32_t* out_positions, uint8_t* is_rejected, uint8_t* is_masked,
    int32_t* hidden_map, int64_t* slot_mapping, int32_t* sample_idx, uint32_t* err,
    void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B < 0 || Kp < 0 || Kp > PE_MAX_KP || K < 1 || K > PE_MAX_K) return PE_EINVAL;
  if (bt_width < 1 || block_size < 1 || R < 0) return PE_EINVAL;
  if (B == 0) {
    if (!out_offsets) return PE_EINVAL;
    return cudaMemsetAsync(out_offsets, 0, sizeof(int32_t), st) == cudaSuccess ? PE_OK
                                                                              : PE_ECUDA;
  }
  if (!in_offsets && (long long)R != (long long)B * (Kp + 1)) return PE_EINVAL;
  if (in_offsets && (long long)R < (long long)B * (Kp + 1)) return PE_EINVAL;
  const long long T = (long long)R + (long long)B * (K - 1);
  if (T > 0x7fffffffLL) return PE_EINVAL;
  if (!in_tokens || !in_positions || !bonus_token || !block_table || !out_offsets ||
      !out_tokens || !out_positions || !is_rejected || !is_masked || !hidden_map ||
      !slot_mapping || !err)
    return PE_EINVAL;
  pe_host::DeviceInfo dev;
  if (pe_host::device_info(&dev) != PE_OK) return PE_ECUDA;

  pe::RebuildParams p;
  p.B = B;
  p.Kp = Kp;
  p.K = K;
  p.mask_id = mask_id;
  p.R = R;
  p.T = (int)T;
  p.bt_width = bt_width;
  p.block_size = block_size;
  p.in_offsets = in_offsets;
  p.in_tokens = in_tokens;
  p.in_positions = in_positions;
  p.accepted_len = accepted_len;
  p.bonus_token = bonus_token;
  p.block_table = block_table;
  p.out_offsets = out_offsets;
  p.out_tokens = out_tokens;
  p.out_positions = out_positions;
  p.is_rejected = is_rejected;
  p.is_masked = is_masked;
  p.hidden_map = hidden_map;
  p.slot_mapping = reinterpret_cast<long long*>(slot_mapping);
  p.sample_idx = sample_idx;
  p.err = err;
  const int grid_max = dev.sm_count * 8;
  const int grid = B < grid_max ? B : grid_max;
  pe::rebuild_kernel<<<grid, pe::kThreads, 0, st>>>(p);
  return pe_host::launch_status();
}
