// Drafter input assembly on its own (pe_assemble_draft_inputs).
//
// Sources: "P-EAGLE: Faster LLM Inference with Parallel Speculative Decoding
// in vLLM" -- quick-read equation Input_i (emb(token) (+) hidden state) and
// the vLLM engineering listing (target hidden states copied to their new
// positions, then the masked positions take the learned parallel-drafting
// hidden state); "P-EAGLE: Parallel Speculative Decoding in vLLM" -- Hidden
// State Management.
//
// Work items are half rows of X, one warp each, 16-byte vectors:
//   [0, T)        embedding half of slot t (row gather from the table)
//   [T, 2T)       hidden half of a masked slot t (h_shared broadcast)
//   [2T, 2T+R)    hidden half of the slot target row i maps to, unless that
//                 slot is masked (the broadcast wins, as in scatter-then-where)
// Each half row is written by exactly one item, so no ordering is needed.
#include "pe_internal.cuh"

namespace pe {

struct AssembleParams {
  int H, V, T, R, nvh;
  const uint4* emb;
  const uint4* hidden;
  const uint4* h_shared;
  const int32_t* out_tokens;
  const int32_t* hidden_map;
  const uint8_t* is_masked;
  uint4* X;
  uint32_t* err;
};

__global__ void __launch_bounds__(kThreads) assemble_kernel(const AssembleParams p) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * kThreads) >> 5;
  const long long items = 2LL * p.T + p.R;
  for (long long it = warp; it < items; it += nwarps) {
    const uint4* src = nullptr;  // nullptr: write zeros
    uint4* dst;
    if (it < p.T) {
      const int t = (int)it;
      const int tok = __ldg(p.out_tokens + t);
      dst = p.X + (long long)t * 2 * p.nvh;
      if (tok >= 0 && tok < p.V) {
        src = p.emb + (long long)tok * p.nvh;
      } else if (lane == 0) {
        atomicOr(p.err, PE_ERR_TOKEN_RANGE);
      }
    } else if (it < 2LL * p.T) {
      const int t = (int)(it - p.T);
      if (!__ldg(p.is_masked + t)) continue;
      src = p.h_shared;
      dst = p.X + (long long)t * 2 * p.nvh + p.nvh;
    } else {
      const int i = (int)(it - 2LL * p.T);
      const int t = __ldg(p.hidden_map + i);
      if (t < 0 || t >= p.T) {
        if (lane == 0) atomicOr(p.err, PE_ERR_MAP_RANGE);
        continue;
      }
      if (__ldg(p.is_masked + t)) continue;
      src = p.hidden + (long long)i * p.nvh;
      dst = p.X + (long long)t * 2 * p.nvh + p.nvh;
    }
    constexpr int kU = 4;
    for (int v0 = lane; v0 < p.nvh; v0 += 32 * kU) {
      uint4 buf[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int v = v0 + 32 * j;
        buf[j] = (src && v < p.nvh) ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int v = v0 + 32 * j;
        if (v < p.nvh) dst[v] = buf[j];
      }
    }
  }
}

}  // namespace pe

extern "C" int pe_assemble_draft_inputs(int dtype, int32_t H, int32_t V, int32_t T,
                                        int32_t R, const void* emb,
                                        const void* target_hidden, const void* h_shared,
                                        const int32_t* out_tokens,
                                        const int32_t* hidden_map,
                                        const uint8_t* is_masked, void* X, uint32_t* err,
                                        void* stream) {
  const int elt = pe_host::elt_size(dtype);
  if (!elt) return PE_EDTYPE;
  if (H < 1 || V < 1 || T < 0 || R < 0) return PE_EINVAL;
  if (T == 0 && R == 0) return PE_OK;
  if (!emb || !target_hidden || !h_shared || !out_tokens || !hidden_map || !is_masked ||
      !X || !err)
    return PE_EINVAL;
  if (!pe_host::aligned16(emb) || !pe_host::aligned16(target_hidden) ||
      !pe_host::aligned16(h_shared) || !pe_host::aligned16(X) ||
      ((long long)H * elt) % 16)
    return PE_EALIGN;
  pe_host::DeviceInfo dev;
  if (pe_host::device_info(&dev) != PE_OK) return PE_ECUDA;
  pe::AssembleParams p;
  p.H = H;
  p.V = V;
  p.T = T;
  p.R = R;
  p.nvh = (int)((long long)H * elt / 16);
  p.emb = static_cast<const uint4*>(emb);
  p.hidden = static_cast<const uint4*>(target_hidden);
  p.h_shared = static_cast<const uint4*>(h_shared);
  p.out_tokens = out_tokens;
  p.hidden_map = hidden_map;
  p.is_masked = is_masked;
  p.X = static_cast<uint4*>(X);
  p.err = err;
  const long long items = 2LL * T + R;
  const long long want = (items + pe::kWarps - 1) / pe::kWarps;
  const long long grid_max = (long long)dev.sm_count * 8;
  const int grid = (int)(want < grid_max ? want : grid_max);
  pe::assemble_kernel<<<grid, pe::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return pe_host::launch_status();
}
