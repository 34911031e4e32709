// pe_step_noalloc: the fused step for callers that cannot allocate device
// memory, not even the small scratch that pe_step asks for.
//
// Who needs it: code that runs under a memory manager owning all of the
// device memory (a serving runtime that reserves its pool at start-up and
// forbids later cudaMalloc calls), plug-ins that only receive the tensors
// they work on, and latency-critical loops where a cudaMalloc / cudaFree
// would synchronise the device.  Such callers can still hand over their
// inputs and outputs, but have nowhere to take the scheduling counters and
// per-row argmax keys from.
//
// What it does: the scratch is a fixed array compiled into this library
// (PE_NOALLOC_WS_BYTES bytes, held by every GPU that loads the library until
// the process exits).  Each call clears the part it needs with a memset on
// the caller's stream, then launches the same kernel as pe_step with that
// array as its workspace.  Nothing is allocated or freed.
//
// Limits: batches whose scratch would exceed PE_NOALLOC_WS_BYTES are
// rejected with PE_EINVAL.  All calls in the process share the one array per
// device, so two calls whose work overlaps on the GPU (different streams
// without ordering between them) race on it; order such calls.
#include <mutex>

#include "pe_internal.cuh"

namespace {

// The scratch itself.  In host code this name only stands for the device
// variable; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PE_NOALLOC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device

// Device address of the scratch on the current device.  The first call on a
// device looks it up (which may load this library's GPU code on that device)
// and keeps it until the process exits: it stays valid as long as the
// device's primary context lives, i.e. unless the program resets the device
// (cudaDeviceReset), after which this entry point must not be used there.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PE_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PE_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PE_OK;
}

}  // namespace

extern "C" int pe_step_noalloc(const pe_step_args* args, void* stream) {
  if (!args) return PE_EINVAL;
  if (args->B < 0 || args->Kp < 0 || args->Kp > PE_MAX_KP) return PE_EINVAL;
  const long long rows = (long long)args->B * (args->Kp + 1);
  if (rows > 0x7fffffffLL) return PE_EINVAL;
  const size_t need = pe_workspace_bytes((int32_t)rows, args->B);
  if (need == 0 || need > PE_NOALLOC_WS_BYTES) return PE_EINVAL;  // batch too large
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != PE_OK) return rc;
  if (args->B > 0 &&
      cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PE_ECUDA;
  pe_step_args a = *args;
  a.workspace = scratch;
  return pe_step(&a, stream);
}
