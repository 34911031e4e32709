// Host-side pieces of libpe.so shared by every entry point: device
// properties, launch-shape knobs, workspace size, status names.
#include <atomic>

#include "pe_internal.cuh"
#include "pe_workspace.cuh"

namespace pe_host {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 = not queried yet

std::atomic<int> g_ctas_per_sm{4};
std::atomic<int> g_chunk_batches{3};
std::atomic<int> g_rows_per_unit{4};
std::atomic<int> g_variant{1};
std::atomic<int> g_queue_order{2};
std::atomic<int> g_early_full_read_mb{128};
std::atomic<int> g_single_pass{1};
}  // namespace

int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PE_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return PE_ECUDA;
  int sms = g_sm_count[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess || sms <= 0)
      return PE_ECUDA;
    g_sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  out->sm_count = sms;
  return PE_OK;
}

Tuning tuning() {
  Tuning t;
  t.ctas_per_sm = g_ctas_per_sm.load(std::memory_order_relaxed);
  t.chunk_batches = g_chunk_batches.load(std::memory_order_relaxed);
  t.rows_per_unit = g_rows_per_unit.load(std::memory_order_relaxed);
  t.variant = g_variant.load(std::memory_order_relaxed);
  t.queue_order = g_queue_order.load(std::memory_order_relaxed);
  t.early_full_read_mb = g_early_full_read_mb.load(std::memory_order_relaxed);
  t.single_pass = g_single_pass.load(std::memory_order_relaxed);
  return t;
}

}  // namespace pe_host

extern "C" {

size_t pe_workspace_bytes(int32_t logits_rows, int32_t B) {
  if (logits_rows < 0 || B < 0) return 0;
  return pe::WorkspaceLayout(logits_rows, B).bytes;
}

int pe_get_tuning(pe_tuning* out) {
  if (!out) return PE_EINVAL;
  pe_host::Tuning t = pe_host::tuning();
  out->ctas_per_sm = t.ctas_per_sm;
  out->chunk_batches = t.chunk_batches;
  out->rows_per_unit = t.rows_per_unit;
  out->variant = t.variant;
  out->queue_order = t.queue_order;
  out->early_full_read_mb = t.early_full_read_mb;
  out->single_pass = t.single_pass;
  return PE_OK;
}

int pe_set_tuning(const pe_tuning* in) {
  if (!in) return PE_EINVAL;
  if (in->ctas_per_sm < 0 || in->ctas_per_sm > 8) return PE_EINVAL;
  if (in->chunk_batches < 0 || in->chunk_batches > 64) return PE_EINVAL;
  if (in->rows_per_unit < 0 || in->rows_per_unit > pe::kMaxRowsPerUnit)
    return PE_EINVAL;
  if (in->variant < 0 || in->variant > 2) return PE_EINVAL;
  if (in->queue_order < 0 || in->queue_order > 2) return PE_EINVAL;
  if (in->early_full_read_mb < -1 || in->early_full_read_mb > 65536) return PE_EINVAL;
  if (in->single_pass < -1 || in->single_pass > 1) return PE_EINVAL;
  if (in->ctas_per_sm) pe_host::g_ctas_per_sm.store(in->ctas_per_sm);
  if (in->chunk_batches) pe_host::g_chunk_batches.store(in->chunk_batches);
  if (in->rows_per_unit) pe_host::g_rows_per_unit.store(in->rows_per_unit);
  if (in->variant) pe_host::g_variant.store(in->variant);
  if (in->queue_order) pe_host::g_queue_order.store(in->queue_order);
  if (in->early_full_read_mb) pe_host::g_early_full_read_mb.store(in->early_full_read_mb < 0 ? 0 : in->early_full_read_mb);
  if (in->single_pass) pe_host::g_single_pass.store(in->single_pass);
  return PE_OK;
}

const char* pe_status_str(int status) {
  switch (status) {
    case PE_OK: return "PE_OK";
    case PE_EINVAL: return "PE_EINVAL: invalid argument";
    case PE_EDTYPE: return "PE_EDTYPE: element type must be PE_F32 or PE_BF16";
    case PE_EALIGN: return "PE_EALIGN: pointer, stride or row size not 16-byte aligned";
    case PE_ECUDA: return "PE_ECUDA: CUDA runtime error at launch";
    default: return "unknown pe_status";
  }
}

}  // extern "C"
