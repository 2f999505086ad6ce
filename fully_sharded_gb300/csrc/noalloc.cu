// fsdp_pipeline_step_noalloc: the pipelined step with its staging pool in a
// fixed device array instead of caller memory, for callers that cannot
// allocate device memory where they step the optimizer (their device memory
// belongs to another allocator, or cudaMalloc's possible device
// synchronization would stall the streams the pipeline overlaps).
#include "fsdp.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace fsdp {

// The scheduler of fsdp_pipeline_step (pipeline.cu).
int pipeline_step(const fsdp_pipeline_unit_t* units, int32_t n_units, int32_t rank, uint16_t* staging,
                  int64_t slot_numel, int32_t n_slots, const fsdp_adam_t* adam, cudaStream_t compute,
                  cudaStream_t copy);

namespace {

constexpr int64_t kStagingElems = FSDP_NOALLOC_STAGING_BYTES / 2;  // bf16 elements
constexpr int kMaxDevices = 64;

// The staging pool. In host code this name is only a stand-in for the
// symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint16_t g_noalloc_staging[kStagingElems];

std::atomic<uint16_t*> g_staging_addr[kMaxDevices];

// Device address of the pool on the current device (looked up once per device).
int staging_address(uint16_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FSDP_ECUDA;
  uint16_t* p = g_staging_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_staging) != cudaSuccess || !addr) return FSDP_ECUDA;
    p = static_cast<uint16_t*>(addr);
    g_staging_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return FSDP_OK;
}

}  // namespace
}  // namespace fsdp

extern "C" int fsdp_pipeline_step_noalloc(const fsdp_pipeline_unit_t* units, int32_t n_units,
                                          int32_t rank, int32_t n_slots, const fsdp_adam_t* adam,
                                          fsdp_stream_t compute, fsdp_stream_t copy) {
  if (n_units < 0 || (n_units > 0 && !units) || n_slots < 1) return FSDP_EINVAL;
  int64_t slot = 0;
  for (int32_t i = 0; i < n_units; ++i) {
    if (!units[i].layout || units[i].layout->padded_numel < 0) return FSDP_EINVAL;
    if (units[i].layout->padded_numel > slot) slot = units[i].layout->padded_numel;
  }
  // every slot starts 16-byte aligned (whole 8-element groups), so a unit whose
  // own rows are aligned keeps the vector path in any slot
  if (slot > fsdp::kStagingElems) return FSDP_ENOSPACE;
  slot = (slot + 7) / 8 * 8;
  if (slot > fsdp::kStagingElems / n_slots) return FSDP_ENOSPACE;
  uint16_t* staging = nullptr;
  if (int rc = fsdp::staging_address(&staging)) return rc;
  return fsdp::pipeline_step(units, n_units, rank, staging, slot, n_slots, adam,
                             reinterpret_cast<cudaStream_t>(compute), reinterpret_cast<cudaStream_t>(copy));
}
