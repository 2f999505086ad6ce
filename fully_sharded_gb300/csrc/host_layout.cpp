// Host-only parts of the C ABI: FlatParameter layout, the closed-form
// memory/communication accountant and status strings.
//
// Layout: page "transformer math: FSDP", section "The sharding unit:
// FlatParameter and the wrapping policy" (flatten a unit, split evenly, one
// contiguous slice per rank); page "NOTE-003: PyTorch FSDP", "Key results"
// (sharding factor F). Accountant: "transformer math: FSDP", sections "Why FSDP
// exists" and "Per-unit memory and communication, in numbers".
#include "fsdp.h"

#include <cstdint>
#include <limits>
#include <string>

extern "C" int fsdp_flatten_layout(const int64_t* numels, int32_t n_tensors, int32_t world_size,
                                   int32_t shard_factor, int64_t* offsets_out,
                                   fsdp_layout_t* out) {
  if (!numels || !offsets_out || !out) return FSDP_EINVAL;
  if (n_tensors < 1 || world_size < 1 || world_size > FSDP_MAX_WORLD) return FSDP_EINVAL;
  if (shard_factor < 1 || world_size % shard_factor != 0) return FSDP_EINVAL;
  const int64_t kMax = std::numeric_limits<int64_t>::max() - FSDP_MAX_WORLD;
  int64_t total = 0;
  for (int32_t t = 0; t < n_tensors; ++t) {
    if (numels[t] < 0 || numels[t] > kMax - total) return FSDP_EINVAL;
    total += numels[t];
  }
  // Second pass writes, so a rejected call leaves offsets_out untouched.
  int64_t at = 0;
  for (int32_t t = 0; t < n_tensors; ++t) {
    offsets_out[t] = at;
    at += numels[t];
  }
  offsets_out[n_tensors] = at;
  const int64_t w = world_size;
  const int64_t padded = (total + w - 1) / w * w;
  out->numel = total;
  out->padded_numel = padded;
  out->shard_numel = padded / shard_factor;
  out->world_size = world_size;
  out->shard_factor = shard_factor;
  out->n_tensors = n_tensors;
  return FSDP_OK;
}

extern "C" int fsdp_account(double P, double U, int32_t N, int32_t F, int32_t prefetch,
                            fsdp_account_t* out) {
  if (!out || N < 1 || F < 1 || N % F != 0 || prefetch < 0 || !(P >= 0.0) || !(U >= 0.0))
    return FSDP_EINVAL;
  const double groups = static_cast<double>(N / F);
  const double f = static_cast<double>(F);
  const double n = static_cast<double>(N);
  const double slice = P / f;  // gradient slice all-reduced across groups
  // 16 bytes per parameter: bf16 weight + bf16 grad + fp32 master + fp32 m + fp32 v.
  out->persistent_bytes = 16.0 * slice;
  out->ddp_persistent_bytes = 16.0 * P;
  // bf16 gathered weights of the live unit plus the prefetched ones.
  out->transient_bytes = 2.0 * U * (1.0 + static_cast<double>(prefetch));
  out->peak_bytes = out->persistent_bytes + out->transient_bytes;
  // Ring volumes per rank: all-gather / reduce-scatter (k-1)/k x, all-reduce 2(k-1)/k x.
  const double in_group = 3.0 * (f - 1.0) / f * P;          // AG fwd + AG bwd + RS bwd
  const double across = 2.0 * (groups - 1.0) / groups * slice;  // AR of the slice
  out->comm_elems_ring = in_group + across;
  out->comm_elems = (F > 1 ? 3.0 * P : 0.0) + (N / F > 1 ? 2.0 * slice : 0.0);
  out->ddp_comm_elems = 2.0 * P;
  out->ddp_comm_elems_ring = 2.0 * (n - 1.0) / n * P;
  out->comm_bytes = 2.0 * out->comm_elems;  // bf16 on the wire
  out->ddp_comm_bytes = 2.0 * out->ddp_comm_elems;
  return FSDP_OK;
}

extern "C" int fsdp_account_zero(double P, int32_t N, int32_t stage, fsdp_zero_account_t* out) {
  if (!out || N < 1 || stage < 0 || stage > 3 || !(P >= 0.0)) return FSDP_EINVAL;
  const double n = static_cast<double>(N);
  // bf16 weights, bf16 gradients, fp32 master + m + v; stage k shards the last k of them
  out->optimizer_bytes = stage >= 1 ? 12.0 * P / n : 12.0 * P;
  out->grads_bytes = stage >= 2 ? 2.0 * P / n : 2.0 * P;
  out->weights_bytes = stage >= 3 ? 2.0 * P / n : 2.0 * P;
  out->total_bytes = out->weights_bytes + out->grads_bytes + out->optimizer_bytes;
  out->reduction_vs_ddp = out->total_bytes > 0.0 ? 16.0 * P / out->total_bytes : 1.0;
  out->comm_elems = stage == 3 ? 3.0 * P : 2.0 * P;
  return FSDP_OK;
}

namespace {

// The capacity in the message is FSDP_NOALLOC_STAGING_BYTES itself, so the two
// cannot disagree (built once, thread-safe static initialisation).
const char* enospace_text() {
  static const std::string text =
      "work exceeds the " + std::to_string(FSDP_NOALLOC_STAGING_BYTES >> 20) +
      " MiB staging capacity of the allocation-free entry point";
  return text.c_str();
}

}  // namespace

extern "C" const char* fsdp_status_string(int status) {
  switch (status) {
    case FSDP_OK: return "ok";
    case FSDP_EINVAL: return "invalid argument";
    case FSDP_EALIAS: return "an output overlaps an input or another output";
    case FSDP_ECUDA: return "CUDA launch error";
    case FSDP_ENOSPACE: return enospace_text();
    default: return "unknown status";
  }
}
