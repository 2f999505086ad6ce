// Staged optimizer-state offload (fsdp_offload_step): the rank's fp32 master,
// exp_avg and exp_avg_sq shards live in host memory; each unit's shards are
// copied into a device slot, stepped there by the fused kernel, and copied
// back, on three streams so that both directions of the host link and the
// kernel overlap.
//
// Page "fully sharded data parallel fsdp" (glossary), "CPU Offload": optimizer
// state kept in CPU memory and moved to the GPU for the update. The copies use
// the copy engines, which move the state over the Grace-GPU link in both
// directions at once; the kernel then reads and writes it at HBM speed.
#include "fsdp.h"
#include "host_internal.h"

#include <cstdint>
#include <vector>

namespace fsdp {
namespace {

constexpr int kMaxSlots = 8;

int validate(const fsdp_offload_unit_t* units, int32_t n_units, int32_t rank, const float* staging,
             int64_t slot_numel, int32_t n_slots) {
  if (n_units < 0 || (n_units > 0 && (!units || !staging))) return FSDP_EINVAL;
  if (n_slots < 1 || n_slots > kMaxSlots || slot_numel < 0) return FSDP_EINVAL;
  if (n_units == 0) return FSDP_OK;
  const fsdp_layout_t* L0 = units[0].layout;
  if (!layout_ok(L0) || L0->shard_factor != L0->world_size) return FSDP_EINVAL;
  const int W = L0->world_size;
  if (rank < 0 || rank >= W) return FSDP_EINVAL;
  if (slot_numel > INT64_MAX / (12 * int64_t(n_slots))) return FSDP_EINVAL;
  AliasCheck alias;
  alias.output(staging, slot_numel * 3 * n_slots * 4);
  for (int32_t i = 0; i < n_units; ++i) {
    const fsdp_offload_unit_t& u = units[i];
    const fsdp_layout_t* L = u.layout;
    if (!layout_ok(L) || L->world_size != W || L->shard_factor != W) return FSDP_EINVAL;
    const int64_t S = L->shard_numel, padded = L->padded_numel;
    if (S > slot_numel) return FSDP_EINVAL;
    if (S == 0) continue;
    if (!u.grads || !u.master || !u.exp_avg || !u.exp_avg_sq || !u.full_out || !u.other_shards)
      return FSDP_EINVAL;
    for (int k = 0; k < W; ++k) {
      if (!u.grads[k]) return FSDP_EINVAL;
      alias.input(u.grads[k], padded * 2);
    }
    alias.output(u.master, S * 4);
    alias.output(u.exp_avg, S * 4);
    alias.output(u.exp_avg_sq, S * 4);
    alias.output(u.full_out, padded * 2);
    for (int k = 0; k < W; ++k) {
      if (k == rank) continue;
      if (!u.other_shards[k]) return FSDP_EINVAL;
      if (u.other_shards[k] != u.full_out + k * S) alias.input(u.other_shards[k], S * 2);
    }
  }
  return alias.ok() ? FSDP_OK : FSDP_EALIAS;
}

// Segments of one unit's local-rank step with its state in a device slot.
void unit_segments(const fsdp_offload_unit_t& u, int rank, float* slot, int64_t slot_numel,
                   SegmentList& list) {
  const fsdp_layout_t* L = u.layout;
  const int W = L->world_size;
  const int64_t S = L->shard_numel;
  std::vector<const void*> ptrs;
  for (int k = 0; k < W; ++k) ptrs.push_back(u.grads[k] + rank * S);
  ptrs.push_back(slot);
  ptrs.push_back(slot + slot_numel);
  ptrs.push_back(slot + 2 * slot_numel);
  ptrs.push_back(u.full_out + rank * S);
  list.add_elementwise(kStep, S, 1, ptrs);
  for (int k = 0; k < W; ++k) {
    if (k == rank) continue;
    const uint16_t* src = u.other_shards[k];
    if (src == u.full_out + k * S) continue;  // already in place
    list.add_bytes(kCopy, src, u.full_out + k * S, S * 2);
  }
}

}  // namespace
}  // namespace fsdp

using namespace fsdp;

extern "C" int fsdp_offload_step(const fsdp_offload_unit_t* units, int32_t n_units, int32_t rank,
                                 float* staging, int64_t slot_numel, int32_t n_slots, const fsdp_adam_t* adam,
                                 fsdp_stream_t compute_s, fsdp_stream_t h2d_s, fsdp_stream_t d2h_s) {
  if (int rc = validate(units, n_units, rank, staging, slot_numel, n_slots)) return rc;
  Scalars s{};
  const int W = n_units > 0 ? units[0].layout->world_size : 1;
  if (int rc = make_scalars(adam, W, &s)) return rc;
  if (n_units == 0) return FSDP_OK;
  const cudaStream_t compute = reinterpret_cast<cudaStream_t>(compute_s);
  const cudaStream_t h2d = reinterpret_cast<cudaStream_t>(h2d_s);
  const cudaStream_t d2h = reinterpret_cast<cudaStream_t>(d2h_s);
  EventSet loaded(n_slots), stepped(n_slots), stored(n_slots), start(1), done(1);
  if (!loaded.ok || !stepped.ok || !stored.ok || !start.ok || !done.ok) return FSDP_ECUDA;
  // the copies follow the work queued on `compute` before the call (the state's
  // last use, and the steps of a previous call that used the slots)
  if (cudaEventRecord(start.ev[0], compute) != cudaSuccess) return FSDP_ECUDA;
  if (cudaStreamWaitEvent(h2d, start.ev[0], 0) != cudaSuccess) return FSDP_ECUDA;
  if (cudaStreamWaitEvent(d2h, start.ev[0], 0) != cudaSuccess) return FSDP_ECUDA;
  std::vector<bool> used(n_slots, false);
  SegmentList list;
  for (int32_t i = 0; i < n_units; ++i) {
    const fsdp_offload_unit_t& u = units[i];
    const int64_t S = u.layout->shard_numel;
    if (S == 0) continue;
    const int slot = i % n_slots;
    float* base = staging + int64_t(slot) * 3 * slot_numel;
    float* const dev[3] = {base, base + slot_numel, base + 2 * slot_numel};
    float* const host[3] = {u.master, u.exp_avg, u.exp_avg_sq};
    const size_t bytes = static_cast<size_t>(S) * 4;
    // the slot's previous unit must be back in host memory before it is refilled
    if (used[slot] && cudaStreamWaitEvent(h2d, stored.ev[slot], 0) != cudaSuccess) return FSDP_ECUDA;
    for (int a = 0; a < 3; ++a)
      if (cudaMemcpyAsync(dev[a], host[a], bytes, cudaMemcpyDefault, h2d) != cudaSuccess) return FSDP_ECUDA;
    if (cudaEventRecord(loaded.ev[slot], h2d) != cudaSuccess) return FSDP_ECUDA;
    if (cudaStreamWaitEvent(compute, loaded.ev[slot], 0) != cudaSuccess) return FSDP_ECUDA;
    list.seg.clear();
    list.ptr.clear();
    unit_segments(u, rank, base, slot_numel, list);
    if (int rc = launch(list, s, compute)) return rc;
    if (cudaEventRecord(stepped.ev[slot], compute) != cudaSuccess) return FSDP_ECUDA;
    if (cudaStreamWaitEvent(d2h, stepped.ev[slot], 0) != cudaSuccess) return FSDP_ECUDA;
    for (int a = 0; a < 3; ++a)
      if (cudaMemcpyAsync(host[a], dev[a], bytes, cudaMemcpyDefault, d2h) != cudaSuccess) return FSDP_ECUDA;
    if (cudaEventRecord(stored.ev[slot], d2h) != cudaSuccess) return FSDP_ECUDA;
    used[slot] = true;
  }
  // `compute` follows every copy back (and, through the `loaded` events, every
  // copy in): later work on `compute` sees the updated state in host memory
  if (cudaEventRecord(done.ev[0], d2h) != cudaSuccess) return FSDP_ECUDA;
  if (cudaStreamWaitEvent(compute, done.ev[0], 0) != cudaSuccess) return FSDP_ECUDA;
  return FSDP_OK;
}
