// Optimizer-state entry points beyond the fused step: the gather of any
// per-rank state (full state dict) and the ZeRO stage 1 step.
//
// Glossary entry "fully sharded data parallel fsdp", "Checkpoint/Resume"
// (FULL_STATE_DICT) and "ZeRO Stages"; page "NOTE-003: PyTorch FSDP", "Key
// results" (F = 1 is an all-reduce).
#include "fsdp.h"
#include "host_internal.h"

#include <cstdint>
#include <vector>

using namespace fsdp;

extern "C" int fsdp_all_gather_state(const void* const* shards, const fsdp_layout_t* L, int32_t dtype,
                                     void* full_out, fsdp_stream_t stream) {
  const int es = dtype == FSDP_DTYPE_F32 ? 4 : dtype == FSDP_DTYPE_BF16 ? 2 : 0;
  if (!layout_ok(L) || es == 0 || !shards || !full_out) return FSDP_EINVAL;
  const int F = L->shard_factor;
  const int64_t S = L->shard_numel;
  if (S == 0) return FSDP_OK;
  auto* full = static_cast<unsigned char*>(full_out);
  AliasCheck alias;
  alias.output(full, L->padded_numel * es);
  SegmentList list;
  for (int k = 0; k < F; ++k) {
    if (!shards[k]) return FSDP_EINVAL;
    unsigned char* dst = full + static_cast<int64_t>(k) * S * es;
    if (shards[k] == dst) continue;  // already in place
    alias.input(shards[k], S * es);
    list.add_bytes(kCopy, shards[k], dst, S * es);
  }
  if (!alias.ok()) return FSDP_EALIAS;
  return launch(list, reduce_only_scalars(1), reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fsdp_zero1_step(const uint16_t* const* grads, const fsdp_layout_t* L, int32_t rank,
                               float* avg_grad_out, float* master, float* exp_avg, float* exp_avg_sq,
                               const uint16_t* const* other_shards, uint16_t* full_out,
                               const fsdp_adam_t* adam, fsdp_stream_t stream) {
  if (!layout_ok(L) || L->shard_factor != L->world_size || !grads) return FSDP_EINVAL;
  const int W = L->world_size;
  if (rank < 0 || rank >= W) return FSDP_EINVAL;
  Scalars s{};
  if (int rc = make_scalars(adam, W, &s)) return rc;
  const int64_t S = L->shard_numel, padded = L->padded_numel;
  if (padded == 0) return FSDP_OK;
  if (!avg_grad_out || !master || !exp_avg || !exp_avg_sq || !full_out || !other_shards) return FSDP_EINVAL;
  AliasCheck alias;
  alias.output(avg_grad_out, padded * 4);
  alias.output(master, S * 4);
  alias.output(exp_avg, S * 4);
  alias.output(exp_avg_sq, S * 4);
  alias.output(full_out, padded * 2);
  SegmentList reduce, update;
  std::vector<const void*> rows;
  for (int k = 0; k < W; ++k) {
    if (!grads[k]) return FSDP_EINVAL;
    alias.input(grads[k], padded * 2);
    rows.push_back(grads[k]);
  }
  rows.push_back(avg_grad_out);
  reduce.add_elementwise(kReduce, padded, 0, rows);  // the all-reduce average, every position
  update.add_elementwise(kAdam, S, 1,
                         {avg_grad_out + rank * S, master, exp_avg, exp_avg_sq, full_out + rank * S});
  for (int k = 0; k < W; ++k) {
    if (k == rank) continue;
    if (!other_shards[k]) return FSDP_EINVAL;
    if (other_shards[k] == full_out + k * S) continue;
    alias.input(other_shards[k], S * 2);
    update.add_bytes(kCopy, other_shards[k], full_out + k * S, S * 2);
  }
  if (!alias.ok()) return FSDP_EALIAS;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (int rc = launch(reduce, s, st)) return rc;
  Scalars su = s;
  su.w = 1;  // the second launch carries no fold
  su.inv_w = 1.0f;
  return launch(update, su, st);
}
