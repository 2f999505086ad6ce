// Pipelined multi-unit step (fsdp_pipeline_step): a host-side scheduler over
// two CUDA streams and a bounded pool of gradient staging slots.
//
// Page "NOTE-003: PyTorch FSDP", "Key results": backward prefetching issues
// the next unit's collective before the current one completes; page
// "transformer math: FSDP", "Overlap: prefetching to hide the collectives"
// and "Per-unit memory and communication, in numbers": the transient budget
// 2 U (1 + prefetch). Here the "collective" that brings a unit's data in is
// the copy of its W gradient slices into a staging slot, and n_slots - 1 is
// the prefetch depth: the copy of unit u + n_slots - 1 may run while unit u
// is stepped, never further ahead (the rate limit of the pool).
//
// The first and the last unit move in pieces of at most kEdgePieceElems shard
// elements (one 2D copy of the W slices' ranges per piece, one step launch per
// piece): the first step starts after a piece has arrived instead of a whole
// unit, and after the last copy only a piece's step and copy back remain.
// Measured on GB300 (7B local-rank step, two slots, median of 32 calls):
// 66.24 -> 65.73 ms; pieces of 1 or 2 M elements, pieces in every unit, and one
// copy per slice row instead of a 2D copy were all slower.
#include "fsdp.h"
#include "host_internal.h"

#include <algorithm>
#include <cstdint>
#include <vector>

namespace fsdp {
namespace {

constexpr int kMaxSlots = 8;
constexpr int64_t kEdgePieceElems = int64_t(1) << 22;

// Segments of elements [a0, a0 + n) of one unit's shard, the gradients in a
// slot as W rows of n elements, `pitch` elements apart.
void piece_segments(const fsdp_pipeline_unit_t& u, int rank, const uint16_t* slot, int64_t pitch, int64_t a0,
                    int64_t n, SegmentList& list) {
  const fsdp_layout_t* L = u.layout;
  const int W = L->world_size;
  const int64_t S = L->shard_numel;
  std::vector<const void*> ptrs;
  for (int k = 0; k < W; ++k) ptrs.push_back(slot + k * pitch);
  ptrs.push_back(u.master + a0);
  ptrs.push_back(u.exp_avg + a0);
  ptrs.push_back(u.exp_avg_sq + a0);
  ptrs.push_back(u.full_out + rank * S + a0);
  list.add_elementwise(kStep, n, 1, ptrs);
  for (int k = 0; k < W; ++k) {
    if (k == rank) continue;
    const uint16_t* src = u.other_shards[k];
    if (src == u.full_out + k * S) continue;  // already in place
    list.add_bytes(kCopy, src + a0, u.full_out + k * S + a0, n * 2);
  }
}

// Piece length for an edge unit of shard length S: equal pieces of at most
// kEdgePieceElems, each a whole number of 2048-element chunks (so every piece
// starts 16-byte aligned where the unit does); S itself when the unit is short
// or its rows are too far apart for a 2D copy.
int64_t edge_piece(int64_t S, int64_t max_pitch) {
  if (S <= kEdgePieceElems || S * 2 > max_pitch) return S;
  const int64_t n = (S + kEdgePieceElems - 1) / kEdgePieceElems;
  return ((S + n - 1) / n + kChunkElems - 1) / kChunkElems * kChunkElems;
}

int validate(const fsdp_pipeline_unit_t* units, int32_t n_units, int32_t rank, const uint16_t* staging,
             int64_t slot_numel, int32_t n_slots) {
  if (n_units < 0 || (n_units > 0 && (!units || !staging))) return FSDP_EINVAL;
  if (n_slots < 1 || n_slots > kMaxSlots || slot_numel < 0) return FSDP_EINVAL;
  if (n_units == 0) return FSDP_OK;
  const fsdp_layout_t* L0 = units[0].layout;
  if (!layout_ok(L0) || L0->shard_factor != L0->world_size) return FSDP_EINVAL;
  const int W = L0->world_size;
  if (rank < 0 || rank >= W) return FSDP_EINVAL;
  AliasCheck alias;
  alias.output(staging, slot_numel * n_slots * 2);
  for (int32_t i = 0; i < n_units; ++i) {
    const fsdp_pipeline_unit_t& u = units[i];
    const fsdp_layout_t* L = u.layout;
    if (!layout_ok(L) || L->world_size != W || L->shard_factor != W) return FSDP_EINVAL;
    const int64_t S = L->shard_numel;
    if (L->padded_numel > slot_numel) return FSDP_EINVAL;
    if (S == 0) continue;
    if (!u.grad_slices || !u.master || !u.exp_avg || !u.exp_avg_sq || !u.full_out || !u.other_shards)
      return FSDP_EINVAL;
    alias.input(u.grad_slices, W * S * 2);
    alias.output(u.master, S * 4);
    alias.output(u.exp_avg, S * 4);
    alias.output(u.exp_avg_sq, S * 4);
    alias.output(u.full_out, L->padded_numel * 2);
    if (u.shard_out) alias.output(u.shard_out, S * 2);
    for (int k = 0; k < W; ++k) {
      if (k == rank) continue;
      if (!u.other_shards[k]) return FSDP_EINVAL;
      if (u.other_shards[k] != u.full_out + k * S) alias.input(u.other_shards[k], S * 2);
    }
  }
  return alias.ok() ? FSDP_OK : FSDP_EALIAS;
}

}  // namespace

// The scheduler; `staging` is the caller's pool (or any device buffer of
// n_slots x slot_numel bf16 elements).
int pipeline_step(const fsdp_pipeline_unit_t* units, int32_t n_units, int32_t rank, uint16_t* staging,
                  int64_t slot_numel, int32_t n_slots, const fsdp_adam_t* adam, cudaStream_t compute,
                  cudaStream_t copy) {
  if (int rc = validate(units, n_units, rank, staging, slot_numel, n_slots)) return rc;
  Scalars s{};
  const int W = n_units > 0 ? units[0].layout->world_size : 1;
  if (int rc = make_scalars(adam, W, &s)) return rc;
  if (n_units == 0) return FSDP_OK;
  EventSet ready(n_slots), freed(n_slots), start(1);
  if (!ready.ok || !freed.ok || !start.ok) return FSDP_ECUDA;
  // the copies follow the work queued on `compute` before the call (its inputs,
  // and the steps of a previous call that read the staging slots)
  if (cudaEventRecord(start.ev[0], compute) != cudaSuccess) return FSDP_ECUDA;
  if (cudaStreamWaitEvent(copy, start.ev[0], 0) != cudaSuccess) return FSDP_ECUDA;
  int dev = 0, max_pitch = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&max_pitch, cudaDevAttrMaxPitch, dev) != cudaSuccess)
    return FSDP_ECUDA;
  std::vector<bool> used(n_slots, false);
  SegmentList list;
  int64_t q = 0;  // pieces so far (a whole unit is one piece); piece q uses slot q mod n_slots
  for (int32_t i = 0; i < n_units; ++i) {
    const fsdp_pipeline_unit_t& u = units[i];
    const int64_t S = u.layout->shard_numel;
    if (S == 0) continue;
    const int64_t piece = (i == 0 || i == n_units - 1) ? edge_piece(S, max_pitch) : S;
    for (int64_t a0 = 0; a0 < S; a0 += piece, ++q) {
      const int64_t n = std::min(piece, S - a0);
      const int slot = static_cast<int>(q % n_slots);
      uint16_t* dst = staging + slot * slot_numel;
      // the piece that last used this slot must have been stepped before it is refilled
      if (used[slot] && cudaStreamWaitEvent(copy, freed.ev[slot], 0) != cudaSuccess) return FSDP_ECUDA;
      // a piece's rows sit `piece` elements apart (a multiple of 2048: aligned rows)
      const int64_t pitch = n == S ? S : piece;
      const cudaError_t e =
          n == S ? cudaMemcpyAsync(dst, u.grad_slices, static_cast<size_t>(W) * S * 2, cudaMemcpyDefault, copy)
                 : cudaMemcpy2DAsync(dst, pitch * 2, u.grad_slices + a0, S * 2, n * 2, W, cudaMemcpyDefault, copy);
      if (e != cudaSuccess) return FSDP_ECUDA;
      if (cudaEventRecord(ready.ev[slot], copy) != cudaSuccess) return FSDP_ECUDA;
      if (cudaStreamWaitEvent(compute, ready.ev[slot], 0) != cudaSuccess) return FSDP_ECUDA;
      list.seg.clear();
      list.ptr.clear();
      piece_segments(u, rank, dst, pitch, a0, n, list);
      if (int rc = launch(list, s, compute)) return rc;
      if (cudaEventRecord(freed.ev[slot], compute) != cudaSuccess) return FSDP_ECUDA;
      used[slot] = true;
      if (u.shard_out && cudaMemcpyAsync(u.shard_out + a0, u.full_out + rank * S + a0, n * 2, cudaMemcpyDefault,
                                         compute) != cudaSuccess)
        return FSDP_ECUDA;
    }
  }
  // every copy of the call was waited for by `compute` (the `ready` events), so
  // `compute` is now ordered after all of the call's work on both streams
  return FSDP_OK;
}

}  // namespace fsdp

extern "C" int fsdp_pipeline_step(const fsdp_pipeline_unit_t* units, int32_t n_units, int32_t rank,
                                  uint16_t* staging, int64_t slot_numel, int32_t n_slots,
                                  const fsdp_adam_t* adam, fsdp_stream_t compute, fsdp_stream_t copy) {
  return fsdp::pipeline_step(units, n_units, rank, staging, slot_numel, n_slots, adam,
                             reinterpret_cast<cudaStream_t>(compute), reinterpret_cast<cudaStream_t>(copy));
}
