// GPU entry points of the C ABI (include/fsdp.h, and the diagnostic call of
// include/fsdp_test.h): argument validation, alias
// checks, segment-table construction and launch of the segment kernel.
//
// Nothing here allocates device memory: each launch carries its descriptor
// table as a __grid_constant__ kernel parameter.
#include "fsdp.h"
#include "fsdp_test.h"
#include "segment_kernel.cuh"
#include "host_internal.h"

namespace fsdp {
// Sticky per-device status word: bit 0 is set when a bounded wait of the TMA
// form ran out (see tma_kernel.cuh). Read and cleared with fsdp_device_status.
__device__ unsigned int g_fsdp_status;
}  // namespace fsdp

#include "tma_kernel.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace fsdp {
namespace {

// ------------------------------------------------------------ device facts

constexpr int kMaxDevices = 64;
// Kernel variants: 0..5 the LDG form for W = 1, 2, 4, 8, 16 and any W with the
// 8-consecutive-element mapping, 6 the TMA form (W = 8), 7..12 the LDG form
// again with the split mapping (Map<true> in segment_kernel.cuh), 13 the TMA
// form for W = 16, 14..19 the LDG form with the realigned path (launches that
// hold step segments off 16-byte alignment: kPhased).
constexpr int kTmaVariant = 6;
constexpr int kSplitVariants = 7;
constexpr int kTma16Variant = 13;
constexpr int kRealignVariants = 14;  // 14..19: the LDG form with the realigned path
constexpr int kNumVariants = 20;

std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_blocks_per_sm[kMaxDevices][kNumVariants];

int variant_of(int w) {
  switch (w) {
    case 1: return 0;
    case 2: return 1;
    case 4: return 2;
    case 8: return 3;
    case 16: return 4;
    default: return 5;
  }
}

template <bool kSplit, bool kWithRealign = false>
const void* ldg_kernel_of(int variant) {
  switch (variant) {
    case 0: return reinterpret_cast<const void*>(&segment_kernel<1, kSplit, kWithRealign>);
    case 1: return reinterpret_cast<const void*>(&segment_kernel<2, kSplit, kWithRealign>);
    case 2: return reinterpret_cast<const void*>(&segment_kernel<4, kSplit, kWithRealign>);
    case 3: return reinterpret_cast<const void*>(&segment_kernel<8, kSplit, kWithRealign>);
    case 4: return reinterpret_cast<const void*>(&segment_kernel<16, kSplit, kWithRealign>);
    default: return reinterpret_cast<const void*>(&segment_kernel<0, kSplit, kWithRealign>);
  }
}

const void* kernel_of(int variant) {
  if (variant == kTmaVariant) return reinterpret_cast<const void*>(&tma_kernel<8, false>);
  if (variant == kTma16Variant) return reinterpret_cast<const void*>(&tma_kernel<16, false>);
  if (variant >= kRealignVariants) return ldg_kernel_of<false, true>(variant - kRealignVariants);
  return variant >= kSplitVariants ? ldg_kernel_of<true>(variant - kSplitVariants) : ldg_kernel_of<false>(variant);
}

// Resident-grid size for a kernel variant on the current device (cached).
int grid_capacity(int variant, int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = FSDP_ECUDA;
    return 0;
  }
  int sms = g_sm_count[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
      *err = FSDP_ECUDA;
      return 0;
    }
    g_sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  int per_sm = g_blocks_per_sm[dev][variant].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    const bool tma = variant == kTmaVariant || variant == kTma16Variant;
    const int smem = variant == kTma16Variant ? TmaCfg<16>::kSmemBytes : tma ? TmaCfg<8>::kSmemBytes : 0;
    // every instantiation of the TMA form gets the shared memory of its pipeline
    // (for W = 8 both the one-copy and the four-round one)
    if (tma && (cudaFuncSetAttribute(kernel_of(variant), cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                    cudaSuccess ||
                (variant == kTmaVariant &&
                 (cudaFuncSetAttribute(reinterpret_cast<const void*>(&tma_kernel<8, true>),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
                  cudaFuncSetAttribute(reinterpret_cast<const void*>(&tma_kernel<8, true, true>),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)))) {
      *err = FSDP_ECUDA;
      return 0;
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel_of(variant), tma ? kTmaThreads : kThreads,
                                                      smem) != cudaSuccess ||
        per_sm <= 0) {
      *err = FSDP_ECUDA;
      return 0;
    }
    const int w_variant = variant >= kRealignVariants ? variant - kRealignVariants
                          : variant >= kSplitVariants ? variant - kSplitVariants
                                                      : variant;
    if (!tma && w_variant < 5 && per_sm > kBlocksPerSm) per_sm = kBlocksPerSm;  // fixed-W LDG variants
    g_blocks_per_sm[dev][variant].store(per_sm, std::memory_order_relaxed);
  }
  return sms * per_sm;
}

int64_t chunks_of(const Seg& d) {
  const int64_t unit = (d.kind == kCopy || d.kind == kZero) ? kChunkBytes : kChunkElems;
  return (d.n + unit - 1) / unit;
}

// Programmatic dependent launch: the launch and block placement of this grid
// overlap the tail of the previous kernel on the stream (measured on GB300:
// 1e7-element step 66.3 -> 64.5 us, 7B local-rank step 8.64 -> 8.57 ms); the
// kernel's griddepcontrol.wait keeps every memory access after the previous
// kernel has completed.
template <int W, bool kSplit, bool kWithRealign = false>
cudaError_t launch_variant(const Params& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, segment_kernel<W, kSplit, kWithRealign>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int W, bool kInterleave, bool kOutOfLine = false>
cudaError_t launch_tma_form(const Params& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTmaThreads);
  cfg.dynamicSmemBytes = TmaCfg<W>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, tma_kernel<W, kInterleave, kOutOfLine>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The W = 8 instantiations (copy-only launches take them whatever the W of the call);
// interleaved launches holding copy chunks take the one with its unstaged paths out
// of line (see tma_unstaged).
cudaError_t launch_tma(const Params& p, int grid, cudaStream_t stream, bool interleave = false,
                       bool copies = false) {
  if (interleave && copies) return launch_tma_form<8, true, true>(p, grid, stream);
  return interleave ? launch_tma_form<8, true>(p, grid, stream) : launch_tma_form<8, false>(p, grid, stream);
}

// Largest address span of one step segment's gradient rows in a launch.
uintptr_t max_row_span(const Params& p) {
  uintptr_t span = 0;
  for (int k = 0; k < p.nseg; ++k) {
    const Seg& d = p.seg[k];
    if (d.kind != kStep) continue;
    uintptr_t lo = UINTPTR_MAX, hi = 0;
    for (int r = 0; r < p.s.w; ++r) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(p.ptr[d.ptr + r]);
      lo = std::min(lo, a);
      hi = std::max(hi, a);
    }
    span = std::max(span, hi - lo);
  }
  return span;
}

bool has_step(const Params& p) {
  for (int k = 0; k < p.nseg; ++k)
    if (p.seg[k].kind == kStep) return true;
  return false;
}

// W = 16 step launches take the TMA form when the gradient rows of some step
// segment do not all lie a whole number of 2 KB apart: the LDG form's sixteen
// simultaneous row streams then run below the copy peak, while the TMA form's
// bulk copies do not care. Measured on GB300 (interleaved A/B, fraction of the
// copy peak, LDG -> TMA form with two 88 KB stages; one FlatParameter of P
// elements, so the rows are 2P bytes apart): rows a multiple of 512 B or 1 KB
// apart (P = 1e8, 2e8, 3e8, 5e8, 1e9): 1.008 -> 1.012, 0.994 -> 1.012,
// 1.006 -> 1.017, 1.001 -> 1.008, 0.972 -> 1.005; a multiple of 2, 4, 8, 16 or
// 32 KB (P near 2e8, and the Llama block's 202,383,360): 1.042 -> 1.019,
// 1.047 -> 1.022, 1.050 -> 1.024, 1.050 -> 1.027, 1.050 -> 1.027, 1.041 ->
// 1.024; and near 1e9 with 2 KB and 16 KB: 1.025 -> 1.009, 1.040 -> 1.019.
// The rows' span does not matter (3 to 30 GiB above). Since the TMA form's
// consumers store state as 32-byte sectors it gained 1-2 % (the off-grain
// launches above: 1.026-1.038), and the LDG form still leads on aligned rows:
// 2 KB 1.042 -> 1.037, 4 KB 1.047 -> 1.038, 16 KB 1.051 -> 1.043 and
// 1.054 -> 1.037.
constexpr uintptr_t kTma16RowGrain = 2048;

bool rows_off_grain(const Params& p) {
  for (int k = 0; k < p.nseg; ++k) {
    const Seg& d = p.seg[k];
    if (d.kind != kStep) continue;
    const uintptr_t base = reinterpret_cast<uintptr_t>(p.ptr[d.ptr]);
    for (int r = 1; r < p.s.w; ++r)
      if ((reinterpret_cast<uintptr_t>(p.ptr[d.ptr + r]) - base) % kTma16RowGrain != 0) return true;
  }
  return false;
}

// The TMA form pays off for launches that give every block enough chunks to
// fill its pipeline and that hold either W = 8 steps whose positions each have
// one replica (with any copies; W = 16 ones under the rule above), or only
// copies (with any zero fills: pack, unpack, all-gather, state gather; measured
// on GB300, copies of 0.4-1.7 GB ran 1-3.5 % faster than on the LDG form). Its
// producer stages only step and copy chunks; a launch holding reduce or Adam
// segments, steps of another W or replicated steps stays on the LDG form, whose
// 24 warps per SM carry such chunks better than the TMA form's 8 consumers.
bool use_tma(const Params& p, int tma_grid) {
  bool step = false, copy = false;
  int64_t step_chunks = 0, phased_chunks = 0, copy_chunks = 0, narrow_chunks = 0;
  for (int k = 0; k < p.nseg; ++k) {
    const Seg& d = p.seg[k];
    if (d.kind == kStep) {
      if (d.nrep != 1 || (p.s.w != 8 && p.s.w != 16)) return false;
      const int64_t c = (d.n + kChunkElems - 1) / kChunkElems;
      step_chunks += c;
      if (d.width == kPhased) phased_chunks += c;
      step = true;
    } else if (d.kind == kCopy) {
      const int64_t c = (d.n + kChunkBytes - 1) / kChunkBytes;
      copy_chunks += c;
      if (d.width != 16) narrow_chunks += c;
      copy = true;
    } else if (d.kind != kZero) {
      return false;
    }
  }
  if (step) {
    for (int k = 0; k < p.nseg; ++k)
      if (p.seg[k].kind == kZero) return false;
    if (p.s.w == 16 && !rows_off_grain(p)) return false;
    // the TMA form runs segments with rows or state off alignment by a phase on
    // the scalar path (the realigned one would raise its registers): launches
    // made mostly of them go to the LDG form
    if (phased_chunks * 8 > step_chunks) return false;
  } else if (!copy) {
    return false;
  }
  // likewise copies whose source and destination are not both 16-byte aligned
  // (the TMA form copies them on the narrow path, the LDG form realigns them)
  if (narrow_chunks * 8 > copy_chunks) return false;
  return p.total_chunks >=
         static_cast<int64_t>(step ? kTmaMinStepChunksPerBlock : kTmaMinChunksPerBlock) * tma_grid;
}

// A TMA launch whose step segments have gradient rows spanning 3 GiB or more
// of addresses stages them in interleaved quarter-chunk copies (the second
// instantiation of the kernel). Measured on GB300 (interleaved A/B, W = 8,
// every launch forced to one form or the other): one FlatParameter of 2.5e8
// to 1e9 elements (rows 0.5 to 2 GB apart, spans 3.3 to 13 GiB) ran 2.5-3.1 %
// faster with interleaved 1 KB pieces than with one 4 KB copy per row, likely
// DRAM bank mapping, and the 7B local-rank step (rows 0.52 GB apart, 3.4 GiB)
// 0.1-0.5 %; GPT-2 small (13 units, spans near 0.1 GiB) ran 2 % slower with
// four times as many copies, a 5e7-element FlatParameter 1.4 % and the Llama
// block (2.6 GiB) 1 % slower on one box of three. Below 3 GiB the results
// are mixed (a 2e8-element FlatParameter, 2.6 GiB, gained 2.5 %), so the rule
// keeps the one-copy form there.
constexpr uintptr_t kInterleaveSpread = uintptr_t(3) << 30;

// The split element mapping (Map<true>) for LDG launches whose elementwise
// traffic is mostly fp32 state: Adam segments, and step segments whose replicas'
// state (24 bytes per element each) is at least six times their W bf16
// gradient rows (2 bytes each), i.e. 2 nrep >= W. Reduce segments (W rows in,
// 4 bytes out) keep the other mapping, and so does any launch holding one.
bool wants_split(const Params& p) {
  bool any = false;
  for (int k = 0; k < p.nseg; ++k) {
    const Seg& d = p.seg[k];
    if (d.kind == kAdam) {
      if (d.width == kPhased) return false;  // the realigned path has the consecutive mapping
      any = true;
    } else if (d.kind == kStep) {
      if (2 * d.nrep < p.s.w) return false;
      if (d.width == kPhased) return false;  // the realigned path has the consecutive mapping
      any = true;
    } else if (d.kind == kReduce) {
      return false;
    }
  }
  return any;
}

// (W = 8 launches only: the W = 16 instantiation copies one piece per array.)
bool wants_interleave(const Params& p) { return p.s.w == 8 && max_row_span(p) >= kInterleaveSpread; }

}  // namespace

int launch(const SegmentList& list, const Scalars& s, cudaStream_t stream, int* count, int* tma_count,
           int* interleaved_count) {
  if (count) *count = 0;
  if (tma_count) *tma_count = 0;
  if (interleaved_count) *interleaved_count = 0;
  if (list.seg.empty()) return FSDP_OK;
  const int variant = variant_of(s.w);
  int err = FSDP_OK;
  // the TMA form's grid: one block per SM (its pipeline fills 224 KB of shared memory)
  int tma_cap = 0;
  if (count) {
    int dev = 0, sms = 0;
    tma_cap = (cudaGetDevice(&dev) == cudaSuccess &&
               cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
                  ? sms
                  : 152;
  } else {
    tma_cap = grid_capacity(kTmaVariant, &err);
    if (err != FSDP_OK) return err;
  }
  // ~27 KB: kept off the stack. Entries past this launch's nseg segments and
  // their pointers are left as earlier launches wrote them: the kernels never read
  // them (a chunk's segment index stays below nseg), so they are not cleared
  // (measured on GB300: clearing cost 0.17 us of a 4.65 us call).
  static thread_local Params p;
  size_t i = 0;
  while (i < list.seg.size()) {
    p.s = s;
    int nseg = 0, nptr = 0;
    int64_t chunks = 0;
    while (i < list.seg.size() && nseg < kMaxSeg) {
      const int np = list.pool_size(i);
      if (nptr + np > kMaxPtr) break;
      Seg d = list.seg[i];
      for (int k = 0; k < np; ++k) p.ptr[nptr + k] = list.ptr[d.ptr + k];
      d.ptr = nptr;
      chunks += chunks_of(d);
      d.chunk_end = chunks;
      p.seg[nseg++] = d;
      nptr += np;
      ++i;
    }
    p.nseg = nseg;
    p.total_chunks = chunks;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    p.inject_tx = 0;
    const bool tma = use_tma(p, tma_cap);
    const bool tma16 = tma && p.s.w == 16 && has_step(p);
    if (count) {
      ++*count;
      if (tma && tma_count) ++*tma_count;
      if (tma && !tma16 && interleaved_count && wants_interleave(p)) ++*interleaved_count;
      continue;
    }
    if (tma16) {
      const int cap16 = grid_capacity(kTma16Variant, &err);
      if (err != FSDP_OK) return err;
      if (launch_tma_form<16, false>(p, static_cast<int>(std::min<int64_t>(chunks, cap16)), stream) != cudaSuccess)
        return FSDP_ECUDA;
      continue;
    }
    if (tma) {
      bool copies = false;
      for (int k = 0; k < p.nseg; ++k) copies = copies || p.seg[k].kind == kCopy;
      const int grid = static_cast<int>(std::min<int64_t>(chunks, tma_cap));
      if (launch_tma(p, grid, stream, wants_interleave(p), copies) != cudaSuccess) return FSDP_ECUDA;
      continue;
    }
    bool realign = false;
    for (int k = 0; k < p.nseg; ++k) {
      const Seg& d = p.seg[k];
      const bool bytes = d.kind == kCopy || d.kind == kZero;
      realign = realign || (bytes ? d.width != 16 : d.width == kPhased);
    }
    if (realign) {
      const int cap = grid_capacity(variant + kRealignVariants, &err);
      if (err != FSDP_OK) return err;
      const int grid = static_cast<int>(std::min<int64_t>(chunks, cap));
      cudaError_t e;
      switch (variant) {
        case 0: e = launch_variant<1, false, true>(p, grid, stream); break;
        case 1: e = launch_variant<2, false, true>(p, grid, stream); break;
        case 2: e = launch_variant<4, false, true>(p, grid, stream); break;
        case 3: e = launch_variant<8, false, true>(p, grid, stream); break;
        case 4: e = launch_variant<16, false, true>(p, grid, stream); break;
        default: e = launch_variant<0, false, true>(p, grid, stream); break;
      }
      if (e != cudaSuccess) return FSDP_ECUDA;
      continue;
    }
    const bool split = wants_split(p);
    const int cap = grid_capacity(split ? variant + kSplitVariants : variant, &err);
    if (err != FSDP_OK) return err;
    const int grid = static_cast<int>(std::min<int64_t>(chunks, cap));
    cudaError_t e;
    switch (variant * 2 + (split ? 1 : 0)) {
      case 0: e = launch_variant<1, false>(p, grid, stream); break;
      case 1: e = launch_variant<1, true>(p, grid, stream); break;
      case 2: e = launch_variant<2, false>(p, grid, stream); break;
      case 3: e = launch_variant<2, true>(p, grid, stream); break;
      case 4: e = launch_variant<4, false>(p, grid, stream); break;
      case 5: e = launch_variant<4, true>(p, grid, stream); break;
      case 6: e = launch_variant<8, false>(p, grid, stream); break;
      case 7: e = launch_variant<8, true>(p, grid, stream); break;
      case 8: e = launch_variant<16, false>(p, grid, stream); break;
      case 9: e = launch_variant<16, true>(p, grid, stream); break;
      case 10: e = launch_variant<0, false>(p, grid, stream); break;
      default: e = launch_variant<0, true>(p, grid, stream); break;
    }
    if (e != cudaSuccess) return FSDP_ECUDA;
  }
  return FSDP_OK;
}

// ------------------------------------------------------------ validation

bool layout_ok(const fsdp_layout_t* L) {
  if (!L) return false;
  const int64_t w = L->world_size;
  if (w < 1 || w > FSDP_MAX_WORLD || L->shard_factor < 1 || w % L->shard_factor != 0) return false;
  if (L->n_tensors < 1 || L->numel < 0) return false;
  if (L->numel > INT64_MAX - w) return false;
  if (L->padded_numel != (L->numel + w - 1) / w * w) return false;
  return L->shard_numel * L->shard_factor == L->padded_numel;
}

int make_scalars(const fsdp_adam_t* h, int w, Scalars* s) {
  if (!h) return FSDP_EINVAL;
  if (h->step < 1 || h->weight_decay != 0.0) return FSDP_EINVAL;
  if (!(h->beta1 >= 0.0 && h->beta1 < 1.0) || !(h->beta2 >= 0.0 && h->beta2 < 1.0)) return FSDP_EINVAL;
  if (!(h->eps >= 0.0) || !std::isfinite(h->eps) || !std::isfinite(h->lr)) return FSDP_EINVAL;
  const double t = static_cast<double>(h->step);
  s->lr = static_cast<float>(h->lr);
  s->b1 = static_cast<float>(h->beta1);
  s->b2 = static_cast<float>(h->beta2);
  s->eps = static_cast<float>(h->eps);
  s->omb1 = static_cast<float>(1.0 - h->beta1);
  s->omb2 = static_cast<float>(1.0 - h->beta2);
  s->bc1 = static_cast<float>(1.0 - std::pow(h->beta1, t));
  s->bc2 = static_cast<float>(1.0 - std::pow(h->beta2, t));
  if (!(s->bc1 > 0.0f) || !(s->bc2 > 0.0f)) return FSDP_EINVAL;
  s->w = w;
  s->inv_w = (w > 0 && (w & (w - 1)) == 0) ? 1.0f / static_cast<float>(w) : 0.0f;
  return FSDP_OK;
}

Scalars reduce_only_scalars(int w) {
  Scalars s{};
  s.w = w;
  s.inv_w = (w & (w - 1)) == 0 ? 1.0f / static_cast<float>(w) : 0.0f;
  return s;
}

namespace {

// Appends one unit's fused-step segments; checks pointers and aliasing.
int build_unit(const fsdp_unit_args_t& u, int32_t rb, int32_t re, SegmentList& list,
               AliasCheck& alias) {
  const fsdp_layout_t* L = u.layout;
  const int W = L->world_size, F = L->shard_factor, R = W / F;
  const int64_t S = L->shard_numel, padded = L->padded_numel;
  if (padded == 0) return FSDP_OK;
  if (!u.grads || !u.master || !u.exp_avg || !u.exp_avg_sq || !u.full_out) return FSDP_EINVAL;
  for (int k = 0; k < W; ++k) {
    if (!u.grads[k]) return FSDP_EINVAL;
    alias.input(u.grads[k], padded * 2);
  }
  // positions with at least one owned replica, each reduced once
  std::vector<const void*> ptrs;
  for (int p = 0; p < F; ++p) {
    ptrs.clear();
    for (int k = 0; k < W; ++k) ptrs.push_back(u.grads[k] + p * S);
    int nrep = 0;
    for (int g = 0; g < R; ++g) {
      const int r = g * F + p;
      if (r < rb || r >= re) continue;
      const int o = r - rb;
      float* mp = u.master[o];
      float* mm = u.exp_avg[o];
      float* mv = u.exp_avg_sq[o];
      uint16_t* full = u.full_out[g];
      if (!mp || !mm || !mv || !full) return FSDP_EINVAL;
      alias.output(mp, S * 4);
      alias.output(mm, S * 4);
      alias.output(mv, S * 4);
      ptrs.push_back(mp);
      ptrs.push_back(mm);
      ptrs.push_back(mv);
      ptrs.push_back(full + p * S);
      ++nrep;
    }
    if (nrep > 0) list.add_elementwise(kStep, S, nrep, ptrs);
  }
  // gather the non-owned positions of every group that holds an owned rank
  for (int g = 0; g < R; ++g) {
    const int lo = g * F, hi = lo + F;
    if (hi <= rb || lo >= re) continue;
    uint16_t* full = u.full_out[g];
    alias.output(full, padded * 2);
    for (int p = 0; p < F; ++p) {
      const int r = lo + p;
      if (r >= rb && r < re) continue;
      if (!u.other_shards || !u.other_shards[r]) return FSDP_EINVAL;
      const uint16_t* src = u.other_shards[r];
      if (src == full + p * S) continue;  // already in place
      alias.input(src, S * 2);
      list.add_bytes(kCopy, src, full + p * S, S * 2);
    }
  }
  return FSDP_OK;
}

}  // namespace
}  // namespace fsdp

using namespace fsdp;

namespace {

constexpr int64_t kSplitMinChunksPerSm = 256;  // see the split in grouped()

int grouped(const fsdp_unit_args_t* units, int32_t n_units, int32_t rank_begin, int32_t rank_end,
            const fsdp_adam_t* adam, cudaStream_t stream, int* count, int* tma_count = nullptr,
            int* interleaved_count = nullptr) {
  if (count) *count = 0;
  if (tma_count) *tma_count = 0;
  if (interleaved_count) *interleaved_count = 0;
  if (n_units < 0 || (n_units > 0 && !units)) return FSDP_EINVAL;
  if (n_units == 0) return FSDP_OK;
  const fsdp_layout_t* L0 = units[0].layout;
  if (!layout_ok(L0)) return FSDP_EINVAL;
  const int W = L0->world_size, F = L0->shard_factor;
  if (rank_begin < 0 || rank_end > W || rank_begin >= rank_end) return FSDP_EINVAL;
  Scalars s{};
  if (adam) {
    if (int rc = make_scalars(adam, W, &s)) return rc;
  } else {
    if (!count) return FSDP_EINVAL;
    s = reduce_only_scalars(W);
  }
  SegmentList list;
  AliasCheck alias;
  for (int32_t i = 0; i < n_units; ++i) {
    const fsdp_layout_t* L = units[i].layout;
    if (!layout_ok(L) || L->world_size != W || L->shard_factor != F) return FSDP_EINVAL;
    if (int rc = build_unit(units[i], rank_begin, rank_end, list, alias)) return rc;
  }
  if (!alias.ok()) return FSDP_EALIAS;
  // Every unit's step segment first, then every gather: the launch then changes
  // from step chunks to copy chunks once instead of once per unit, each change
  // costing the pipeline about 2 us. Measured on GB300 (interleaved A/B, the
  // local-rank step per unit -> steps first): the 7B step 8.567 -> 8.451 ms and
  // 8.562 -> 8.471 ms (two boxes), four Llama blocks 1.031 -> 1.006 ms, GPT-2
  // small 0.173 -> 0.165 ms; the gathers first instead were 2 % slower than this
  // on the last two and equal on the 7B step.
  // (the aligned and off-alignment lists below are built only when some
  // segment is off alignment: the common launch pays for one list)
  auto off_alignment = [](const Seg& d) { return d.kind == kCopy ? d.width != 16 : d.width == kPhased; };
  bool any_off = false;
  for (const Seg& d : list.seg) any_off = any_off || off_alignment(d);
  SegmentList ordered, aligned, off;
  ordered.seg.reserve(list.seg.size());
  ordered.ptr.reserve(list.ptr.size());
  for (int pass = 0; pass < 2; ++pass) {
    for (size_t i = 0; i < list.seg.size(); ++i) {
      const Seg& d = list.seg[i];
      if ((pass == 0) != (d.kind == kStep)) continue;
      for (SegmentList* to : {&ordered, any_off ? (off_alignment(d) ? &off : &aligned) : nullptr}) {
        if (!to) continue;
        Seg e = d;
        e.ptr = static_cast<int32_t>(to->ptr.size());
        to->seg.push_back(e);
        const int np = list.pool_size(i);
        for (int k = 0; k < np; ++k) to->ptr.push_back(list.ptr[d.ptr + k]);
      }
    }
  }
  // A launch that holds too many segments off alignment for the TMA form (its
  // realigned paths are in the LDG form only) is split in two when its aligned
  // segments alone make a TMA launch of at least kSplitMinChunksPerSm chunks per
  // SM: those first, then the others on the LDG form (the units are
  // independent, as the order above already assumes). Measured on GB300
  // (interleaved A/B, one LDG launch -> TMA launch + LDG launch; local-rank
  // steps of four aligned units and two with odd shard lengths): aligned
  // segments of 5.8 GB (about 740 chunks per SM) 0.774 -> 0.865 of the copy
  // peak, of 2.1 GB (about 270 per SM) 0.793 -> 0.870, of 0.73 GB (about 92 per
  // SM) 0.761 -> 0.728: the second launch costs tens of microseconds.
  int64_t aligned_chunks = 0;
  int dev = 0, sms = 0;
  if (!off.seg.empty()) {
    for (const Seg& d : aligned.seg) aligned_chunks += chunks_of(d);
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 152;
  }
  if (!off.seg.empty() && aligned_chunks >= kSplitMinChunksPerSm * sms) {
    int c = 0, t = 0, c_al = 0, t_al = 0, i_al = 0;
    if (int rc = launch(ordered, s, nullptr, &c, &t, nullptr)) return rc;
    if (int rc = launch(aligned, s, nullptr, &c_al, &t_al, &i_al)) return rc;
    if (t < c && t_al == c_al) {
      if (!count) {
        if (int rc = launch(aligned, s, stream, nullptr, nullptr, nullptr)) return rc;
        return launch(off, s, stream, nullptr, nullptr, nullptr);
      }
      int c_off = 0, t_off = 0, i_off = 0;
      if (int rc = launch(off, s, nullptr, &c_off, &t_off, &i_off)) return rc;
      *count = c_al + c_off;
      if (tma_count) *tma_count = t_al + t_off;
      if (interleaved_count) *interleaved_count = i_al + i_off;
      return FSDP_OK;
    }
  }
  return launch(ordered, s, stream, count, tma_count, interleaved_count);
}

}  // namespace

extern "C" int fsdp_shard_step_grouped(const fsdp_unit_args_t* units, int32_t n_units,
                                       int32_t rank_begin, int32_t rank_end,
                                       const fsdp_adam_t* adam, fsdp_stream_t stream) {
  return grouped(units, n_units, rank_begin, rank_end, adam, reinterpret_cast<cudaStream_t>(stream),
                 nullptr);
}

extern "C" int fsdp_shard_step_grouped_launches(const fsdp_unit_args_t* units, int32_t n_units,
                                                int32_t rank_begin, int32_t rank_end,
                                                int32_t* launches_out) {
  return fsdp_shard_step_grouped_plan(units, n_units, rank_begin, rank_end, launches_out, nullptr, nullptr);
}

extern "C" int fsdp_shard_step_grouped_plan(const fsdp_unit_args_t* units, int32_t n_units, int32_t rank_begin,
                                            int32_t rank_end, int32_t* launches_out, int32_t* tma_launches_out,
                                            int32_t* tma_interleaved_out) {
  if (!launches_out) return FSDP_EINVAL;
  int count = 0, tma = 0, interleaved = 0;
  const int rc = grouped(units, n_units, rank_begin, rank_end, nullptr, nullptr, &count, &tma, &interleaved);
  if (rc == FSDP_OK) {
    *launches_out = count;
    if (tma_launches_out) *tma_launches_out = tma;
    if (tma_interleaved_out) *tma_interleaved_out = interleaved;
  }
  return rc;
}

extern "C" int fsdp_device_status(int32_t clear, uint32_t* status_out) {
  if (!status_out) return FSDP_EINVAL;
  // the symbol copy runs on the legacy default stream, which does not wait for
  // non-blocking streams: finish all work of the device first
  if (cudaDeviceSynchronize() != cudaSuccess) return FSDP_ECUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fsdp_status, sizeof(v)) != cudaSuccess) return FSDP_ECUDA;
  if (clear) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_fsdp_status, &z, sizeof(z)) != cudaSuccess) return FSDP_ECUDA;
  }
  *status_out = v;
  return FSDP_OK;
}

extern "C" int fsdp_selftest_wait_timeout(const void* src, void* dst, int64_t bytes, int64_t wait_limit_ns,
                                          fsdp_stream_t stream, uint32_t* status_out) {
  if (!src || !dst || !status_out || bytes < kChunkBytes || bytes > (int64_t(1) << 30)) return FSDP_EINVAL;
  if (wait_limit_ns <= 0 || wait_limit_ns > 10000000000ll) return FSDP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) return FSDP_EINVAL;
  AliasCheck alias;
  alias.output(dst, bytes);
  alias.input(src, bytes);
  if (!alias.ok()) return FSDP_EALIAS;
  int err = FSDP_OK;
  const int cap = grid_capacity(kTmaVariant, &err);
  if (err != FSDP_OK) return err;
  const unsigned int z = 0;
  if (cudaMemcpyToSymbol(g_fsdp_status, &z, sizeof(z)) != cudaSuccess) return FSDP_ECUDA;
  SegmentList list;
  list.add_bytes(kCopy, src, dst, bytes & ~int64_t(15));
  static thread_local Params p;
  std::memset(&p, 0, sizeof(p));
  p.s = reduce_only_scalars(8);
  p.nseg = 1;
  p.seg[0] = list.seg[0];
  p.seg[0].ptr = 0;
  p.ptr[0] = list.ptr[0];
  p.ptr[1] = list.ptr[1];
  p.total_chunks = (p.seg[0].n + kChunkBytes - 1) / kChunkBytes;
  p.seg[0].chunk_end = p.total_chunks;
  p.wait_limit_ns = static_cast<uint64_t>(wait_limit_ns);
  p.inject_tx = 16;  // block 0's first stage expects 16 bytes that no copy delivers
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_tma(p, static_cast<int>(std::min<int64_t>(p.total_chunks, cap)), st) != cudaSuccess) return FSDP_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FSDP_ECUDA;
  return fsdp_device_status(1, status_out);
}

extern "C" int fsdp_shard_step(const uint16_t* const* grads, const fsdp_layout_t* layout,
                               int32_t rank_begin, int32_t rank_end, float* const* master,
                               float* const* exp_avg, float* const* exp_avg_sq,
                               const uint16_t* const* other_shards, uint16_t* const* full_out,
                               const fsdp_adam_t* adam, fsdp_stream_t stream) {
  fsdp_unit_args_t u{layout, grads, master, exp_avg, exp_avg_sq, other_shards, full_out};
  return fsdp_shard_step_grouped(&u, 1, rank_begin, rank_end, adam, stream);
}

extern "C" int fsdp_reduce_scatter_ranks(const uint16_t* const* grads, const fsdp_layout_t* L,
                                         int32_t rank_begin, int32_t rank_end, float* const* grad_shards_out,
                                         fsdp_stream_t stream) {
  if (!layout_ok(L) || !grads || !grad_shards_out) return FSDP_EINVAL;
  const int W = L->world_size, F = L->shard_factor;
  if (rank_begin < 0 || rank_end > W || rank_begin >= rank_end) return FSDP_EINVAL;
  const int64_t S = L->shard_numel;
  if (S == 0) return FSDP_OK;
  AliasCheck alias;
  for (int k = 0; k < W; ++k) {
    if (!grads[k]) return FSDP_EINVAL;
    alias.input(grads[k], L->padded_numel * 2);
  }
  // one reduce segment per owned rank, in rank order
  SegmentList list;
  std::vector<const void*> ptrs;
  for (int r = rank_begin; r < rank_end; ++r) {
    float* out = grad_shards_out[r - rank_begin];
    if (!out) return FSDP_EINVAL;
    alias.output(out, S * 4);
    const int p = r % F;
    ptrs.clear();
    for (int k = 0; k < W; ++k) ptrs.push_back(grads[k] + p * S);
    ptrs.push_back(out);
    list.add_elementwise(kReduce, S, 0, ptrs);
  }
  if (!alias.ok()) return FSDP_EALIAS;
  return launch(list, reduce_only_scalars(W), reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fsdp_reduce_scatter(const uint16_t* const* grads, const fsdp_layout_t* L,
                                   int32_t rank, float* grad_shard_out, fsdp_stream_t stream) {
  if (!grad_shard_out || rank < 0 || rank >= FSDP_MAX_WORLD) return FSDP_EINVAL;
  return fsdp_reduce_scatter_ranks(grads, L, rank, rank + 1, &grad_shard_out, stream);
}

extern "C" int fsdp_adam_shard_step_grouped(const fsdp_adam_shard_t* shards, int32_t n_shards,
                                            const fsdp_adam_t* adam, fsdp_stream_t stream) {
  if (n_shards < 0 || (n_shards > 0 && !shards)) return FSDP_EINVAL;
  Scalars s{};
  if (int rc = make_scalars(adam, 1, &s)) return rc;
  AliasCheck alias;
  SegmentList list;
  for (int32_t i = 0; i < n_shards; ++i) {
    const fsdp_adam_shard_t& a = shards[i];
    if (a.n < 0) return FSDP_EINVAL;
    if (a.n == 0) continue;
    if (!a.master || !a.exp_avg || !a.exp_avg_sq || !a.grad_shard) return FSDP_EINVAL;
    alias.output(a.master, a.n * 4);
    alias.output(a.exp_avg, a.n * 4);
    alias.output(a.exp_avg_sq, a.n * 4);
    if (a.bf16_shard_out) alias.output(a.bf16_shard_out, a.n * 2);
    alias.input(a.grad_shard, a.n * 4);
    list.add_elementwise(kAdam, a.n, 1, {a.grad_shard, a.master, a.exp_avg, a.exp_avg_sq, a.bf16_shard_out});
  }
  if (!alias.ok()) return FSDP_EALIAS;
  return launch(list, s, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fsdp_adam_shard_step(float* master, float* exp_avg, float* exp_avg_sq,
                                    const float* grad_shard, int64_t n, const fsdp_adam_t* adam,
                                    uint16_t* bf16_shard_out, fsdp_stream_t stream) {
  const fsdp_adam_shard_t one{master, exp_avg, exp_avg_sq, grad_shard, bf16_shard_out, n};
  return fsdp_adam_shard_step_grouped(&one, 1, adam, stream);
}

extern "C" int fsdp_all_gather(const uint16_t* const* shards, const fsdp_layout_t* L,
                               uint16_t* full_out, fsdp_stream_t stream) {
  if (!layout_ok(L) || !shards || !full_out) return FSDP_EINVAL;
  const int F = L->shard_factor;
  const int64_t S = L->shard_numel;
  if (S == 0) return FSDP_OK;
  AliasCheck alias;
  alias.output(full_out, L->padded_numel * 2);
  SegmentList list;
  for (int k = 0; k < F; ++k) {
    if (!shards[k]) return FSDP_EINVAL;
    if (shards[k] == full_out + k * S) continue;
    alias.input(shards[k], S * 2);
    list.add_bytes(kCopy, shards[k], full_out + k * S, S * 2);
  }
  if (!alias.ok()) return FSDP_EALIAS;
  return launch(list, reduce_only_scalars(1), reinterpret_cast<cudaStream_t>(stream));
}

namespace {

int elem_size_of(int32_t dtype) {
  return dtype == FSDP_DTYPE_F32 ? 4 : dtype == FSDP_DTYPE_BF16 ? 2 : 0;
}

bool offsets_ok(const fsdp_layout_t* L, const int64_t* offsets) {
  if (!offsets || offsets[0] != 0 || offsets[L->n_tensors] != L->numel) return false;
  for (int32_t t = 0; t < L->n_tensors; ++t)
    if (offsets[t + 1] < offsets[t]) return false;
  return true;
}

}  // namespace

extern "C" int fsdp_pack_flat(const void* const* tensors, const fsdp_layout_t* L,
                              const int64_t* offsets, int32_t dtype, void* flat_out,
                              fsdp_stream_t stream) {
  const int es = elem_size_of(dtype);
  if (!layout_ok(L) || es == 0 || !tensors || !flat_out || !offsets_ok(L, offsets)) return FSDP_EINVAL;
  auto* flat = static_cast<unsigned char*>(flat_out);
  AliasCheck alias;
  alias.output(flat, L->padded_numel * es);
  SegmentList list;
  for (int32_t t = 0; t < L->n_tensors; ++t) {
    const int64_t bytes = (offsets[t + 1] - offsets[t]) * es;
    if (bytes == 0) continue;
    if (!tensors[t]) return FSDP_EINVAL;
    alias.input(tensors[t], bytes);
    list.add_bytes(kCopy, tensors[t], flat + offsets[t] * es, bytes);
  }
  list.add_bytes(kZero, nullptr, flat + L->numel * es, (L->padded_numel - L->numel) * es);
  if (!alias.ok()) return FSDP_EALIAS;
  return launch(list, reduce_only_scalars(1), reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fsdp_unpack_flat(const void* flat_in, const fsdp_layout_t* L, const int64_t* offsets,
                                int32_t dtype, void* const* tensors_out, fsdp_stream_t stream) {
  const int es = elem_size_of(dtype);
  if (!layout_ok(L) || es == 0 || !tensors_out || !flat_in || !offsets_ok(L, offsets)) return FSDP_EINVAL;
  const auto* flat = static_cast<const unsigned char*>(flat_in);
  AliasCheck alias;
  alias.input(flat, L->padded_numel * es);
  SegmentList list;
  for (int32_t t = 0; t < L->n_tensors; ++t) {
    const int64_t bytes = (offsets[t + 1] - offsets[t]) * es;
    if (bytes == 0) continue;
    if (!tensors_out[t]) return FSDP_EINVAL;
    alias.output(tensors_out[t], bytes);
    list.add_bytes(kCopy, flat + offsets[t] * es, tensors_out[t], bytes);
  }
  if (!alias.ok()) return FSDP_EALIAS;
  return launch(list, reduce_only_scalars(1), reinterpret_cast<cudaStream_t>(stream));
}
