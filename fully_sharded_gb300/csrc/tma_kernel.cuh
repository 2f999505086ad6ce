// TMA form of the segment kernel (sm_103a): bulk copies into a shared-memory
// pipeline, one producer lane and 8 consumer warps per block.
//
// The producer (lane 0 of warp 8) stages each eligible chunk with
// cp.async.bulk (global -> shared; completion counted in bytes on the stage's
// "full" mbarrier) up to kStages chunks ahead; the consumer warps wait on
// that barrier, run the fused step from shared memory and store its results
// to global memory (a staged copy chunk goes back out as one bulk store,
// shared -> global), then release the stage on its "empty" mbarrier. Chunks that
// cannot be staged (misaligned segments, other kinds) are run by the
// consumers from global memory as in segment_kernel.
//
// Instantiations: for W = 8, kInterleave = false stages a step chunk with one
// bulk copy per array and kInterleave = true (the host picks it when a
// launch's gradient rows span 3 GiB or more of addresses) in four rounds of
// quarter chunks over the arrays; for W = 16 (one copy per array, two stages
// of 88 KB), the host picks it for launches whose gradient rows do not all lie
// a multiple of 2 KB apart.
//
// Measured on GB300 against segment_kernel (same chunks, same arithmetic,
// bit-identical results): W = 8 single-replica step launches gain 2-6 %
// (Llama block 1.246 -> 1.179 ms); W <= 4, replica-heavy hybrid steps, short
// launches and launches of reduce chunks lose, so the host uses this form only
// for W = 8 launches made of one-replica step segments (and copies), for W = 16
// ones whose rows are not all 2 KB-aligned to each other (see abi.cu), and for launches of copies
// only (and zero fills: pack, unpack, the gathers; 1-3.5 % faster), with at
// least kTmaMinStepChunksPerBlock (steps) or kTmaMinChunksPerBlock (copies
// only) chunks per block. Measured on GB300 (interleaved A/B, LDG -> TMA form):
// W = 8 steps of 64-96 chunks per block 1.4-3.2 % faster and W = 16 ones
// 0.5-1.5 %, 32 chunks per block 1-1.5 % slower; copies alone of 64 chunks per
// block 3.5 % slower, of 128 and more faster.
//
// Every mbarrier wait is bounded in time (Params::wait_limit_ns, read from
// %globaltimer): when a wait runs out the block sets bit 0 of g_fsdp_status,
// every thread of the block stops, the producer waits (again bounded) for the
// bulk copies it has issued, and the block returns. This never happens in a
// correct run; fsdp_selftest_wait_timeout provokes it on purpose.
//
// Requires g_fsdp_status (a __device__ unsigned int) to be defined before
// this header is included.
#pragma once

#include "segment_kernel.cuh"

namespace fsdp {

constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaThreads = (kTmaConsumerWarps + 1) * 32;
constexpr int kTmaStages = 4;  // 4 x 56 KB at W = 8 (W = 16: 2 x 88 KB)
constexpr int kTmaMinChunksPerBlock = 128;     // launches of copies only
constexpr int kTmaMinStepChunksPerBlock = 64;  // launches with step chunks
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

template <int W>
struct TmaCfg {
  static constexpr int kStages = W > 8 ? 2 : kTmaStages;
  static constexpr int kRowBytes = int(kChunkElems) * 2;
  static constexpr int kStateBytes = int(kChunkElems) * 4;
  static constexpr int kStepBytes = W * kRowBytes + 3 * kStateBytes;
  static constexpr int kStageBytes = kStepBytes > int(kChunkBytes) ? kStepBytes : int(kChunkBytes);
  static constexpr int kSmemBytes = kStages * kStageBytes;
};
static_assert(TmaCfg<8>::kSmemBytes + 128 <= 232448, "TMA pipeline exceeds 227 KB of shared memory");
static_assert(TmaCfg<16>::kSmemBytes + 128 <= 232448, "TMA pipeline exceeds 227 KB of shared memory");

struct Cursor {
  int s = 0;
  int64_t first = 0;
  __device__ __forceinline__ const Seg& at(const Params& p, int64_t c, int64_t& local) {
    while (c >= p.seg[s].chunk_end) {
      first = p.seg[s].chunk_end;
      ++s;
    }
    local = c - first;
    return p.seg[s];
  }
};

__device__ __forceinline__ uint32_t sm_addr(const void* q) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(q));
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_arrive(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// 16-byte aligned global source, shared destination and size (checked by the caller).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Bulk store of `bytes` from shared memory (16-byte aligned) to global memory
// (16-byte aligned, bytes a multiple of 16), as its own bulk async-group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The issuing thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The issuing thread's bulk stores have completed their writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Waits for the phase of `parity` to complete. False when the block aborted
// or the time limit ran out (then the abort flag and the status word are set).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(&g_fsdp_status, 1u);
      return false;
    }
  }
}

// Bytes staged for a chunk (0: the consumers read it from global memory);
// issues the bulk copies when `issue` is set. Rows at k * kRowBytes, state
// array a at W * kRowBytes + a * kStateBytes, copy data at 0. *staged_n is
// the number of staged elements (step) or bytes (copy). kInterleave: a step
// chunk is copied in four rounds over its arrays (a quarter chunk of every row,
// then of every state array) instead of one copy per array.
template <int W, bool kInterleave>
__device__ __forceinline__ uint32_t tma_chunk(const Params& p, const Seg& d, int64_t local, unsigned char* stage,
                                              uint32_t bar, bool issue, uint32_t extra_tx, int64_t* staged_n) {
  *staged_n = 0;
  if (d.width != 16) return 0;
  if (d.kind == kStep && d.nrep == 1) {
    const int64_t e0 = local * kChunkElems;
    int64_t nc = d.n - e0;
    if (nc > kChunkElems) nc = kChunkElems;
    nc &= ~int64_t(7);  // whole 16-byte rows; the last < 8 elements go through global memory
    if (nc <= 0) return 0;
    *staged_n = nc;
    const uint32_t total = static_cast<uint32_t>(nc * (2 * W + 12));
    if (!issue) return total;
    mbar_expect_tx_arrive(bar, total + extra_tx);
    if constexpr (kInterleave) {
      constexpr int64_t kPiece = kChunkElems / 4;
      for (int64_t q0 = 0; q0 < nc; q0 += kPiece) {
        const int64_t pe = (nc - q0 < kPiece) ? nc - q0 : kPiece;  // a multiple of 8
#pragma unroll
        for (int k = 0; k < W; ++k)
          bulk_load(sm_addr(stage + k * TmaCfg<W>::kRowBytes + q0 * 2),
                    static_cast<const uint16_t*>(p.ptr[d.ptr + k]) + e0 + q0, static_cast<uint32_t>(pe * 2), bar);
#pragma unroll
        for (int a = 0; a < 3; ++a)
          bulk_load(sm_addr(stage + W * TmaCfg<W>::kRowBytes + a * TmaCfg<W>::kStateBytes + q0 * 4),
                    static_cast<const float*>(p.ptr[d.ptr + W + a]) + e0 + q0, static_cast<uint32_t>(pe * 4), bar);
      }
    } else {
#pragma unroll
      for (int k = 0; k < W; ++k)
        bulk_load(sm_addr(stage + k * TmaCfg<W>::kRowBytes), static_cast<const uint16_t*>(p.ptr[d.ptr + k]) + e0,
                  static_cast<uint32_t>(nc * 2), bar);
#pragma unroll
      for (int a = 0; a < 3; ++a)
        bulk_load(sm_addr(stage + W * TmaCfg<W>::kRowBytes + a * TmaCfg<W>::kStateBytes),
                  static_cast<const float*>(p.ptr[d.ptr + W + a]) + e0, static_cast<uint32_t>(nc * 4), bar);
    }
    return total;
  }
  if (d.kind == kCopy) {
    const int64_t b0 = local * kChunkBytes;
    int64_t nb = d.n - b0;
    if (nb > kChunkBytes) nb = kChunkBytes;
    nb &= ~int64_t(15);
    if (nb <= 0) return 0;
    *staged_n = nb;
    if (!issue) return static_cast<uint32_t>(nb);
    mbar_expect_tx_arrive(bar, static_cast<uint32_t>(nb) + extra_tx);
    bulk_load(sm_addr(stage), static_cast<const unsigned char*>(p.ptr[d.ptr]) + b0, static_cast<uint32_t>(nb), bar);
    return static_cast<uint32_t>(nb);
  }
  return 0;
}

// The consumers take 8 consecutive elements per thread (Map<false>): measured on
// GB300, the split mapping of segment_kernel (two groups of 4, two 8-byte
// shared-memory reads per row) made the Llama block's step 4.6 % slower here
// (1.189 -> 1.244 ms; the 7B local-rank step 8.562 -> 8.580 ms). Each thread
// stores its 8 new fp32 values of an array as one 32-byte sector when the
// three state arrays are 32-byte aligned (else as two float4): a warp's store
// then fills 32 whole sectors in one instruction instead of half of them in
// each of two (interleaved A/B on GB300: Llama block 1.193 -> 1.183 ms, the
// 1e8-element W = 8 step 0.596 -> 0.588 ms, the 1e9-element W = 16 step
// 8.461 -> 8.344 ms, the 7B step unchanged at 8.56-8.57 ms). The LDG form
// keeps its 16-byte accesses: there 32-byte loads and stores were 2-5 % slower.
template <int W>
__device__ __forceinline__ void tma_consume_step(const Params& p, const Seg& d, int64_t local,
                                                 const unsigned char* stage, int64_t nc) {
  const int64_t e0 = local * kChunkElems;
  const int64_t j = int64_t(threadIdx.x) * kVec;
  if (j + kVec <= nc) {
    float g[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k)
      add_bf16x8(g, *reinterpret_cast<const uint4*>(stage + k * TmaCfg<W>::kRowBytes + j * 2));
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = mean_of<W>(g[i], p.s);
    const unsigned char* sb = stage + W * TmaCfg<W>::kRowBytes;
    State8 st;
    const float4 a0 = *reinterpret_cast<const float4*>(sb + j * 4);
    const float4 a1 = *reinterpret_cast<const float4*>(sb + j * 4 + 16);
    const float4 b0 = *reinterpret_cast<const float4*>(sb + TmaCfg<W>::kStateBytes + j * 4);
    const float4 b1 = *reinterpret_cast<const float4*>(sb + TmaCfg<W>::kStateBytes + j * 4 + 16);
    const float4 c0 = *reinterpret_cast<const float4*>(sb + 2 * TmaCfg<W>::kStateBytes + j * 4);
    const float4 c1 = *reinterpret_cast<const float4*>(sb + 2 * TmaCfg<W>::kStateBytes + j * 4 + 16);
    st.p[0] = a0.x; st.p[1] = a0.y; st.p[2] = a0.z; st.p[3] = a0.w;
    st.p[4] = a1.x; st.p[5] = a1.y; st.p[6] = a1.z; st.p[7] = a1.w;
    st.m[0] = b0.x; st.m[1] = b0.y; st.m[2] = b0.z; st.m[3] = b0.w;
    st.m[4] = b1.x; st.m[5] = b1.y; st.m[6] = b1.z; st.m[7] = b1.w;
    st.v[0] = c0.x; st.v[1] = c0.y; st.v[2] = c0.z; st.v[3] = c0.w;
    st.v[4] = c1.x; st.v[5] = c1.y; st.v[6] = c1.z; st.v[7] = c1.w;
    const int b = d.ptr + W;
#pragma unroll
    for (int i = 0; i < 8; ++i) adam1(g[i], st.p[i], st.m[i], st.v[i], p.s);
    float* mp = static_cast<float*>(const_cast<void*>(p.ptr[b]));
    float* mm = static_cast<float*>(const_cast<void*>(p.ptr[b + 1]));
    float* mv = static_cast<float*>(const_cast<void*>(p.ptr[b + 2]));
    uint16_t* out = static_cast<uint16_t*>(const_cast<void*>(p.ptr[b + 3]));
    const int64_t e = e0 + j;  // a multiple of 8 elements: 32 bytes of fp32
    if (((reinterpret_cast<uintptr_t>(mp) | reinterpret_cast<uintptr_t>(mm) | reinterpret_cast<uintptr_t>(mv)) &
         31u) == 0) {
      st_stream_f8(mp + e, st.p);
      st_stream_f8(mm + e, st.m);
      st_stream_f8(mv + e, st.v);
      if (out)
        st_stream_u4(out + e, make_uint4(bf16x2_rn(st.p[0], st.p[1]), bf16x2_rn(st.p[2], st.p[3]),
                                         bf16x2_rn(st.p[4], st.p[5]), bf16x2_rn(st.p[6], st.p[7])));
    } else {
      store_state8<false>(st, mp, mm, mv, out, e);
    }
  } else {
    // this thread's elements beyond the staged part (the chunk's last < 8)
    int64_t end = d.n - e0;
    if (end > kChunkElems) end = kChunkElems;
    const int64_t lo = j > nc ? j : nc;
    const int64_t hi = j + kVec < end ? j + kVec : end;
    for (int64_t q = lo; q < hi; ++q) step_scalar<W>(p, d, e0 + q);
  }
}

// A staged copy chunk goes back out as one bulk store issued by thread 0, so
// the consumer warps never handle copy data; the thread copies the chunk's
// last < 16 bytes itself and waits until the store has read the stage before
// its warp releases it.
__device__ __forceinline__ void tma_store_copy(const Params& p, const Seg& d, int64_t local,
                                               const unsigned char* stage, int64_t nb) {
  if (threadIdx.x != 0) return;
  const int64_t b0 = local * kChunkBytes;
  unsigned char* dst = static_cast<unsigned char*>(const_cast<void*>(p.ptr[d.ptr + 1]));
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  bulk_store(dst + b0, sm_addr(stage), static_cast<uint32_t>(nb));
  const unsigned char* src = static_cast<const unsigned char*>(p.ptr[d.ptr]);
  const int64_t end = (b0 + kChunkBytes < d.n) ? b0 + kChunkBytes : d.n;
  for (int64_t q = b0 + nb; q < end; ++q) dst[q] = src[q];
  bulk_wait_read_all();
}

// The chunks the producer did not stage, run from global memory as in
// segment_kernel. With kOutOfLine the kernel calls this out of line, so that
// its staged paths are compiled without the fallbacks (108 registers instead of
// 128). Measured on GB300 (interleaved A/B): the interleaved launches that hold
// copy chunks (the 7B local-rank step and its gathers) gain, 8.467 -> 8.402,
// 8.470 -> 8.410 and 8.448 -> 8.404 ms on three boxes; the interleaved
// all-ranks steps (no copies) lose 0.1-1.6 % (1e9 elements: 5.972 -> 6.066 ms),
// and so do the one-copy launches (the Llama block 1.6 %, four Llama blocks in
// the local-rank mode 0.4 %). So only interleaved launches with copy chunks
// take it.
template <int W>
__device__ __noinline__ void tma_unstaged(const Params& p, const Seg& d, int64_t l) {
  switch (d.kind) {
    case kStep: step_chunk<W, false, false>(p, d, l * kChunkElems); break;
    case kReduce: reduce_chunk<W, false>(p, d, l * kChunkElems); break;
    case kAdam: adam_chunk<false>(p, d, l * kChunkElems); break;
    case kCopy: bytes_chunk<false>(p, d, l * kChunkBytes); break;
    default: bytes_chunk<true>(p, d, l * kChunkBytes); break;
  }
}

// One block per SM (its pipeline fills the shared memory). The interleaved
// instantiation without copy chunks (all-ranks steps of rows spread over 3 GiB
// or more) is compiled for two blocks' registers (96 instead of 128): measured
// on GB300 (interleaved A/B, two boxes), the 1e9 / 5e8 / 4e8-element W = 8
// steps 5.976 -> 5.924, 2.988 -> 2.961 and 2.397 -> 2.373 ms; the other
// instantiations lost 2-5 % under the same bound.
template <int W, bool kInterleave, bool kOutOfLine = false>
__global__ void __launch_bounds__(kTmaThreads, (kInterleave && !kOutOfLine) ? 2 : 1)
    tma_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[TmaCfg<W>::kStages];
  __shared__ __align__(8) uint64_t empty_bar[TmaCfg<W>::kStages];
  __shared__ int abort_store;
  volatile int* abort_flag = &abort_store;
  // programmatic dependent launch, as in segment_kernel
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < TmaCfg<W>::kStages; ++s) {
      mbar_init(sm_addr(&full_bar[s]), 1);
      mbar_init(sm_addr(&empty_bar[s]), kTmaConsumerWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  constexpr int kStage = TmaCfg<W>::kStageBytes;
  const int64_t G = gridDim.x;
  const uint64_t limit = p.wait_limit_ns;
  if (warp == kTmaConsumerWarps) {  // producer
    if (lane != 0) return;
    int pending[TmaCfg<W>::kStages];  // parity of the last issued phase of each stage, -1 if none
    for (int s = 0; s < TmaCfg<W>::kStages; ++s) pending[s] = -1;
    Cursor cur;
    uint32_t i = 0;
    for (int64_t c = blockIdx.x; c < p.total_chunks; c += G, ++i) {
      const int stage = static_cast<int>(i % TmaCfg<W>::kStages);
      const uint32_t round = i / TmaCfg<W>::kStages;
      if (!wait_phase(sm_addr(&empty_bar[stage]), (round & 1u) ^ 1u, abort_flag, limit)) break;
      int64_t l, staged;
      const Seg& d = cur.at(p, c, l);
      const uint32_t extra = (blockIdx.x == 0 && i == 0) ? static_cast<uint32_t>(p.inject_tx) : 0u;
      const uint32_t bytes =
          tma_chunk<W, kInterleave>(p, d, l, smem + stage * kStage, sm_addr(&full_bar[stage]), true, extra, &staged);
      if (bytes == 0) mbar_arrive(sm_addr(&full_bar[stage]));
      pending[stage] = static_cast<int>(round & 1u);
    }
    {  // every issued bulk copy lands before the block can exit (bounded)
      for (int s = 0; s < TmaCfg<W>::kStages; ++s) {
        if (pending[s] < 0) continue;
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(sm_addr(&full_bar[s]), static_cast<uint32_t>(pending[s])) &&
               global_ns() - t0 <= limit) {
        }
      }
    }
    return;
  }
  Cursor cur;  // consumers
  uint32_t i = 0;
  for (int64_t c = blockIdx.x; c < p.total_chunks; c += G, ++i) {
    const int stage = static_cast<int>(i % TmaCfg<W>::kStages);
    const uint32_t round = i / TmaCfg<W>::kStages;
    if (!wait_phase(sm_addr(&full_bar[stage]), round & 1u, abort_flag, limit)) break;
    int64_t l, staged;
    const Seg& d = cur.at(p, c, l);
    const unsigned char* st = smem + stage * kStage;
    const uint32_t bytes = tma_chunk<W, kInterleave>(p, d, l, const_cast<unsigned char*>(st), 0, false, 0u, &staged);
    if (bytes != 0 && d.kind == kStep) {
      tma_consume_step<W>(p, d, l, st, staged);
    } else if (bytes != 0) {
      tma_store_copy(p, d, l, st, staged);
    } else if constexpr (kOutOfLine) {
      tma_unstaged<W>(p, d, l);
    } else {
      switch (d.kind) {
        case kStep: step_chunk<W, false, false>(p, d, l * kChunkElems); break;
        case kReduce: reduce_chunk<W, false>(p, d, l * kChunkElems); break;
        case kAdam: adam_chunk<false>(p, d, l * kChunkElems); break;
        case kCopy: bytes_chunk<false>(p, d, l * kChunkBytes); break;
        default: bytes_chunk<true>(p, d, l * kChunkBytes); break;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sm_addr(&empty_bar[stage]));
  }
  if (threadIdx.x == 0) bulk_wait_all();  // every bulk store written before the block exits
}

}  // namespace fsdp
