// Device code of the FSDP FlatParameter step for sm_103a.
//
// Every GPU entry point of the C ABI becomes a list of *segments* run by one
// persistent, grid-strided kernel:
//   kStep    reduce-scatter + Adam + bf16 cast for one shard position, with the
//            reduced gradient applied to every replica that owns the position
//            (the fused step; page "transformer math: FSDP", "The backward
//            cycle: all-gather, grads, reduce-scatter")
//   kReduce  reduce-scatter only (fp32 gradient shard out)
//   kAdam    Adam + bf16 cast only
//   kCopy    byte copy (all-gather of bf16 shards, pack, unpack; "The forward
//            cycle: all-gather, compute, reshard")
//   kZero    zero fill (FlatParameter padding)
// A segment is cut into fixed-size chunks (2048 elements, or 16 KB for
// copies); chunk c of the whole launch is processed by block c mod gridDim, so
// all resident blocks stream through the same region of HBM together. The
// grid is persistent: kBlocksPerSm blocks on every SM. The path is HBM-bound
// (no dense contraction, ~10 fp32 operations per 42+ bytes), so the design
// goals are 16-byte coalesced accesses, many independent loads in flight per
// thread, and streaming cache hints; no tensor cores.
//
// Arithmetic is bit-identical to the definition: fp32 left fold of the W bf16
// gradients in rank order starting from +0, IEEE division by W (a multiply by
// the exact reciprocal when W is a power of two, which rounds identically),
// Adam with one rounding per operation (__f*_rn intrinsics: no contraction
// into FMA), round-to-nearest-even bf16 cast.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fsdp {

constexpr int kThreads = 256;
constexpr int kVec = 8;                                 // elements per thread per chunk
constexpr int64_t kChunkElems = int64_t(kThreads) * kVec;  // 2048 elements
constexpr int64_t kHalf = kChunkElems / 2;

// Which 8 elements of a step / reduce / Adam chunk thread t takes, as two
// groups of 4 (the arithmetic per element is the same either way):
//   kSplit = false: 8t .. 8t+7. Each gradient row is one 16-byte load, but a
//     warp's 16-byte fp32 access spans 1 KB at a 32-byte stride (32 half-used
//     sectors per instruction, each sector requested twice).
//   kSplit = true: 4t .. 4t+3 and kHalf + 4t .. kHalf + 4t+3. A warp's fp32
//     access covers 512 contiguous bytes (16 whole sectors), at the price of
//     two 8-byte loads per gradient row.
// Measured on GB300 (interleaved A/B, LDG form, fraction of the copy peak):
// the split mapping gains where fp32 state dominates the traffic (1e9 elements
// at W = 1 / 2: 0.952 -> 0.985 / 0.984; 16 replicas at W = 16: 0.944 -> 0.980;
// Adam alone: 0.879 -> 0.935) and loses where the gradient rows do (W = 4:
// 0.993 -> 0.983, W = 16 with one replica: 0.989 -> 0.963), so the host picks
// it per launch.
// The consecutive mapping's code paths (partial chunks included) are kept in the
// form they had before the split mapping existed: the TMA form inlines them, and
// a rewrite of just its unstaged fallbacks made the Llama block's step 0.7-0.9 %
// slower on GB300 (interleaved A/B, against 0.1-0.2 % between identical builds).
template <bool kSplit>
struct Map {
  static constexpr int64_t kStride = kSplit ? 4 : 8;      // thread t's first element: kStride * t
  static constexpr int64_t kSecond = kSplit ? kHalf : 4;  // its second group, relative to the first
};
constexpr int kCopyVecs = 4;                              // 16-byte vectors per thread per copy chunk
constexpr int64_t kChunkBytes = int64_t(kThreads) * 16 * kCopyVecs;  // 16 KB (copy / zero)
// Resident blocks per SM. Measured on GB300: 3 blocks of 256 threads stream
// closer to the HBM peak than 4 (W = 2..8: +3..9 %), and replica-heavy hybrid
// steps at W = 16 gain from 3 over the 2 their register use would allow.
constexpr int kBlocksPerSm = 3;

enum SegKind : int32_t { kStep = 0, kReduce = 1, kAdam = 2, kCopy = 3, kZero = 4 };

// Width code of a step, reduce or Adam segment with some pointer off 16-byte
// alignment but every pointer aligned to its element (2 bytes for bf16, 4 for
// fp32): its chunks take the realigned vector path.
constexpr int32_t kPhased = 32;

// One segment. Pointer pool layout (Params::ptr, starting at `ptr`):
//   kStep   : W gradient rows (bf16, already offset to the position),
//             then nrep x {master, exp_avg, exp_avg_sq, bf16 out}
//   kReduce : W gradient rows, fp32 out
//   kAdam   : fp32 grad, master, exp_avg, exp_avg_sq, bf16 out (may be null)
//   kCopy   : src, dst          (n in bytes)
//   kZero   : dst               (n in bytes)
struct Seg {
  int64_t n;          // elements (kStep/kReduce/kAdam) or bytes (kCopy/kZero)
  int64_t chunk_end;  // running total of chunks up to and including this segment
  int32_t kind;
  int32_t nrep;       // kStep: replicas updated from the reduced gradient
  int32_t ptr;        // first pool entry
  int32_t width;      // kStep/kReduce/kAdam: 16 if every pointer is 16-byte aligned, else 0;
                      // kStep / kReduce / kAdam also kPhased (see there);
                      // kCopy/kZero: access width in bytes (16, 8, 4, 2 or 1)
};

// Per-launch fp32 scalars (formed on the host in double, rounded once).
struct Scalars {
  float lr, b1, b2, eps;
  float omb1, omb2;   // 1 - b1, 1 - b2
  float bc1, bc2;     // 1 - b1^t, 1 - b2^t
  float inv_w;        // 1 / W if W is a power of two (exact), else 0
  int32_t w;          // W
};

constexpr int kMaxSeg = 320;
constexpr int kMaxPtr = 2048;

// Passed by value as a __grid_constant__ kernel parameter (~26.7 KB, within the
// 32,764-byte limit): the whole descriptor table arrives with the launch, no
// device allocation or copy is needed.
struct Params {
  Scalars s;
  int32_t nseg;
  int32_t inject_tx;       // self-test only: extra bytes expected on block 0's first staged chunk
  int64_t total_chunks;
  uint64_t wait_limit_ns;  // bound of every mbarrier wait in the TMA form
  Seg seg[kMaxSeg];
  const void* ptr[kMaxPtr];
};
static_assert(sizeof(Params) <= 32764, "kernel parameter block too large");

// ------------------------------------------------------------ memory access

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ void st_stream_u2(void* p, uint2 v) {
  __stcs(reinterpret_cast<uint2*>(p), v);
}
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_stream_f4(float* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}
__device__ __forceinline__ void st_stream_u4(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}
// 8 consecutive fp32 (one 32-byte sector) in one streaming store; p must be
// 32-byte aligned.
__device__ __forceinline__ void st_stream_f8(float* p, const float (&x)[8]) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(x[0]), "f"(x[1]), "f"(x[2]),
               "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7])
               : "memory");
}

// ------------------------------------------------------------- arithmetic

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint16_t bf16_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Mean over W of the folded sum.
template <int W>
__device__ __forceinline__ float mean_of(float acc, const Scalars& s) {
  if constexpr (W > 0 && (W & (W - 1)) == 0) {
    return __fmul_rn(acc, 1.0f / W);  // exact reciprocal: same rounding as acc / W
  } else {
    return s.inv_w != 0.0f ? __fmul_rn(acc, s.inv_w) : __fdiv_rn(acc, static_cast<float>(s.w));
  }
}

// Adam (Kingma & Ba 2015, Algorithm 1, weight decay 0) on one element.
__device__ __forceinline__ void adam1(float g, float& p, float& m, float& v, const Scalars& s) {
  m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  const float m_hat = __fdiv_rn(m, s.bc1);
  const float v_hat = __fdiv_rn(v, s.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), s.eps);
  p = __fsub_rn(p, __fmul_rn(s.lr, __fdiv_rn(m_hat, denom)));
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& r) {
  acc[0] = __fadd_rn(acc[0], bf16_lo(r.x));
  acc[1] = __fadd_rn(acc[1], bf16_hi(r.x));
  acc[2] = __fadd_rn(acc[2], bf16_lo(r.y));
  acc[3] = __fadd_rn(acc[3], bf16_hi(r.y));
  acc[4] = __fadd_rn(acc[4], bf16_lo(r.z));
  acc[5] = __fadd_rn(acc[5], bf16_hi(r.z));
  acc[6] = __fadd_rn(acc[6], bf16_lo(r.w));
  acc[7] = __fadd_rn(acc[7], bf16_hi(r.w));
}

// acc[o .. o+3] += the 4 bf16 values of r (element order: r.x low, r.x high, r.y low, r.y high).
__device__ __forceinline__ void add_bf16x4(float (&acc)[8], int o, const uint2& r) {
  acc[o + 0] = __fadd_rn(acc[o + 0], bf16_lo(r.x));
  acc[o + 1] = __fadd_rn(acc[o + 1], bf16_hi(r.x));
  acc[o + 2] = __fadd_rn(acc[o + 2], bf16_lo(r.y));
  acc[o + 3] = __fadd_rn(acc[o + 3], bf16_hi(r.y));
}

// One gradient row's contribution to a thread's 8 elements (Map<kSplit>).
template <bool kSplit>
struct RowLoad {
  uint4 a;  // kSplit = false: the 8 consecutive elements
};
template <>
struct RowLoad<true> {
  uint2 a, b;  // the two groups of 4
};

template <bool kSplit>
__device__ __forceinline__ RowLoad<kSplit> load_row(const uint16_t* row, int64_t e) {
  RowLoad<kSplit> r;
  if constexpr (kSplit) {
    r.a = ld_stream_u2(row + e);
    r.b = ld_stream_u2(row + e + kHalf);
  } else {
    r.a = ld_stream_u4(row + e);
  }
  return r;
}

template <bool kSplit>
__device__ __forceinline__ void add_row(float (&acc)[8], const RowLoad<kSplit>& r) {
  if constexpr (kSplit) {
    add_bf16x4(acc, 0, r.a);
    add_bf16x4(acc, 4, r.b);
  } else {
    add_bf16x8(acc, r.a);
  }
}

// A request that the line holding x be brought into L2; it returns no data
// and holds no register.
__device__ __forceinline__ void prefetch_l2(const void* x) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(x));
}

// The lines of the thread's 8 elements (from e) in its block's next chunk of
// the same segment, for every gradient row and the first replica's three state
// arrays: requested into L2 now, read one round of the grid later (the block's
// next chunk is gridDim.x chunks on). Only elements inside the segment.
template <int W>
__device__ __forceinline__ void prefetch_next_step(const Params& p, const Seg& d, int64_t e) {
  const int64_t en = e + int64_t(gridDim.x) * kChunkElems;
  if (en + kVec > d.n) return;
  const int w = W > 0 ? W : p.s.w;
  for (int k = 0; k < w; ++k) prefetch_l2(static_cast<const uint16_t*>(p.ptr[d.ptr + k]) + en);
  for (int a = 0; a < 3; ++a) prefetch_l2(static_cast<const float*>(p.ptr[d.ptr + w + a]) + en);
}

// The 16 bytes that start `phase` bytes (0..15) into the aligned block lo, hi
// being the aligned block after it: a shift by whole words (phase / 4, by
// selects on its two bits: the phase is the same for every thread of a row or
// array) and then by whole bytes.
__device__ __forceinline__ uint4 shift_bytes(const uint4& lo, const uint4& hi, int phase) {
  uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const bool by2 = (phase & 8) != 0, by1 = (phase & 4) != 0;
#pragma unroll
  for (int i = 0; i < 6; ++i) w[i] = by2 ? w[i + 2] : w[i];
#pragma unroll
  for (int i = 0; i < 5; ++i) w[i] = by1 ? w[i + 1] : w[i];
  const uint32_t h = static_cast<uint32_t>(phase & 3) * 8u;
  return make_uint4(__funnelshift_r(w[0], w[1], h), __funnelshift_r(w[1], w[2], h), __funnelshift_r(w[2], w[3], h),
                    __funnelshift_r(w[3], w[4], h));
}

// The aligned 16-byte block that holds the first of the 16 bytes at x, and the
// block after it (the same block again when x is aligned), for shift_bytes:
// every block read holds one of the bytes used, so the reads stay within their
// pages. Branch-free, so that a caller's loads of several rows are all in
// flight before the first shift (measured on GB300: a branch on the phase, or
// the second load predicated on it, kept fewer loads in flight and ran 4-20 %
// slower).
__device__ __forceinline__ void load_blocks(const void* x, uint4& lo, uint4& hi, int& phase) {
  phase = static_cast<int>(reinterpret_cast<uintptr_t>(x) & 15u);
  const unsigned char* al = static_cast<const unsigned char*>(x) - phase;
  lo = ld_stream_u4(al);
  hi = ld_stream_u4(al + (phase != 0 ? 16 : 0));
}

// fold8 (consecutive mapping) for rows at any even byte phase: each row's
// phase is read from its pointer (the same for every thread: e is a multiple of
// 8 elements, 16 bytes); the thread's 8 elements start at e.
template <int W>
__device__ __forceinline__ void fold8_realigned(const Params& p, const Seg& d, int64_t e, float (&g)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) g[i] = 0.0f;
  const int w = W > 0 ? W : p.s.w;
  // rows loaded before they are shifted and added (8 at W >= 8; 4 for a
  // runtime W, whose instantiation would spill more with 8)
  constexpr int kBatch = W == 0 ? 4 : (W < 8 ? W : 8);
  for (int k0 = 0; k0 < w; k0 += kBatch) {
    uint4 lo[kBatch], hi[kBatch];
    int ph[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (W > 0 || k0 + k < w) load_blocks(static_cast<const uint16_t*>(p.ptr[d.ptr + k0 + k]) + e, lo[k], hi[k], ph[k]);
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (W > 0 || k0 + k < w) add_bf16x8(g, shift_bytes(lo[k], hi[k], ph[k]));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) g[i] = mean_of<W>(g[i], p.s);
}

// Reduced gradient of a thread's 8 elements (first group at e): the rows of a
// batch (up to 8) are all loaded first (independent loads in flight), then
// folded in rank order.
template <int W, bool kSplit>
__device__ __forceinline__ void fold8(const Params& p, const Seg& d, int64_t e, float (&g)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) g[i] = 0.0f;
  if constexpr (W > 0) {
    // rows in batches of at most 8 (rank order kept) to bound register use
    constexpr int kBatch = W < 8 ? W : 8;
#pragma unroll
    for (int k0 = 0; k0 < W; k0 += kBatch) {
      RowLoad<kSplit> r[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        r[k] = load_row<kSplit>(static_cast<const uint16_t*>(p.ptr[d.ptr + k0 + k]), e);
#pragma unroll
      for (int k = 0; k < kBatch; ++k) add_row<kSplit>(g, r[k]);
    }
  } else {
    const int w = p.s.w;
    for (int k0 = 0; k0 < w; k0 += 8) {
      RowLoad<kSplit> r[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k0 + k < w) r[k] = load_row<kSplit>(static_cast<const uint16_t*>(p.ptr[d.ptr + k0 + k]), e);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k0 + k < w) add_row<kSplit>(g, r[k]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) g[i] = mean_of<W>(g[i], p.s);
}

template <int W>
__device__ __forceinline__ float fold1(const Params& p, const Seg& d, int64_t i) {
  float acc = 0.0f;
  const int w = W > 0 ? W : p.s.w;
  for (int k = 0; k < w; ++k)
    acc = __fadd_rn(acc, bf16_to_f32(static_cast<const uint16_t*>(p.ptr[d.ptr + k])[i]));
  return mean_of<W>(acc, p.s);
}

// A thread's state: [0..3] at elements e .. e+3, [4..7] at the second group.
struct State8 {
  float p[8], m[8], v[8];
};

template <bool kSplit>
__device__ __forceinline__ void load_state8(State8& st, const float* mp, const float* mm,
                                            const float* mv, int64_t e) {
  constexpr int64_t o = Map<kSplit>::kSecond;
  const float4 p0 = ld_stream_f4(mp + e), p1 = ld_stream_f4(mp + e + o);
  const float4 m0 = ld_stream_f4(mm + e), m1 = ld_stream_f4(mm + e + o);
  const float4 v0 = ld_stream_f4(mv + e), v1 = ld_stream_f4(mv + e + o);
  st.p[0] = p0.x; st.p[1] = p0.y; st.p[2] = p0.z; st.p[3] = p0.w;
  st.p[4] = p1.x; st.p[5] = p1.y; st.p[6] = p1.z; st.p[7] = p1.w;
  st.m[0] = m0.x; st.m[1] = m0.y; st.m[2] = m0.z; st.m[3] = m0.w;
  st.m[4] = m1.x; st.m[5] = m1.y; st.m[6] = m1.z; st.m[7] = m1.w;
  st.v[0] = v0.x; st.v[1] = v0.y; st.v[2] = v0.z; st.v[3] = v0.w;
  st.v[4] = v1.x; st.v[5] = v1.y; st.v[6] = v1.z; st.v[7] = v1.w;
}

template <bool kSplit>
__device__ __forceinline__ void store_state8(const State8& st, float* mp, float* mm, float* mv,
                                             uint16_t* out, int64_t e) {
  constexpr int64_t o = Map<kSplit>::kSecond;
  st_stream_f4(mp + e, make_float4(st.p[0], st.p[1], st.p[2], st.p[3]));
  st_stream_f4(mp + e + o, make_float4(st.p[4], st.p[5], st.p[6], st.p[7]));
  st_stream_f4(mm + e, make_float4(st.m[0], st.m[1], st.m[2], st.m[3]));
  st_stream_f4(mm + e + o, make_float4(st.m[4], st.m[5], st.m[6], st.m[7]));
  st_stream_f4(mv + e, make_float4(st.v[0], st.v[1], st.v[2], st.v[3]));
  st_stream_f4(mv + e + o, make_float4(st.v[4], st.v[5], st.v[6], st.v[7]));
  if (out) {
    if constexpr (kSplit) {
      st_stream_u2(out + e, make_uint2(bf16x2_rn(st.p[0], st.p[1]), bf16x2_rn(st.p[2], st.p[3])));
      st_stream_u2(out + e + o, make_uint2(bf16x2_rn(st.p[4], st.p[5]), bf16x2_rn(st.p[6], st.p[7])));
    } else {
      uint4 v;
      v.x = bf16x2_rn(st.p[0], st.p[1]);
      v.y = bf16x2_rn(st.p[2], st.p[3]);
      v.z = bf16x2_rn(st.p[4], st.p[5]);
      v.w = bf16x2_rn(st.p[6], st.p[7]);
      st_stream_u4(out + e, v);
    }
  }
}

// First element of thread t's first group in a chunk starting at e0.
template <bool kSplit>
__device__ __forceinline__ int64_t group_start(int64_t e0) {
  return e0 + int64_t(threadIdx.x) * Map<kSplit>::kStride;
}

// Both of the thread's groups lie inside the segment: the vector path applies.
template <bool kSplit>
__device__ __forceinline__ bool groups_inside(int64_t e, int64_t n) {
  return e + Map<kSplit>::kSecond + 4 <= n;
}

// ------------------------------------------------------------- segment work

template <int W>
__device__ __forceinline__ void step_scalar(const Params& p, const Seg& d, int64_t i) {
  const float g = fold1<W>(p, d, i);
  const int w = W > 0 ? W : p.s.w;
  for (int r = 0; r < d.nrep; ++r) {
    const int b = d.ptr + w + 4 * r;
    float* mp = static_cast<float*>(const_cast<void*>(p.ptr[b]));
    float* mm = static_cast<float*>(const_cast<void*>(p.ptr[b + 1]));
    float* mv = static_cast<float*>(const_cast<void*>(p.ptr[b + 2]));
    uint16_t* out = static_cast<uint16_t*>(const_cast<void*>(p.ptr[b + 3]));
    float pv = mp[i], mvv = mm[i], vv = mv[i];
    adam1(g, pv, mvv, vv, p.s);
    mp[i] = pv;
    mm[i] = mvv;
    mv[i] = vv;
    out[i] = bf16_rn(pv);
  }
}

// The state of a thread's 8 elements from arrays at any 4-byte phase (each
// array's own, read from its pointer).
// Three aligned blocks from the one holding q[0] (at phase 0 the third is the
// second again: every block read holds one of the 32 bytes used), shifted by
// whole words; branch-free like load_blocks.
__device__ __forceinline__ void load_f32x8_any(const float* q, float (&x)[8]) {
  const int phase = static_cast<int>(reinterpret_cast<uintptr_t>(q) & 15u);
  const float* al = q - phase / 4;
  const float4 a = ld_stream_f4(al), b = ld_stream_f4(al + 4), c = ld_stream_f4(al + (phase != 0 ? 8 : 4));
  float w[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
  const bool by2 = (phase & 8) != 0, by1 = (phase & 4) != 0;
#pragma unroll
  for (int i = 0; i < 10; ++i) w[i] = by2 ? w[i + 2] : w[i];
#pragma unroll
  for (int i = 0; i < 9; ++i) w[i] = by1 ? w[i + 1] : w[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = w[i];
}

// A warp's 256 results of one array, thread `lane` holding elements 8 lane ..
// 8 lane + 7, stored through the warp's staging row `buf` so that every store
// instruction writes 32 consecutive elements (q: the warp's first element).
__device__ __forceinline__ void store_f32_transposed(float* buf, float* q, const float (&x)[8], int lane) {
  reinterpret_cast<float4*>(buf)[2 * lane] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(buf)[2 * lane + 1] = make_float4(x[4], x[5], x[6], x[7]);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j) __stcs(q + 32 * j + lane, buf[32 * j + lane]);
  __syncwarp();
}
__device__ __forceinline__ void store_bf16_transposed(float* buf, uint16_t* q, const float (&x)[8], int lane) {
  reinterpret_cast<uint4*>(buf)[lane] = make_uint4(bf16x2_rn(x[0], x[1]), bf16x2_rn(x[2], x[3]),
                                                   bf16x2_rn(x[4], x[5]), bf16x2_rn(x[6], x[7]));
  __syncwarp();
  const unsigned short* b16 = reinterpret_cast<const unsigned short*>(buf);
#pragma unroll
  for (int j = 0; j < 8; ++j) __stcs(reinterpret_cast<unsigned short*>(q) + 32 * j + lane, b16[32 * j + lane]);
  __syncwarp();
}

// A step chunk of a kPhased segment (consecutive mapping). Each warp covers 256
// consecutive elements: rows read as aligned 16-byte blocks shifted into place,
// state read as aligned blocks shifted by whole words (every pointer at its own
// phase), results stored through a per-warp staging row in shared memory so
// that each store instruction writes 32 consecutive elements. A warp whose 256
// elements pass the segment's end takes one element per lane. Same arithmetic
// in the same order as the aligned path. Out of line, so that the aligned path
// keeps its registers.
// The warp's staging row (256 floats) of the realigned paths, one per warp.
__device__ __forceinline__ float* realign_stage(int warp) {
  __shared__ __align__(16) float stage[kThreads / 32][32 * kVec];
  return stage[warp];
}

template <int W>
__device__ __noinline__ void step_chunk_realigned(const Params& p, const Seg& d, int64_t e0) {
  const int w = W > 0 ? W : p.s.w;
  const int warp = static_cast<int>(threadIdx.x / 32), lane = static_cast<int>(threadIdx.x % 32);
  const int64_t ew = e0 + int64_t(warp) * 32 * kVec;  // the warp's first element
  if (ew >= d.n) return;
  if (ew + 32 * kVec > d.n) {
    for (int64_t i = ew + lane; i < d.n; i += 32) step_scalar<W>(p, d, i);
    return;
  }
  const int64_t e = ew + int64_t(lane) * kVec;
  // at W = 2 and 4 the next chunk's lines are requested into L2 first.
  // Measured on GB300 (interleaved A/B, odd S, about 1e8 elements, all ranks):
  // W = 2 0.620 -> 0.713 of the copy peak, W = 4 0.637 -> 0.652; W = 8 and 16
  // lost 2-9 % with it (their loads already fill the memory pipeline), and so
  // did every aligned LDG step (7-15 %).
  if constexpr (W == 2 || W == 4) prefetch_next_step<W>(p, d, e);
  const int b0 = d.ptr + w;
  State8 st;
  load_f32x8_any(static_cast<const float*>(p.ptr[b0]) + e, st.p);
  load_f32x8_any(static_cast<const float*>(p.ptr[b0 + 1]) + e, st.m);
  load_f32x8_any(static_cast<const float*>(p.ptr[b0 + 2]) + e, st.v);
  float g[8];
  fold8_realigned<W>(p, d, e, g);
  float* buf = realign_stage(warp);
  for (int r = 0; r < d.nrep; ++r) {
    const int b = b0 + 4 * r;
    float* mp = static_cast<float*>(const_cast<void*>(p.ptr[b]));
    float* mm = static_cast<float*>(const_cast<void*>(p.ptr[b + 1]));
    float* mv = static_cast<float*>(const_cast<void*>(p.ptr[b + 2]));
    uint16_t* out = static_cast<uint16_t*>(const_cast<void*>(p.ptr[b + 3]));
    if (r > 0) {
      load_f32x8_any(mp + e, st.p);
      load_f32x8_any(mm + e, st.m);
      load_f32x8_any(mv + e, st.v);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) adam1(g[i], st.p[i], st.m[i], st.v[i], p.s);
    store_f32_transposed(buf, mp + ew, st.p, lane);
    store_f32_transposed(buf, mm + ew, st.m, lane);
    store_f32_transposed(buf, mv + ew, st.v, lane);
    store_bf16_transposed(buf, out + ew, st.p, lane);
  }
}

// kRealign: kPhased segments take the realigned path, else the scalar one. Only
// the kernel instantiations for launches that hold kPhased segments include it:
// reachable, its code and its shared-memory staging rows slowed the aligned
// path by 2-5 % (registers, spills, shared memory).
template <int W, bool kSplit, bool kRealign = false>
__device__ __forceinline__ void step_chunk(const Params& p, const Seg& d, int64_t e0) {
  const int w = W > 0 ? W : p.s.w;
  if (d.width == 16) {
    const int64_t e = group_start<kSplit>(e0);
    if (groups_inside<kSplit>(e, d.n)) {
      const int b0 = d.ptr + w;
      State8 st;
      // state of the first replica is requested before the gradient fold
      load_state8<kSplit>(st, static_cast<const float*>(p.ptr[b0]), static_cast<const float*>(p.ptr[b0 + 1]),
                          static_cast<const float*>(p.ptr[b0 + 2]), e);
      float g[8];
      fold8<W, kSplit>(p, d, e, g);
      for (int r = 0; r < d.nrep; ++r) {
        const int b = b0 + 4 * r;
        float* mp = static_cast<float*>(const_cast<void*>(p.ptr[b]));
        float* mm = static_cast<float*>(const_cast<void*>(p.ptr[b + 1]));
        float* mv = static_cast<float*>(const_cast<void*>(p.ptr[b + 2]));
        uint16_t* out = static_cast<uint16_t*>(const_cast<void*>(p.ptr[b + 3]));
        if (r > 0) load_state8<kSplit>(st, mp, mm, mv, e);
#pragma unroll
        for (int i = 0; i < 8; ++i) adam1(g[i], st.p[i], st.m[i], st.v[i], p.s);
        store_state8<kSplit>(st, mp, mm, mv, out, e);
      }
    } else {  // the segment's last, partial chunk
      if constexpr (kSplit) {
        constexpr int64_t o = Map<kSplit>::kSecond;
        for (int h = 0; h < 2; ++h)
          for (int64_t i = e + h * o; i < e + h * o + 4 && i < d.n; ++i) step_scalar<W>(p, d, i);
      } else {
        for (int64_t i = e; i < d.n; ++i) step_scalar<W>(p, d, i);
      }
    }
  } else {
    if constexpr (!kSplit && kRealign) {
      if (d.width == kPhased) {  // pointers off 16-byte alignment, each at its own phase
        step_chunk_realigned<W>(p, d, e0);
        return;
      }
    }
#pragma unroll 1
    for (int k = 0; k < kVec; ++k) {
      const int64_t i = e0 + int64_t(k) * kThreads + threadIdx.x;
      if (i < d.n) step_scalar<W>(p, d, i);
    }
  }
}

// A reduce chunk of a kPhased segment: rows realigned as in
// step_chunk_realigned, the fp32 results stored through the warp's staging row.
template <int W>
__device__ __noinline__ void reduce_chunk_realigned(const Params& p, const Seg& d, int64_t e0) {
  const int w = W > 0 ? W : p.s.w;
  float* out = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + w]));
  const int warp = static_cast<int>(threadIdx.x / 32), lane = static_cast<int>(threadIdx.x % 32);
  const int64_t ew = e0 + int64_t(warp) * 32 * kVec;
  if (ew >= d.n) return;
  if (ew + 32 * kVec > d.n) {
    for (int64_t i = ew + lane; i < d.n; i += 32) out[i] = fold1<W>(p, d, i);
    return;
  }
  float g[8];
  fold8_realigned<W>(p, d, ew + int64_t(lane) * kVec, g);
  store_f32_transposed(realign_stage(warp), out + ew, g, lane);
}

template <int W, bool kSplit, bool kRealign = false>
__device__ __forceinline__ void reduce_chunk(const Params& p, const Seg& d, int64_t e0) {
  const int w = W > 0 ? W : p.s.w;
  float* out = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + w]));
  if constexpr (!kSplit && kRealign) {
    if (d.width == kPhased) {
      reduce_chunk_realigned<W>(p, d, e0);
      return;
    }
  }
  if (d.width == 16) {
    constexpr int64_t o = Map<kSplit>::kSecond;
    const int64_t e = group_start<kSplit>(e0);
    if (groups_inside<kSplit>(e, d.n)) {
      float g[8];
      fold8<W, kSplit>(p, d, e, g);
      st_stream_f4(out + e, make_float4(g[0], g[1], g[2], g[3]));
      st_stream_f4(out + e + o, make_float4(g[4], g[5], g[6], g[7]));
    } else {  // the segment's last, partial chunk
      if constexpr (kSplit) {
        for (int h = 0; h < 2; ++h)
          for (int64_t i = e + h * o; i < e + h * o + 4 && i < d.n; ++i) out[i] = fold1<W>(p, d, i);
      } else {
        for (int64_t i = e; i < d.n; ++i) out[i] = fold1<W>(p, d, i);
      }
    }
  } else {
#pragma unroll 1
    for (int k = 0; k < kVec; ++k) {
      const int64_t i = e0 + int64_t(k) * kThreads + threadIdx.x;
      if (i < d.n) out[i] = fold1<W>(p, d, i);
    }
  }
}

// An Adam chunk of a kPhased segment: gradient and state read as realigned
// blocks, results stored through the warp's staging row.
static __device__ __noinline__ void adam_chunk_realigned(const Params& p, const Seg& d, int64_t e0) {
  const float* gp = static_cast<const float*>(p.ptr[d.ptr]);
  float* mp = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + 1]));
  float* mm = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + 2]));
  float* mv = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + 3]));
  uint16_t* out = static_cast<uint16_t*>(const_cast<void*>(p.ptr[d.ptr + 4]));
  const int warp = static_cast<int>(threadIdx.x / 32), lane = static_cast<int>(threadIdx.x % 32);
  const int64_t ew = e0 + int64_t(warp) * 32 * kVec;
  if (ew >= d.n) return;
  if (ew + 32 * kVec > d.n) {
    for (int64_t i = ew + lane; i < d.n; i += 32) {
      float pv = mp[i], mvv = mm[i], vv = mv[i];
      adam1(gp[i], pv, mvv, vv, p.s);
      mp[i] = pv;
      mm[i] = mvv;
      mv[i] = vv;
      if (out) out[i] = bf16_rn(pv);
    }
    return;
  }
  const int64_t e = ew + int64_t(lane) * kVec;
  // the next chunk's lines requested into L2 first, as the realigned step does
  // at W = 2 and 4 (measured on GB300, 8 odd-S shards of 12.6 M elements: 0.779
  // -> 0.796 of the copy peak; the realigned copies lost 3 % with it)
  const int64_t en = e + int64_t(gridDim.x) * kChunkElems;
  if (en + kVec <= d.n) {
    prefetch_l2(gp + en);
    prefetch_l2(mp + en);
    prefetch_l2(mm + en);
    prefetch_l2(mv + en);
  }
  float g[8];
  State8 st;
  load_f32x8_any(gp + e, g);
  load_f32x8_any(mp + e, st.p);
  load_f32x8_any(mm + e, st.m);
  load_f32x8_any(mv + e, st.v);
#pragma unroll
  for (int i = 0; i < 8; ++i) adam1(g[i], st.p[i], st.m[i], st.v[i], p.s);
  float* buf = realign_stage(warp);
  store_f32_transposed(buf, mp + ew, st.p, lane);
  store_f32_transposed(buf, mm + ew, st.m, lane);
  store_f32_transposed(buf, mv + ew, st.v, lane);
  if (out) store_bf16_transposed(buf, out + ew, st.p, lane);
}

template <bool kSplit, bool kRealign = false>
__device__ __forceinline__ void adam_chunk(const Params& p, const Seg& d, int64_t e0) {
  if constexpr (!kSplit && kRealign) {
    if (d.width == kPhased) {
      adam_chunk_realigned(p, d, e0);
      return;
    }
  }
  const float* gp = static_cast<const float*>(p.ptr[d.ptr]);
  float* mp = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + 1]));
  float* mm = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + 2]));
  float* mv = static_cast<float*>(const_cast<void*>(p.ptr[d.ptr + 3]));
  uint16_t* out = static_cast<uint16_t*>(const_cast<void*>(p.ptr[d.ptr + 4]));
  if (d.width == 16) {
    const int64_t e = group_start<kSplit>(e0);
    if (groups_inside<kSplit>(e, d.n)) {
      State8 st;
      load_state8<kSplit>(st, mp, mm, mv, e);
      const float4 g0 = ld_stream_f4(gp + e), g1 = ld_stream_f4(gp + e + Map<kSplit>::kSecond);
      const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) adam1(g[i], st.p[i], st.m[i], st.v[i], p.s);
      store_state8<kSplit>(st, mp, mm, mv, out, e);
      return;
    }
  }
  // misaligned segments, and the last, partial chunk of an aligned one
  const bool vec = d.width == 16;
  const int64_t lo = vec ? group_start<kSplit>(e0) : 0;
  for (int k = 0; k < kVec; ++k) {
    const int64_t i = vec ? (kSplit ? lo + (k >> 2) * Map<kSplit>::kSecond + (k & 3) : lo + k)
                          : e0 + int64_t(k) * kThreads + threadIdx.x;
    if (i >= d.n) continue;
    float pv = mp[i], mvv = mm[i], vv = mv[i];
    adam1(gp[i], pv, mvv, vv, p.s);
    mp[i] = pv;
    mm[i] = mvv;
    mv[i] = vv;
    if (out) out[i] = bf16_rn(pv);
  }
}

// A copy (or zero-fill) chunk whose source and destination are not both 16-byte
// aligned: every 16-byte block of the destination that lies inside the chunk is
// written with one aligned store (its source bytes read as two aligned blocks
// and shifted into place), the chunk's first and last bytes around them one
// byte at a time (those blocks are shared with the neighbouring chunks).
template <bool kZeroFill>
__device__ __noinline__ void bytes_chunk_realigned(const Params& p, const Seg& d, int64_t b0) {
  const unsigned char* src = kZeroFill ? nullptr : static_cast<const unsigned char*>(p.ptr[d.ptr]);
  unsigned char* dst = static_cast<unsigned char*>(const_cast<void*>(p.ptr[d.ptr + (kZeroFill ? 0 : 1)]));
  const int64_t end = (b0 + kChunkBytes < d.n) ? b0 + kChunkBytes : d.n;
  const uintptr_t ds = reinterpret_cast<uintptr_t>(dst) + static_cast<uintptr_t>(b0);
  const uintptr_t de = reinterpret_cast<uintptr_t>(dst) + static_cast<uintptr_t>(end);
  const uintptr_t a = (ds + 15) & ~uintptr_t(15), z = de & ~uintptr_t(15);
  if (a >= z) {
    for (int64_t q = b0 + threadIdx.x; q < end; q += kThreads) dst[q] = kZeroFill ? 0 : src[q];
    return;
  }
  const int64_t head = static_cast<int64_t>(a - ds), tail = static_cast<int64_t>(de - z);
  if (int64_t(threadIdx.x) < head) dst[b0 + threadIdx.x] = kZeroFill ? 0 : src[b0 + threadIdx.x];
  if (int64_t(threadIdx.x) < tail) {
    const int64_t q = end - tail + threadIdx.x;
    dst[q] = kZeroFill ? 0 : src[q];
  }
  // at most kThreads * kCopyVecs blocks: all loads first (the source's aligned
  // block holding the first byte and, off its boundary, the block after it;
  // at phase 0 the same block twice), then the shifts and stores
  const int64_t nblk = static_cast<int64_t>(z - a) / 16;
  const int64_t first = b0 + head;  // segment byte offset of the first whole block
  const int py = kZeroFill ? 0 : static_cast<int>((reinterpret_cast<uintptr_t>(src) + first) & 15u);
  const int64_t next = py != 0 ? 16 : 0;
  uint4 lo[kCopyVecs], hi[kCopyVecs];
#pragma unroll
  for (int k = 0; k < kCopyVecs; ++k) {
    const int64_t i = int64_t(k) * kThreads + threadIdx.x;
    lo[k] = hi[k] = make_uint4(0, 0, 0, 0);
    if (!kZeroFill && i < nblk) {
      const unsigned char* al = src + first + 16 * i - py;
      lo[k] = ld_stream_u4(al);
      hi[k] = ld_stream_u4(al + next);
    }
  }
#pragma unroll
  for (int k = 0; k < kCopyVecs; ++k) {
    const int64_t i = int64_t(k) * kThreads + threadIdx.x;
    if (i < nblk) st_stream_u4(dst + first + 16 * i, kZeroFill ? lo[k] : shift_bytes(lo[k], hi[k], py));
  }
}

template <bool kZeroFill, bool kRealign = false>
__device__ __forceinline__ void bytes_chunk(const Params& p, const Seg& d, int64_t b0) {
  if constexpr (kRealign) {
    if (d.width != 16) {
      bytes_chunk_realigned<kZeroFill>(p, d, b0);
      return;
    }
  }
  const unsigned char* src =
      kZeroFill ? nullptr : static_cast<const unsigned char*>(p.ptr[d.ptr]);
  unsigned char* dst = static_cast<unsigned char*>(const_cast<void*>(p.ptr[d.ptr + (kZeroFill ? 0 : 1)]));
  const int64_t end = (b0 + kChunkBytes < d.n) ? b0 + kChunkBytes : d.n;
  switch (d.width) {
    case 16: {
      // all loads of the chunk first (64 bytes in flight per thread), then the stores
      uint4 v[kCopyVecs];
#pragma unroll
      for (int k = 0; k < kCopyVecs; ++k) {
        const int64_t b = b0 + (int64_t(k) * kThreads + threadIdx.x) * 16;
        if (!kZeroFill && b + 16 <= end) v[k] = ld_stream_u4(src + b);
      }
#pragma unroll
      for (int k = 0; k < kCopyVecs; ++k) {
        const int64_t b = b0 + (int64_t(k) * kThreads + threadIdx.x) * 16;
        if (b + 16 <= end) {
          st_stream_u4(dst + b, kZeroFill ? make_uint4(0, 0, 0, 0) : v[k]);
        } else {
          for (int64_t i = b; i < end; ++i) dst[i] = kZeroFill ? 0 : src[i];
        }
      }
      break;
    }
    case 8:
      for (int64_t b = b0 + int64_t(threadIdx.x) * 8; b < end; b += int64_t(kThreads) * 8)
        *reinterpret_cast<uint2*>(dst + b) =
            kZeroFill ? make_uint2(0, 0) : *reinterpret_cast<const uint2*>(src + b);
      break;
    case 4:
      for (int64_t b = b0 + int64_t(threadIdx.x) * 4; b < end; b += int64_t(kThreads) * 4)
        *reinterpret_cast<uint32_t*>(dst + b) =
            kZeroFill ? 0u : *reinterpret_cast<const uint32_t*>(src + b);
      break;
    case 2:
      for (int64_t b = b0 + int64_t(threadIdx.x) * 2; b < end; b += int64_t(kThreads) * 2)
        *reinterpret_cast<uint16_t*>(dst + b) =
            kZeroFill ? uint16_t(0) : *reinterpret_cast<const uint16_t*>(src + b);
      break;
    default:
      for (int64_t b = b0 + threadIdx.x; b < end; b += kThreads) dst[b] = kZeroFill ? 0 : src[b];
      break;
  }
}

// -------------------------------------------------------------- the kernel

// kWithRealign: the instantiation for launches that hold kPhased segments or
// copies off 16-byte alignment (the consecutive mapping, with the realigned
// paths).
template <int W, bool kSplit, bool kWithRealign = false>
__global__ void __launch_bounds__(kThreads, (W > 0 ? kBlocksPerSm : 2))
    segment_kernel(const __grid_constant__ Params p) {
  // Launched with programmatic stream serialization (see abi.cu): this grid
  // may be placed on the SMs while the previous kernel of the stream drains.
  // Wait for that kernel to complete, with its writes visible, before the
  // first memory access; then allow the next launch to be scheduled early.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  int s = 0;
  int64_t first = 0;  // first chunk of segment s
  for (int64_t c = blockIdx.x; c < p.total_chunks; c += gridDim.x) {
    while (c >= p.seg[s].chunk_end) {
      first = p.seg[s].chunk_end;
      ++s;
    }
    const Seg& d = p.seg[s];
    const int64_t local = c - first;
    switch (d.kind) {
      case kStep: step_chunk<W, kSplit, kWithRealign>(p, d, local * kChunkElems); break;
      case kReduce: reduce_chunk<W, kSplit, kWithRealign>(p, d, local * kChunkElems); break;
      case kAdam: adam_chunk<kSplit, kWithRealign>(p, d, local * kChunkElems); break;
      case kCopy: bytes_chunk<false, kWithRealign>(p, d, local * kChunkBytes); break;
      default: bytes_chunk<true, kWithRealign>(p, d, local * kChunkBytes); break;
    }
  }
}

}  // namespace fsdp
