// Host-side internals shared by the translation units of the C ABI: the
// segment list an entry point builds, the overlap check it runs, and the
// launcher of fsdp::segment_kernel. Not part of the public interface.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "fsdp.h"
#include "segment_kernel.cuh"

namespace fsdp {

// ------------------------------------------------------------ segment table

struct SegmentList {
  std::vector<Seg> seg;
  std::vector<const void*> ptr;

  static bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

  // kStep / kReduce / kAdam: `ptrs` in pool order; width 16 iff all are aligned.
  // A segment with some pointer off 16-byte alignment but every pointer aligned
  // to its element (2 bytes for bf16, 4 for fp32) gets kPhased (the realigned
  // vector path).
  void add_elementwise(SegKind kind, int64_t n, int nrep, const std::vector<const void*>& ptrs) {
    if (n <= 0) return;
    bool ok = true;
    for (const void* q : ptrs) ok = ok && (q == nullptr || aligned16(q));
    Seg d{};
    d.n = n;
    d.kind = kind;
    d.nrep = nrep;
    d.ptr = static_cast<int32_t>(ptr.size());
    d.width = ok ? 16 : 0;
    if (!ok) d.width = phased_code(kind, nrep, ptrs);
    seg.push_back(d);
    ptr.insert(ptr.end(), ptrs.begin(), ptrs.end());
  }

  // The width code of an elementwise segment (not every pointer 16-byte
  // aligned) whose pointers are all aligned to their elements: kPhased, else 0.
  // Pools: kStep W bf16 rows, then nrep x {3 fp32, bf16 out}; kReduce W bf16
  // rows, fp32 out; kAdam fp32 grad, 3 fp32, bf16 out (may be null).
  static int phased_code(SegKind kind, int nrep, const std::vector<const void*>& ptrs) {
    const auto fits = [](const void* q, uintptr_t a) {  // non-null and aligned to a bytes
      return q != nullptr && (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0;
    };
    if (kind == kStep) {
      const size_t w = ptrs.size() - 4 * static_cast<size_t>(nrep);
      if (nrep < 1 || w < 1 || w > ptrs.size()) return 0;
      for (size_t k = 0; k < w; ++k)
        if (!fits(ptrs[k], 2)) return 0;
      for (int r = 0; r < nrep; ++r) {
        const size_t b = w + 4 * static_cast<size_t>(r);
        if (!fits(ptrs[b], 4) || !fits(ptrs[b + 1], 4) || !fits(ptrs[b + 2], 4) || !fits(ptrs[b + 3], 2)) return 0;
      }
      return kPhased;
    }
    if (kind == kReduce) {
      if (ptrs.size() < 2) return 0;
      for (size_t k = 0; k + 1 < ptrs.size(); ++k)
        if (!fits(ptrs[k], 2)) return 0;
      return fits(ptrs.back(), 4) ? kPhased : 0;
    }
    if (kind == kAdam) {
      if (ptrs.size() != 5) return 0;
      for (int a = 0; a < 4; ++a)
        if (!fits(ptrs[a], 4)) return 0;
      return (ptrs[4] == nullptr || fits(ptrs[4], 2)) ? kPhased : 0;
    }
    return 0;
  }

  void add_bytes(SegKind kind, const void* src, void* dst, int64_t bytes) {
    if (bytes <= 0) return;
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | (src ? reinterpret_cast<uintptr_t>(src) : 0);
    int width = 1;
    if ((a & 15u) == 0) {
      width = 16;  // a ragged tail is copied byte by byte
    } else {
      const uintptr_t b = a | static_cast<uintptr_t>(bytes);
      width = (b & 7u) == 0 ? 8 : (b & 3u) == 0 ? 4 : (b & 1u) == 0 ? 2 : 1;
    }
    Seg d{};
    d.n = bytes;
    d.kind = kind;
    d.ptr = static_cast<int32_t>(ptr.size());
    d.width = width;
    seg.push_back(d);
    if (kind == kCopy) ptr.push_back(src);
    ptr.push_back(dst);
  }

  int pool_size(size_t i) const {
    const int32_t end = (i + 1 < seg.size()) ? seg[i + 1].ptr : static_cast<int32_t>(ptr.size());
    return end - seg[i].ptr;
  }
};


// Byte ranges for overlap checks.
struct Range {
  uintptr_t lo, hi;
};

inline Range range_of(const void* p, int64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + static_cast<uintptr_t>(bytes)};
}

class AliasCheck {
 public:
  void output(const void* p, int64_t bytes) {
    if (bytes > 0) out_.push_back(range_of(p, bytes));
  }
  void input(const void* p, int64_t bytes) {
    if (bytes > 0) in_.push_back(range_of(p, bytes));
  }
  // True when outputs are pairwise disjoint and no input overlaps an output.
  bool ok() {
    std::sort(out_.begin(), out_.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
    for (size_t i = 1; i < out_.size(); ++i)
      if (out_[i].lo < out_[i - 1].hi) return false;
    for (const Range& r : in_) {
      // first output whose end lies beyond r.lo (outputs are disjoint, so ends are sorted too)
      auto it = std::upper_bound(out_.begin(), out_.end(), r.lo,
                                 [](uintptr_t v, const Range& o) { return v < o.hi; });
      if (it != out_.end() && it->lo < r.hi) return false;
    }
    return true;
  }

 private:
  std::vector<Range> out_, in_;
};


// Events of one scheduler call: created on construction, released on
// destruction (the runtime releases a pending event once it completes).
struct EventSet {
  std::vector<cudaEvent_t> ev;
  bool ok = true;
  explicit EventSet(int n) : ev(n, nullptr) {
    for (auto& e : ev) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
  }
  ~EventSet() {
    for (auto e : ev)
      if (e) cudaEventDestroy(e);
  }
  EventSet(const EventSet&) = delete;
  EventSet& operator=(const EventSet&) = delete;
};

// Launch the list, splitting it where a descriptor table would overflow. With
// `count` set, nothing is launched and the number of launches is returned there.
// `tma_count`, if set, receives how many of those launches use the TMA form,
// and `interleaved_count` how many of those stage their step chunks in
// interleaved quarter-chunk copies (the second instantiation of the TMA form).
int launch(const SegmentList& list, const Scalars& s, cudaStream_t stream, int* count = nullptr,
           int* tma_count = nullptr, int* interleaved_count = nullptr);

// Layout consistent with its own definition (padding, shard length, W, F).
bool layout_ok(const fsdp_layout_t* L);

// Per-launch fp32 scalars from the Adam hyper-parameters (EINVAL on bad values).
int make_scalars(const fsdp_adam_t* h, int w, Scalars* s);

// Scalars for launches without Adam (reduce-scatter, copies).
Scalars reduce_only_scalars(int w);

}  // namespace fsdp
