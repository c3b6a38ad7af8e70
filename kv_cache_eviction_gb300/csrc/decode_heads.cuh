// Per-head geometry of a decode step over the flat cache, shared by the decode kernels that
// cut heads into parts (decode_parts.cu, decode_tc.cu).
#pragma once

#include "kv_internal.cuh"

namespace kv {

// The flat rows a head holds and whether the new row is appended to it: a head reads
// min(len, end - base) rows (clipped to the flat capacity) and appends at base + len when
// that row is below both its end and the capacity.  Rows at or past the head's end or the
// capacity are never touched.
struct HeadRows {
  int64_t base;
  int32_t flat, len;
  bool app;
};

__device__ __forceinline__ HeadRows head_rows_of(int64_t base, int64_t end, int len, int64_t cap,
                                                 bool has_new) {
  const int64_t e = end < cap ? end : cap;
  HeadRows r{base, 0, len, false};
  if (e > base && base >= 0) {
    int64_t f = len > 0 ? (int64_t)len : 0;
    if (f > e - base) f = e - base;
    r.flat = (int32_t)f;
    r.app = has_new && len >= 0 && base + len < end && base + len < cap;
  }
  return r;
}

__device__ __forceinline__ HeadRows head_rows(const int64_t* __restrict__ cu,
                                              const int32_t* lens, int h, int Hkv,
                                              int64_t cap, bool has_new) {
  const int seg = h / Hkv, g = h - seg * Hkv;
  const int64_t base = cu[(int64_t)seg * (Hkv + 1) + g];
  const int64_t end = cu[(int64_t)seg * (Hkv + 1) + g + 1];
  return head_rows_of(base, end, lens[h], cap, has_new);
}

// Atomic add with release semantics (this thread's earlier memory accesses, and those
// ordered before them by a CTA barrier, are ordered before it); returns the old value.  Like
// any fence, it holds the thread until the bulk copies it issued have landed: use it only
// where the thread has none in flight.
__device__ __forceinline__ uint32_t atom_add_release_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

}  // namespace kv
