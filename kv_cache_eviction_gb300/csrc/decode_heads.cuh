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

}  // namespace kv
