// Internal helpers shared by the sm_103a kernels of libkvevict.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvevict.h"

namespace kv {

// ---------------------------------------------------------------------------
// Workspace header: the first 256 bytes of every workspace.
// ---------------------------------------------------------------------------
struct WsHeader {
  unsigned int err;       // first device check code that fired (0 = none)
  unsigned int info;      // optional detail of that check
  unsigned int pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");
constexpr size_t kWsHeader = 256;

// Device check codes (written to WsHeader::err).
enum DevErr : unsigned int {
  DEV_OK = 0,
  DEV_BUDGET_RANGE = 1,     // a budget outside [w*Hkv, n*Hkv] (clamped)
  DEV_FLAT_CAPACITY = 2,    // the offsets exceed flat_capacity_rows (rows skipped)
  DEV_NO_RESERVE = 3,       // decode append with no reserve row left (append skipped)
  DEV_HEAD_BUDGET = 4,      // head_budget outside [w, n] (clamped)
  DEV_WAIT_TIMEOUT = 5,     // a bounded wait gave up
  DEV_SELECT = 6,           // a selection invariant failed (should never happen)
};

__device__ __forceinline__ void raise_dev(WsHeader* h, unsigned int code, unsigned int info = 0) {
  if (atomicCAS(&h->err, 0u, code) == 0u) h->info = info;
}

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Monotone key of a non-negative float: larger float <=> larger key.  Anything
// that is not > 0 (zero, -0, negative, NaN) maps to 0.
__device__ __forceinline__ uint32_t score_key(float x) {
  return x > 0.0f ? __float_as_uint(x) : 0u;
}

// ---------------------------------------------------------------------------
// Warp / block reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned int warp_sum_u(unsigned int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Inclusive block-wide prefix sum of one unsigned value per thread.
// `scratch` holds at least blockDim.x/32 entries.  Returns the inclusive prefix;
// *total gets the block total.  All threads must call it.
__device__ __forceinline__ unsigned int block_incl_scan(unsigned int v, unsigned int* scratch,
                                                        unsigned int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned int s = lane < nw ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) scratch[lane] = s;
  }
  __syncthreads();
  unsigned int base = warp > 0 ? scratch[warp - 1] : 0u;
  *total = scratch[nw - 1];
  __syncthreads();
  return base + x;
}

// 64-bit inclusive block scan (one value per thread, blockDim.x a multiple of 32, at most
// 1024); *total receives the block's sum.  Ends with a barrier.
__device__ __forceinline__ int64_t block_incl_scan64(int64_t v, int64_t* scratch, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t s = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) scratch[lane] = s;
  }
  __syncthreads();
  const int64_t base = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[nw - 1];
  __syncthreads();
  return base + x;
}

// Histogram update of one bin per lane (0xFFFFFFFF = none) with runs of equal bins in
// adjacent lanes merged into one add (max-pooled scores come in plateaus, so equal keys
// sit next to each other; other repeats fall back to the atomic unit).  Warps with no
// bin skip the vote.  All 32 lanes must call it.
__device__ __forceinline__ void hist_add_runs(uint32_t* hist, uint32_t bin) {
  if (__ballot_sync(0xFFFFFFFFu, bin != 0xFFFFFFFFu) == 0u) return;
  const int lane = threadIdx.x & 31;
  const uint32_t prev = __shfl_up_sync(0xFFFFFFFFu, bin, 1);
  const bool start = lane == 0 || prev != bin;
  const uint32_t starts = __ballot_sync(0xFFFFFFFFu, start);
  const uint32_t after = starts & ~((2u << lane) - 1u);   // run starts after this lane
  const int next = after ? __ffs(after) - 1 : 32;
  if (start && bin != 0xFFFFFFFFu) atomicAdd(&hist[bin], (uint32_t)(next - lane));
}

__host__ __device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace kv
