// Block-wide radix select of the K largest 32-bit keys, in shared memory.
//
// Used for the layer-wide Top-B' of Ada-KV Algorithm 1 (and LAVa's
// head-flattened eviction) and for the per-head Top-B_g of Algorithm 2 /
// CriticalKV.  No sort: three histogram passes over the keys (11, 11 and 10
// bits, most significant first) narrow down tau, the K-th largest key.  The
// result is (tau, keq): every key > tau is selected, plus the keq lowest-index
// keys equal to tau, which is the (key desc, index asc) total order.
#pragma once

#include "kv_common.cuh"

namespace kv {

struct RadixSmem {
  uint32_t hist[2048];
  uint32_t scratch[32];
  uint32_t res[2];
};

// All threads of the block must call this with the same N and K, 0 <= K <= N.
// key_of(i) must return the same key on every call for the same i.
template <int BLOCK, typename KeyFn>
__device__ void block_topk_threshold(int64_t N, int64_t K, KeyFn key_of, RadixSmem& sm,
                                     uint32_t& tau_out, uint32_t& keq_out) {
  static_assert(BLOCK <= 1024 && (1024 % BLOCK) == 0, "block must divide 1024");
  if (K <= 0) {
    tau_out = 0xFFFFFFFFu;
    keq_out = 0;
    return;
  }
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)K;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = threadIdx.x; i < nb; i += BLOCK) sm.hist[i] = 0u;
    __syncthreads();
    // equal bins in adjacent lanes are added once (see hist_add_runs)
    // 8 keys per thread per step, all fetched before use (latency hiding); the step
    // count is the same for every thread so the warp votes stay convergent
    constexpr int U = 8;
    for (int64_t base = 0; base < N; base += (int64_t)U * BLOCK) {
      uint32_t key[U];
      bool valid[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int64_t i = base + (int64_t)k * BLOCK + threadIdx.x;
        valid[k] = i < N;
        key[k] = valid[k] ? key_of(i) : 0u;
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const uint32_t bin = (valid[k] && (key[k] & mask) == prefix)
                                 ? (key[k] >> sh) & (uint32_t)(nb - 1) : 0xFFFFFFFFu;
        hist_add_runs(sm.hist, bin);
      }
    }
    __syncthreads();
    // Counts from the top bin downwards: thread t owns reversed bins [t*per, (t+1)*per).
    const int per = nb / BLOCK;
    uint32_t local = 0;
    for (int q = 0; q < per; ++q) local += sm.hist[nb - 1 - (threadIdx.x * per + q)];
    uint32_t total;
    const uint32_t incl = block_incl_scan(local, sm.scratch, &total);
    const uint32_t excl = incl - local;
    if (excl < krem && krem <= incl) {
      uint32_t acc = excl;
      for (int q = 0; q < per; ++q) {
        const int bin = nb - 1 - (threadIdx.x * per + q);
        const uint32_t c = sm.hist[bin];
        if (acc + c >= krem) {
          sm.res[0] = (uint32_t)bin;
          sm.res[1] = krem - acc;
          break;
        }
        acc += c;
      }
    }
    __syncthreads();
    prefix |= sm.res[0] << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    krem = sm.res[1];
    __syncthreads();
  }
  tau_out = prefix;
  keq_out = krem;
}

}  // namespace kv
