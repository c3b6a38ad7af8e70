// A CTA's ring of shared-memory stages filled by untiled bulk copies, for kernels that
// stream long contiguous ranges of global memory (the score sweeps of the selection and
// allocation kernels).
//
// cp.async.bulk moves a chunk from global to shared memory and counts its bytes on the
// stage's mbarrier, so a CTA keeps NS - 1 chunks in flight without holding them in
// registers.  Thread 0 issues; every thread waits for the stage (bounded), reads it, and a
// block barrier frees it before thread 0 refills it with the chunk NS ahead.  Chunks carry a
// sequence number that runs over every pass of the kernel: chunk k lands in stage k % NS
// and completes phase (k / NS) & 1 of that stage's barrier.
#pragma once

#include "kv_common.cuh"
#include "tc_ptx.cuh"

namespace kv {

template <int NS, int SB>
struct BulkRing {
  static_assert(SB % 32 == 0, "stage size");
  unsigned char* buf;   // NS * SB bytes, 16-byte aligned
  uint64_t* full;       // NS barriers
  uint32_t seq;         // chunks of the passes before the current one

  // Thread 0 initialises the barriers; the caller synchronises the block before any pass.
  __device__ void init(unsigned char* b, uint64_t* f) {
    buf = b;
    full = f;
    seq = 0;
    if (threadIdx.x == 0) {
      for (int s = 0; s < NS; ++s) ptx::mbar_init(&full[s], 1);
      ptx::fence_mbar_init();
    }
  }
};

// Streams `nstreams` (1 or 2) byte ranges of n bytes each, src0 and src1 (16-byte aligned,
// n a multiple of 16), through the ring in chunks of SB / nstreams bytes, first chunk to
// last or (rev) last to first.  fn(stage0, stage1, offset, bytes) runs on every thread of
// the block for each chunk, stage0/stage1 holding bytes [offset, offset + bytes) of
// src0/src1.  Returns false, the same in every thread, when a wait gave up: the chunks in
// flight have then been waited for (bounded) and the ring must not be used again.
template <int NS, int SB, typename Fn>
__device__ bool ring_pass(BulkRing<NS, SB>& R, const unsigned char* src0,
                         const unsigned char* src1, int64_t n, bool rev, Fn&& fn) {
  const int ns = src1 ? 2 : 1;
  const int64_t CB = SB / ns;
  const int64_t nch = n > 0 ? (n + CB - 1) / CB : 0;
  auto chunk_off = [&](int64_t t) { return (rev ? nch - 1 - t : t) * CB; };
  auto issue = [&](int64_t t) {
    const int64_t off = chunk_off(t);
    const uint32_t bytes = (uint32_t)(n - off < CB ? n - off : CB);
    const uint32_t k = R.seq + (uint32_t)t;
    unsigned char* st = R.buf + (k % NS) * SB;
    uint64_t* bar = &R.full[k % NS];
    ptx::mbar_arrive_expect_tx(bar, bytes * (uint32_t)ns);
    ptx::bulk_load(st, src0 + off, bytes, bar);
    if (src1) ptx::bulk_load(st + CB, src1 + off, bytes, bar);
  };
  if (threadIdx.x == 0)
    for (int64_t t = 0; t < nch && t < NS; ++t) issue(t);
  bool ok = true;
  int64_t t = 0;
  for (; t < nch; ++t) {
    const uint32_t k = R.seq + (uint32_t)t;
    const bool landed = ptx::mbar_wait_sleep(&R.full[k % NS], (k / NS) & 1u, 500);
    if (__syncthreads_or(!landed)) {
      ok = false;
      break;
    }
    const int64_t off = chunk_off(t);
    const unsigned char* st = R.buf + (k % NS) * SB;
    fn(st, st + CB, off, (uint32_t)(n - off < CB ? n - off : CB));
    __syncthreads();
    if (threadIdx.x == 0 && t + NS < nch) issue(t + NS);
  }
  if (!ok) {
    // chunks [t, t + NS) may still be in flight: let them land before the memory is reused
    if (threadIdx.x == 0)
      for (int64_t u = t; u < nch && u < t + NS; ++u) {
        const uint32_t k = R.seq + (uint32_t)u;
        (void)ptx::mbar_wait(&R.full[k % NS], (k / NS) & 1u, 20000000ull);
      }
    __syncthreads();
  }
  R.seq += (uint32_t)nch;
  return ok;
}

}  // namespace kv
