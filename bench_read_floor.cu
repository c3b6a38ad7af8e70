// The floor under any HBM-bound kernel at a given size: how long does merely reading S bytes
// that are not in L2 take on this GPU?  A decode step over a 128K-context flat cache moves
// 17-33 MB, where launch and DRAM latency weigh as much as bandwidth, so the fraction of
// HBM peak that a kernel of that size can reach is bounded well below 1 by this measurement,
// not by the kernel.
//
// Two read-only kernels, each summing what it reads so the loads cannot be dropped:
//   read_ldg  - 16-byte loads, 4 in flight per thread, grid-stride, k CTAs per SM;
//   read_bulk - one CTA per SM requests its whole contiguous share up front as bulk copies
//               into shared memory (chunks of 16 KB, one mbarrier each), then reads it.
// For each size: L2 flushed (a 512 MB write) before every launch ("cold") or not ("warm");
// CUDA events around the launch and the kernel's own %globaltimer span (first CTA start to
// last CTA end), median of 7 launches.  Under ncu (gpu__time_duration.sum), the launches
// give the kernel durations that a decode kernel's ncu time compares with.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o /tmp/read_floor bench_read_floor.cu
//   /tmp/read_floor
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <vector>

#include "kv_cache_eviction_gb300/csrc/tc_ptx.cuh"

using namespace kv::ptx;

namespace {
constexpr int kMaxCtas = 4096;
__device__ unsigned long long g_t0[kMaxCtas], g_t1[kMaxCtas];

__global__ void flush_l2(uint4* p, size_t n16, unsigned v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(v, v, v, v);
}

__global__ void __launch_bounds__(256) read_ldg(const uint4* __restrict__ p, size_t n16,
                                                unsigned* sink) {
  if (threadIdx.x == 0) g_t0[blockIdx.x] = globaltimer();
  unsigned acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldg(p + i), b = __ldg(p + i + stride), c = __ldg(p + i + 2 * stride),
                d = __ldg(p + i + 3 * stride);
    acc ^= a.x ^ b.y ^ c.z ^ d.w;
  }
  for (; i < n16; i += stride) acc ^= __ldg(p + i).x;
  if (acc == 0x12345678u) *sink = acc;
  __syncthreads();
  if (threadIdx.x == 0) g_t1[blockIdx.x] = globaltimer();
}

// CTA c reads bytes [c * share, (c + 1) * share) (share a multiple of 16, at most 208 KB).
constexpr unsigned kChunk = 16384;
constexpr int kMaxChunks = 16;
__global__ void __launch_bounds__(256) read_bulk(const unsigned char* __restrict__ p,
                                                 unsigned share, unsigned* sink,
                                                 unsigned* timeouts) {
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ uint64_t bar[kMaxChunks];
  if (threadIdx.x == 0) g_t0[blockIdx.x] = globaltimer();
  const int nch = (int)((share + kChunk - 1) / kChunk);
  if (threadIdx.x == 0) {
    for (int c = 0; c < nch; ++c) mbar_init(&bar[c], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const unsigned char* src = p + (size_t)blockIdx.x * share;
  if (threadIdx.x == 0)
    for (int c = 0; c < nch; ++c) {
      const unsigned b = share - c * kChunk < kChunk ? share - c * kChunk : kChunk;
      mbar_arrive_expect_tx(&bar[c], b);
      bulk_load(sm + c * kChunk, src + (size_t)c * kChunk, b, &bar[c]);
    }
  unsigned acc = 0;
  bool ok = true;
  for (int c = 0; c < nch; ++c) {   // every wait is bounded (0.2 s each)
    if (!mbar_wait(&bar[c], 0, 200000000ull)) ok = false;
    const unsigned b = share - c * kChunk < kChunk ? share - c * kChunk : kChunk;
    for (unsigned o = threadIdx.x * 16; o < b; o += 256 * 16)
      acc ^= *reinterpret_cast<const unsigned*>(sm + c * kChunk + o);
  }
  if (!ok) atomicAdd(timeouts, 1u);
  if (acc == 0x12345678u) *sink = acc;
  __syncthreads();
  if (threadIdx.x == 0) g_t1[blockIdx.x] = globaltimer();
}

double median(std::vector<double> v) {
  std::sort(v.begin(), v.end());
  return v[v.size() / 2];
}
}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const size_t flush_bytes = 512ull << 20, data_bytes = 512ull << 20;
  void *fl = nullptr, *data = nullptr;
  unsigned *sink = nullptr, *timeouts = nullptr;
  if (cudaMalloc(&fl, flush_bytes) != cudaSuccess || cudaMalloc(&data, data_bytes) != cudaSuccess ||
      cudaMalloc(&sink, 4) != cudaSuccess || cudaMalloc(&timeouts, 4) != cudaSuccess) {
    std::printf("allocation failed\n");
    return 1;
  }
  cudaMemset(data, 1, data_bytes);
  cudaMemset(timeouts, 0, 4);
  cudaFuncSetAttribute(read_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, 212 * 1024);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  std::vector<unsigned long long> t0(kMaxCtas), t1(kMaxCtas);
  auto run = [&](const char* name, int grid, size_t bytes, bool cold, auto launch) {
    std::vector<double> ev, span;
    for (int rep = 0; rep < 9; ++rep) {
      if (cold) flush_l2<<<sms * 4, 512>>>(static_cast<uint4*>(fl), flush_bytes / 16, rep);
      cudaEventRecord(a);
      launch();
      cudaEventRecord(b);
      cudaEventSynchronize(b);
      float ms = 0.f;
      cudaEventElapsedTime(&ms, a, b);
      cudaMemcpyFromSymbol(t0.data(), g_t0, grid * sizeof(unsigned long long));
      cudaMemcpyFromSymbol(t1.data(), g_t1, grid * sizeof(unsigned long long));
      const unsigned long long lo = *std::min_element(t0.begin(), t0.begin() + grid);
      const unsigned long long hi = *std::max_element(t1.begin(), t1.begin() + grid);
      if (rep >= 2) {
        ev.push_back(ms * 1e3);
        span.push_back((hi - lo) * 1e-3);
      }
    }
    const double e = median(ev), s = median(span);
    std::printf("%-18s %7.2f MB %s  events %7.2f us (%5.2f TB/s)  span %7.2f us (%5.2f TB/s)  %s\n",
                name, bytes / 1e6, cold ? "cold" : "warm", e, bytes / e / 1e6, s, bytes / s / 1e6,
                cudaGetErrorString(cudaGetLastError()));
  };
  const double sizes_mb[] = {4, 8, 17, 26, 32, 64, 256};
  for (double mb : sizes_mb) {
    // a multiple of 32 bytes per SM, so that both kernels read exactly `bytes`
    const size_t bytes = ((size_t)(mb * 1e6) / (32 * (size_t)sms)) * 32 * sms;
    for (int cold = 1; cold >= 0; --cold) {
      for (int per : {2, 4, 8}) {
        if (sms * per > kMaxCtas) continue;
        char nm[32];
        std::snprintf(nm, sizeof nm, "ldg %d CTA/SM", per);
        run(nm, sms * per, bytes, cold != 0, [&]() {
          read_ldg<<<sms * per, 256>>>(static_cast<const uint4*>(data), bytes / 16, sink);
        });
      }
      const unsigned share = (unsigned)(bytes / sms);
      if (share <= 208 * 1024)
        run("bulk 1 CTA/SM", sms, bytes, cold != 0, [&]() {
          read_bulk<<<sms, 256, share>>>(static_cast<const unsigned char*>(data), share, sink,
                                         timeouts);
        });
    }
  }
  unsigned h = 0;
  cudaMemcpy(&h, timeouts, 4, cudaMemcpyDeviceToHost);
  std::printf("bulk waits that gave up: %u\n", h);
  return h == 0 ? 0 : 1;
}
