// Per-head selection and the flat cache gather.
//
// Ada-KV Algorithm 2: per-head Top-B_g eviction decision, selection of the kept
// K/V rows, concatenation of the observation window; the flat layout that puts
// every head of a layer into one tensor (cu_seqlens-style offsets), filled by a
// cache-update kernel.  CriticalKV: two-stage greedy selection, stage 1 by the
// attention score, stage 2 by (A + eps) * ||(V W^O)_j||_1.
#include <cstdlib>
#include <cstring>

#include "kv_internal.cuh"
#include "radix_select.cuh"

namespace kv {

namespace {
constexpr int kScanThreads = 1024;
constexpr int kSelThreads = 512;
constexpr int kSelCl = 8;       // CTAs (one cluster) per head
constexpr int kGatherThreads = 256;
}

// 64-bit inclusive block scan (one value per thread).
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

// Offsets of every head in the flat buffer and the initial lengths.
__global__ void __launch_bounds__(kScanThreads)
compact_offsets(const int32_t* __restrict__ head_budget, int64_t H, int Hkv, int w, int n,
                int reserve, int64_t cap, int64_t* __restrict__ cu, int32_t* __restrict__ lens,
                WsHeader* hdr) {
  __shared__ int64_t scratch[32];
  int64_t carry = 0;
  for (int64_t t0 = 0; t0 < H; t0 += kScanThreads) {
    const int64_t h = t0 + threadIdx.x;
    int64_t val = 0;
    if (h < H) {
      int hb = head_budget[h];
      if (hb < w || hb > n) {
        raise_dev(hdr, DEV_HEAD_BUDGET, (unsigned)h);
        hb = hb < w ? w : n;
      }
      lens[h] = hb;
      val = (int64_t)hb + reserve;
    }
    int64_t tot;
    const int64_t incl = block_incl_scan64(val, scratch, &tot);
    if (h < H) {
      const int64_t seg = h / Hkv;
      const int g = (int)(h - seg * Hkv);
      cu[seg * (Hkv + 1) + g] = carry + incl - val;
      if (g == Hkv - 1) cu[seg * (Hkv + 1) + Hkv] = carry + incl;
    }
    carry += tot;
  }
  if (threadIdx.x == 0 && carry > cap) raise_dev(hdr, DEV_FLAT_CAPACITY, 0);
}


// One thread-block cluster of kSelCl CTAs per head: threshold(s), ordered kept positions,
// window and reserve rows.  CTA r of the cluster owns candidate positions
// [r * span, (r + 1) * span), span a multiple of 32 (whole words of the stage-1 bits).
// STAGED: the CTA first copies its span of scores into shared memory (16-byte loads, the
// copy aligned like the source) and every pass of the selection reads it from there, so the
// scores cross HBM once; CriticalKV's stage-2 keys then replace the staged scores in place
// (0 marks a stage-1 position).  Otherwise every pass reads the scores from global memory.
template <bool STAGED>
__global__ void __launch_bounds__(kSelThreads, 2)
compact_select(const float* __restrict__ scores, const float* __restrict__ crit, uint32_t can,
               uint32_t cad, float ceps, const int32_t* __restrict__ lens,
               const int64_t* __restrict__ cu, int Hkv, int C, int w, int reserve,
               int32_t* __restrict__ kept, int64_t cap, uint32_t* __restrict__ flags,
               int64_t words, WsHeader* hdr) {
  __shared__ ClusterSelectSmem rs;
  extern __shared__ float4 stage4[];
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank(), ncta = (int)cl.num_blocks();
  const int64_t h = blockIdx.y;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g];
  const int64_t Bg = (int64_t)lens[h] - w;   // lens was clamped to [w, n]
  const float* S = scores + h * (int64_t)C;
  const int span = ((C + ncta - 1) / ncta + 31) & ~31;
  const int p0 = min(C, rank * span), p1 = min(C, p0 + span);
  auto no = [](int) { return false; };
  float* sv = reinterpret_cast<float*>(stage4);
  int shift = 0;   // sv[i + shift] holds S[i] for i in [p0, p1)
  if (STAGED) {
    // rank 0's cluster histogram starts clear: cleared here, published by the cluster barrier
    // whose wait comes after the staging
    if (rank == 0)
      for (int i = threadIdx.x; i < 2048; i += kSelThreads) rs.ghist[i] = 0u;
    auto arrived = cl.barrier_arrive();
    for (int i = threadIdx.x; i < 2048; i += kSelThreads) rs.hist[i] = 0u;
    const int64_t f0 = h * (int64_t)C + p0, f1 = h * (int64_t)C + p1;
    const int64_t a0 = f0 & ~(int64_t)3;            // aligned start (inside the array)
    const int64_t a1 = f1 > a0 ? (f1 & ~(int64_t)3) : a0;
    shift = (int)(f0 - a0) - p0;
    const int sl0 = p0 + shift, sl1 = p1 + shift;   // the span's slots
    auto valid = [&](int slot) { return (unsigned)(slot - sl0) < (unsigned)(sl1 - sl0); };
    const float4* src = reinterpret_cast<const float4*>(scores + a0);
    const int nv = (int)((a1 - a0) >> 2);
    __syncthreads();   // hist clear
    // copy, and the group-max histogram of the first digit on the way (Ada-KV scores: the
    // key of a score is its score_key)
    constexpr int U = 4;
    for (int jb = 0; jb < nv; jb += U * kSelThreads) {
      float4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = jb + u * kSelThreads + (int)threadIdx.x;
        x[u] = j < nv ? src[j] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = jb + u * kSelThreads + (int)threadIdx.x;
        if (j < nv) stage4[j] = x[u];
        const uint4 r = make_uint4(__float_as_uint(x[u].x), __float_as_uint(x[u].y),
                                   __float_as_uint(x[u].z), __float_as_uint(x[u].w));
        add_group_max<ScoreKeys>(rs, r, j, j < nv, valid);
      }
    }
    for (int64_t f = a1 + threadIdx.x; f < f1; f += kSelThreads) sv[f - a0] = scores[f];
    __syncthreads();
    if (a1 < f1 && threadIdx.x < 32) {   // the group of the scalar tail
      const int q = nv;
      add_group_max<ScoreKeys>(rs, reinterpret_cast<const uint4*>(sv)[q], q, threadIdx.x == 0,
                               valid);
    }
    cl.barrier_wait(std::move(arrived));
  }
  auto sval = [&](int64_t i) -> float { return STAGED ? sv[i + shift] : S[i]; };
  const uint32_t* raw = reinterpret_cast<const uint32_t*>(sv);
  const int s0 = p0 + shift, s1 = p1 + shift;   // the span's slots when staged
  if (crit == nullptr) {
    auto key = [&](int j) { return score_key(sval(j)); };
    const uint32_t n =
        STAGED ? cluster_topk_select_staged<kSelThreads, false, ScoreKeys>(
                     raw, s0, s1, shift, Bg, kept, base, cap, nullptr, rs, true)
               : cluster_topk_select<kSelThreads, false>(p0, p1, Bg, key, no, kept, base, cap,
                                                         nullptr, rs);
    if (rank == 0 && threadIdx.x == 0 && n != (uint32_t)Bg) raise_dev(hdr, DEV_SELECT, (unsigned)h);
  } else {
    const float* Cn = crit + h * (int64_t)C;
    uint32_t* F = flags + h * words;
    const int64_t K1 = ((int64_t)can * Bg) / cad;
    const int64_t K2 = Bg - K1;
    auto key1 = [&](int j) { return score_key(sval(j)); };
    // stage-1 membership bits (each CTA writes and later reads the words of its own span)
    if (STAGED)
      cluster_topk_select_staged<kSelThreads, true, ScoreKeys>(raw, s0, s1, shift, K1, nullptr, 0,
                                                                0, F, rs, true);
    else
      cluster_topk_select<kSelThreads, true>(p0, p1, K1, key1, no, nullptr, 0, 0, F, rs);
    auto in1 = [&](int64_t i) { return ((F[i >> 5] >> (i & 31)) & 1u) != 0u; };
    auto key2g = [&](int64_t i) -> uint32_t {
      if (in1(i)) return 0u;
      const float kap = __fmul_rn(__fadd_rn(sval(i), ceps), Cn[i]);
      return score_key(kap) + 1u;
    };
    uint32_t* sk = reinterpret_cast<uint32_t*>(sv);
    if (STAGED) {
      // the bits were written by this CTA before the barrier that ends the selection
      for (int i = p0 + threadIdx.x; i < p1; i += kSelThreads) sk[i + shift] = key2g(i);
      __syncthreads();
    }
    auto key2 = [&](int j) -> uint32_t { return STAGED ? sk[j + shift] : key2g(j); };
    auto forced2 = [&](int j) { return STAGED ? sk[j + shift] == 0u : in1(j); };
    const uint32_t n =
        STAGED ? cluster_topk_select_staged<kSelThreads, false, StoredKeys>(
                     raw, s0, s1, shift, K2, kept, base, cap, nullptr, rs, false)
               : cluster_topk_select<kSelThreads, false>(p0, p1, K2, key2, forced2, kept, base,
                                                         cap, nullptr, rs);
    if (rank == 0 && threadIdx.x == 0 && n != (uint32_t)Bg) raise_dev(hdr, DEV_SELECT, (unsigned)h);
  }
  for (int t = rank * kSelThreads + threadIdx.x; t < w + reserve; t += ncta * kSelThreads) {
    const int64_t row = base + Bg + t;
    if (row < cap) kept[row] = t < w ? C + t : -1;
  }
  // rank 0's shared memory was read by the other CTAs: none leaves before all are done
  cl.sync();
}

// Copy the kept rows of K and V into the flat buffers, 16 bytes per thread.
__global__ void __launch_bounds__(kGatherThreads)
compact_gather(const char* __restrict__ k, const char* __restrict__ v,
               const int32_t* __restrict__ kept, const int64_t* __restrict__ cu,
               const int32_t* __restrict__ lens, int Hkv, int n, int row_bytes, int64_t cap,
               char* __restrict__ kf, char* __restrict__ vf) {
  const int64_t h = blockIdx.y;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g];
  const int64_t len = lens[h];
  const int vecs = row_bytes >> 4;
  const char* Ks = k + h * (int64_t)n * row_bytes;
  const char* Vs = v + h * (int64_t)n * row_bytes;
  const int64_t total = len * vecs;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / vecs;
    const int c = (int)(idx - r * vecs);
    const int64_t row = base + r;
    if (row >= cap) continue;
    const int64_t src = kept[row];
    if (src < 0 || src >= n) continue;   // never read outside the source head
    const uint4 a = reinterpret_cast<const uint4*>(Ks + src * row_bytes)[c];
    const uint4 b = reinterpret_cast<const uint4*>(Vs + src * row_bytes)[c];
    reinterpret_cast<uint4*>(kf + row * row_bytes)[c] = a;
    reinterpret_cast<uint4*>(vf + row * row_bytes)[c] = b;
  }
}

// KVEVICT_SELECT_PATH=global forces the selection that reads the scores from global memory
// on every pass (the one spans too long for shared memory take); tests compare the two.
static bool global_select_forced() {
  const char* e = std::getenv("KVEVICT_SELECT_PATH");
  return e != nullptr && std::strcmp(e, "global") == 0;
}

CompactPlan compact_plan(const Shape& s, bool critical) {
  CompactPlan p{};
  size_t off = kWsHeader;
  p.off_flags = off;
  p.flag_words = critical ? cdiv(s.C() > 0 ? s.C() : 1, 32) : 0;
  off += align_up((size_t)s.units() * p.flag_words * sizeof(uint32_t), 256);
  p.off_end = off;
  return p;
}

cudaError_t launch_compact(const Shape& s, const void* k, const void* v, const float* scores,
                           const float* crit, uint32_t can, uint32_t cad, float ceps,
                           const int32_t* head_budget, int reserve, int32_t* kept,
                           int64_t* cu, int32_t* lens, void* kf, void* vf, int64_t cap,
                           char* ws, const CompactPlan& p, cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t H = s.units();
  compact_offsets<<<1, kScanThreads, 0, st>>>(head_budget, H, s.Hkv, s.w, s.n, reserve, cap, cu,
                                               lens, hdr);
  {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(kSelCl, (unsigned)H);
    cfg.blockDim = dim3(kSelThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSelCl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // staged when a span (plus the alignment slack) fits next to the selection's own state
    const int C = s.C();
    const int span = ((C + kSelCl - 1) / kSelCl + 31) & ~31;
    const size_t stage_bytes = align_up(((size_t)span + 8) * sizeof(float), 16);
    const bool staged = C > 0 && !global_select_forced() &&
                        stage_bytes + sizeof(ClusterSelectSmem) + 1024 <= max_smem_optin();
    auto kern = staged ? compact_select<true> : compact_select<false>;
    if (staged) {
      static size_t opted = 0;   // the largest size opted in so far
      if (stage_bytes > opted) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)stage_bytes);
        if (e != cudaSuccess) return e;
        opted = stage_bytes;
      }
      cfg.dynamicSmemBytes = stage_bytes;
    }
    cudaError_t e = cudaLaunchKernelEx(
        &cfg, kern, scores, crit, can, cad, ceps, (const int32_t*)lens,
        (const int64_t*)cu, s.Hkv, C, s.w, reserve, kept, cap,
        reinterpret_cast<uint32_t*>(ws + p.off_flags), p.flag_words, hdr);
    if (e != cudaSuccess) return e;
  }
  const int row_bytes = s.d * s.esize();
  int gx = (int)cdiv((int64_t)num_sms() * 16, H);
  if (gx < 1) gx = 1;
  if (gx > 64) gx = 64;
  compact_gather<<<dim3(gx, (unsigned)H), kGatherThreads, 0, st>>>(
      (const char*)k, (const char*)v, kept, cu, lens, s.Hkv, s.n, row_bytes, cap, (char*)kf,
      (char*)vf);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace kv
