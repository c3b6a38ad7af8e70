// Per-head budgets of every (sequence, layer).
//
// Ada-KV Algorithm 1: concatenate the heads' scores, take the layer-wide top B', count how
// many of them each head owns (f_g).  Ada-KV Algorithm 2, safeguard: blend f_g with the
// uniform share B'/Hkv, exact integers, alpha on the uniform side.  LAVa, uncertainty-based
// layer budgets: each layer's share of the sequence's total is proportional to the entropy
// of its normalised scores.
//
// Two sweeps over the scores, each one wave of CTAs streaming its chunk of a layer through a
// ring of bulk copies, and no sort:
//  1. per layer, a histogram of the first digit (top 11 bits of the fp32 bit pattern) of the
//     largest key of every aligned group of 4, and (LAVa) the partial sums of s and s ln s;
//  2. after the layer budgets, the bin g holding the B'-th largest group maximum bounds tau,
//     the B'-th largest key, from below: at least B' groups, so at least B' keys, have a
//     first digit >= g.  The second sweep lists every key with a first digit >= g, in
//     position order, per CTA.  The last CTA of the layer to finish finds tau and the
//     tau-equal quota with an exact radix select (11/11/10 bits) over that union, counts
//     each head's keys above and at tau from it, and blends the head budgets.
// A union longer than its capacity (large budgets) makes that CTA run the radix select over
// every key of the layer instead.  Consecutive sweeps walk their chunks in opposite
// directions, so the second starts on the part of the scores the first left in L2.
#include "bulk_ring.cuh"
#include "kv_internal.cuh"
#include "radix_select.cuh"

namespace kv {

namespace {
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMinBlocks = 3;        // resident CTAs per SM the sweeps are sized for
constexpr int kRingStages = 4;
constexpr int kRingStage = 12288;    // bytes per ring stage (768 groups of 4 keys)
constexpr int kRingBytes = kRingStages * kRingStage;
constexpr int kGroups = kRingStage / 16;   // 4-key groups per ring stage
using SweepRing = BulkRing<kRingStages, kRingStage>;
constexpr int kBins = 2048;
constexpr int kMaxHeads = 256;
constexpr int kMaxChunks = 512;      // CTAs per layer
constexpr int64_t kUnionPerLayer = 65536;   // candidate keys a layer's union can hold
constexpr uint32_t kNoBin = 0xFFFFFFFFu;

// Keys per CTA of a layer: a multiple of 4, so the chunks of an aligned layer are aligned.
__host__ __device__ __forceinline__ int64_t chunk_len(int64_t N, int nch) {
  return cdiv(cdiv(N, nch), 4) * 4;
}

// The index a >= i0 of x's first 16-byte aligned key at or after x + i0 (at most i1).
__device__ __forceinline__ int64_t aligned_from(const float* x, int64_t i0, int64_t i1) {
  const uintptr_t addr = reinterpret_cast<uintptr_t>(x + i0);
  const int64_t a = i0 + (int64_t)(((16u - (uint32_t)(addr & 15u)) & 15u) >> 2);
  return a < i1 ? a : i1;
}

// True in every thread of the CTA that is the n-th and last of its layer to get here; its
// reads of the other CTAs' results come after a fence.  The counter is left at zero.
__device__ __forceinline__ bool last_of_layer(uint32_t* done, uint32_t n, uint32_t* flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t t = atomicAdd(done, 1u);
    *flag = t == n - 1 ? 1u : 0u;
    if (t == n - 1) *done = 0u;
  }
  __syncthreads();
  const bool last = *flag != 0u;
  if (last) __threadfence();
  return last;
}

// Block-wide sums; every thread gets the total (the same order for every thread).
__device__ __forceinline__ double block_sum_dbl(double v, double* red) {
  v = warp_sum_d(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  double t = 0.0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  __syncthreads();
  return t;
}
__device__ __forceinline__ long long block_sum_ll(long long v, long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  long long t = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
  __syncthreads();
  return t;
}
}  // namespace

// ---------------------------------------------------------------------------------------
// Sweep 1: first digit of every group's largest key; (LAVa) partial sums of s, s ln s
// ---------------------------------------------------------------------------------------

// Grid (chunks, layers).  The chunk's aligned middle streams through the ring; the < 4 keys
// on either side are read directly by thread 0 as one more group each.  LAVa: s ln s in
// float; float runs of 16 keys are added into a compensated float sum (Kahan), which goes to
// fp64 once per thread (fp64 arithmetic is scarce on this part).
template <bool ENTROPY>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
alloc_sweep1(const float* __restrict__ scores, int64_t N, int nch, double2* __restrict__ part,
             uint32_t* __restrict__ ghist, WsHeader* hdr) {
  __shared__ uint32_t hist[kBins];
  __shared__ double sa[kWarps], sb[kWarps];
  __shared__ uint64_t rfull[kRingStages];
  extern __shared__ __align__(128) unsigned char ring_mem[];
  const int64_t seg = blockIdx.y;
  SweepRing R;
  R.init(ring_mem, rfull);
  for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0u;
  __syncthreads();
  const float* x = scores + seg * N;
  const int64_t per = chunk_len(N, nch);
  const int64_t i0 = min(N, (int64_t)blockIdx.x * per), i1 = min(N, i0 + per);
  const int64_t a = aligned_from(x, i0, i1);
  const int64_t nv = (i1 - a) >> 2, b = a + 4 * nv;
  float sA = 0.f, cA = 0.f, sB = 0.f, cB = 0.f;   // compensated sums and their corrections
  float ra = 0.f, rb = 0.f;
  int groups = 0;
  auto kahan = [](float& sum, float& c, float v) {
    const float y = v - c;
    const float t = sum + y;
    c = (t - sum) - y;
    sum = t;
  };
  // one group: the four values v, bit c of vm set when value c is a key of the chunk
  auto visit = [&](const float4& v, uint32_t vm) {
    const float xs[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if ((vm >> c) & 1u) {
        m = max(m, score_key(xs[c]));
        if (ENTROPY && xs[c] > 0.0f) {
          ra += xs[c];
          rb += xs[c] * (__log2f(xs[c]) * 0.69314718055994531f);
        }
      }
    }
    hist_add_runs(hist, vm ? m >> 21 : kNoBin);
    if (ENTROPY && ++groups == 4) {
      kahan(sA, cA, ra);
      kahan(sB, cB, rb);
      ra = rb = 0.f;
      groups = 0;
    }
  };
  // the partial groups on either side: keys [i0, a) and [b, i1)
  {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t vm = 0u;
    if (threadIdx.x == 0)
      for (int64_t i = i0; i < a; ++i) {
        (&v.x)[i - i0] = x[i];
        vm |= 1u << (i - i0);
      }
    visit(v, vm);
    v = make_float4(0.f, 0.f, 0.f, 0.f);
    vm = 0u;
    if (threadIdx.x == 0)
      for (int64_t i = b; i < i1; ++i) {
        (&v.x)[i - b] = x[i];
        vm |= 1u << (i - b);
      }
    visit(v, vm);
  }
  const bool ok = ring_pass(R, reinterpret_cast<const unsigned char*>(x + a), nullptr, nv * 16,
                            false, [&](const unsigned char* st, const unsigned char*, int64_t,
                                       uint32_t bytes) {
    const int ng = (int)(bytes / 16);
    const float4* v4 = reinterpret_cast<const float4*>(st);
    for (int jb = 0; jb < kGroups; jb += kThreads) {
      const int j = jb + (int)threadIdx.x;
      visit(j < ng ? v4[j] : make_float4(0.f, 0.f, 0.f, 0.f), j < ng ? 0xFu : 0u);
    }
  });
  if (!ok && threadIdx.x == 0) raise_dev(hdr, DEV_WAIT_TIMEOUT, 0xA00u);
  if (ENTROPY) {
    kahan(sA, cA, ra);
    kahan(sB, cB, rb);
    const double dA = warp_sum_d((double)sA - (double)cA);
    const double dB = warp_sum_d((double)sB - (double)cB);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
      sa[warp] = dA;
      sb[warp] = dB;
    }
  }
  __syncthreads();
  if (ENTROPY && threadIdx.x == 0) {
    double ta = 0.0, tb = 0.0;
    for (int i = 0; i < kWarps; ++i) {
      ta += sa[i];
      tb += sb[i];
    }
    part[seg * nch + blockIdx.x] = make_double2(ta, tb);
  }
  uint32_t* G = ghist + seg * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads) {
    const uint32_t c = hist[i];
    if (c) atomicAdd(&G[i], c);
  }
}

// ---------------------------------------------------------------------------------------
// Layer budgets (B' of every layer) and the bound g of every layer
// ---------------------------------------------------------------------------------------

// LAVa: the capped proportional split of R = total - L*w*Hkv over the L layers of sequence
// b, with floors and largest remainders (ties to the lower layer); returns B' of layer lme.
// Every thread owns the layers l = tid (mod blockDim); sums over the active layers are block
// reductions and the largest remainders are ranks each thread counts for its own layers.
// Every CTA of a sequence computes the same split (same inputs, same order).
constexpr int kMaxLayers = 1024;
struct SplitSmem {
  double e[kMaxLayers], frac[kMaxLayers];
  int64_t sel[kMaxLayers];   // -1: active; >= 0: capped at that value
  double red_d[kWarps];
  long long red_i[kWarps];
  int64_t mine;
};
__device__ int64_t lava_layer_share(SplitSmem& sm, const double2* part, int nch, int L, int Hkv,
                                    int n, int w, int C, int64_t total, int b, int lme,
                                    WsHeader* hdr) {
  for (int l = threadIdx.x; l < L; l += blockDim.x) {
    double S = 0.0, T = 0.0;
    const double2* p = part + ((int64_t)b * L + l) * nch;
    for (int c = 0; c < nch; ++c) {
      const double2 v = p[c];
      S += v.x;
      T += v.y;
    }
    double el = 0.0;
    if (S > 0.0) el = (log(S) - T / S) / ((double)Hkv * (double)n);
    sm.e[l] = el > 0.0 ? el : 0.0;
    sm.sel[l] = -1;
  }
  const int64_t cap = (int64_t)Hkv * C;
  int64_t R = total - (int64_t)L * w * Hkv;
  if (R < 0 || R > (int64_t)L * cap) {
    if (threadIdx.x == 0 && lme == 0) raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)b);
    R = R < 0 ? 0 : (int64_t)L * cap;
  }
  // a thread reads and writes only its own layers' e/sel/frac until the ranks below
  int64_t rem = R;
  for (;;) {
    double es = 0.0;
    long long na = 0;
    for (int l = threadIdx.x; l < L; l += blockDim.x)
      if (sm.sel[l] < 0) {
        es += sm.e[l];
        ++na;
      }
    const double esum = block_sum_dbl(es, sm.red_d);
    const long long active = block_sum_ll(na, sm.red_i);
    long long nover = 0;
    for (int l = threadIdx.x; l < L; l += blockDim.x) {
      if (sm.sel[l] >= 0) continue;
      const double q = esum > 0.0 ? (double)rem * sm.e[l] / esum : (double)rem / (double)active;
      sm.frac[l] = q;
      if (q > (double)cap) ++nover;
    }
    nover = block_sum_ll(nover, sm.red_i);
    if (nover == 0 || active == 0) break;
    for (int l = threadIdx.x; l < L; l += blockDim.x)
      if (sm.sel[l] < 0 && sm.frac[l] > (double)cap) sm.sel[l] = cap;
    rem -= (int64_t)nover * cap;
  }
  long long used = 0;
  for (int l = threadIdx.x; l < L; l += blockDim.x) {
    if (sm.sel[l] >= 0) continue;
    const double f = floor(sm.frac[l]);
    sm.frac[l] -= f;                 // keep only the fractional part
    sm.sel[l] = -2 - (int64_t)f;     // active: the floor is stored as -2 - floor
    used += (long long)f;
  }
  const int64_t left = rem - (int64_t)block_sum_ll(used, sm.red_i);   // also a barrier
  // largest remainders: an active layer gets one more unit when fewer than `left` active
  // layers precede it in (fraction desc, layer asc) order
  if (lme % (int)blockDim.x == (int)threadIdx.x) {
    int64_t v = sm.sel[lme];
    if (v <= -2) {
      const double fl = sm.frac[lme];
      int64_t before = 0;
      for (int m = 0; m < L; ++m)
        if (sm.sel[m] <= -2 && (sm.frac[m] > fl || (sm.frac[m] == fl && m < lme))) ++before;
      v = (-2 - v) + (before < left ? 1 : 0);
    }
    sm.mine = v;
  }
  __syncthreads();
  return sm.mine;
}

// One CTA per (sequence, layer): B' (LAVa split, or the given layer budget less the window,
// range-checked), then g, the bin of the group-maximum histogram holding the B'-th largest
// group maximum (2048 when B' == 0: no candidates).
__global__ void __launch_bounds__(kThreads)
alloc_bound(const double2* __restrict__ part, int nch, int L, int Hkv, int n, int w, int C,
            const int64_t* __restrict__ budget, int entropy, int32_t* __restrict__ layer_budget,
            int64_t* __restrict__ bprime, const uint32_t* __restrict__ ghist,
            uint32_t* __restrict__ gbin, WsHeader* hdr) {
  __shared__ SplitSmem sm;
  __shared__ uint32_t scr[40], res[2];
  const int64_t seg = blockIdx.x;
  const int64_t N = (int64_t)Hkv * C;
  int64_t Bp;
  if (entropy) {
    const int b = (int)(seg / L), lme = (int)(seg - (int64_t)b * L);
    Bp = lava_layer_share(sm, part, nch, L, Hkv, n, w, C, budget[b], b, lme, hdr);
  } else {
    Bp = budget[seg] - (int64_t)w * Hkv;
    if (Bp < 0 || Bp > N) {
      if (threadIdx.x == 0) raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)seg);
      Bp = Bp < 0 ? 0 : N;
    }
  }
  block_pick<kThreads>(ghist + seg * kBins, kBins, (uint32_t)(Bp > 0 ? Bp : 1), scr, res);
  __syncthreads();
  if (threadIdx.x == 0) {
    bprime[seg] = Bp;
    layer_budget[seg] = (int32_t)(Bp + (int64_t)w * Hkv);
    gbin[seg] = Bp > 0 ? res[0] : 2048u;
  }
}

// ---------------------------------------------------------------------------------------
// Sweep 2: the union of keys with first digit >= g; the last CTA of a layer finishes it
// ---------------------------------------------------------------------------------------

struct FinishSmem {
  union {
    uint32_t hist[kBins];          // the radix passes
    struct {                       // then the blend
      int64_t srem[kMaxHeads];
      int32_t sBg[kMaxHeads];
    } b;
  };
  uint32_t scr[40], res[2];
  uint32_t cnt[2 * kMaxHeads];     // per head: keys above tau, keys equal to tau
  uint32_t cstart[kMaxChunks + 1]; // the union's chunk regions, concatenated
  int64_t sleft;
  uint32_t flag;
};

// Radix select of the Bp-th largest key over a sequence of keys visited by each(fn), where
// each(fn) calls fn(key, ok) the same number of times in every thread; pass 0 counts only
// first digits >= g.  Leaves (tau, keq) in res[0..1].
template <typename Each>
__device__ void radix_tau(FinishSmem& sm, uint32_t Bp, uint32_t g, Each&& each) {
  uint32_t prefix = 0, mask = 0, krem = Bp;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = threadIdx.x; i < nb; i += kThreads) sm.hist[i] = 0u;
    __syncthreads();
    each([&](uint32_t k, bool ok) {
      const bool in = ok && (pass == 0 ? (k >> 21) >= g : (k & mask) == prefix);
      hist_add_runs(sm.hist, in ? (k >> sh) & (uint32_t)(nb - 1) : kNoBin);
    });
    __syncthreads();
    block_pick<kThreads>(sm.hist, nb, krem, sm.scr, sm.res);
    __syncthreads();
    prefix |= sm.res[0] << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    krem = sm.res[1];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    sm.res[0] = prefix;
    sm.res[1] = krem;
  }
  __syncthreads();
}

// Grid (chunks, layers).  Walks the chunk backwards (the tail keys, the ring's chunks last to
// first, the head keys) and fills the CTA's union region from its end, so the region
// [fill, UC) lists the chunk's candidate positions in ascending order.
__global__ void __launch_bounds__(kThreads, kMinBlocks)
alloc_sweep2(const float* __restrict__ scores, int Hkv, int C, int nch,
             const uint32_t* __restrict__ gbin, const int64_t* __restrict__ bprime,
             int32_t* __restrict__ upos, uint32_t* __restrict__ ukey, uint32_t* __restrict__ ufill,
             uint32_t* __restrict__ uover, int64_t UC, uint32_t* __restrict__ done, int w,
             uint32_t an, uint32_t ad, int32_t* __restrict__ head_budget, WsHeader* hdr) {
  __shared__ FinishSmem sm;
  __shared__ uint64_t rfull[kRingStages];
  extern __shared__ __align__(128) unsigned char ring_mem[];
  const int64_t seg = blockIdx.y;
  const int64_t N = (int64_t)Hkv * C;
  const uint32_t g = gbin[seg];
  const int64_t Bp = bprime[seg];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* x = scores + seg * N;
  const int64_t per = chunk_len(N, nch);
  const int64_t i0 = min(N, (int64_t)blockIdx.x * per), i1 = min(N, i0 + per);
  int32_t* P = upos + (seg * nch + blockIdx.x) * UC;
  uint32_t* K = ukey + (seg * nch + blockIdx.x) * UC;
  uint32_t fill = (uint32_t)UC;
  bool over = false;
  if (g < 2048u) {
    SweepRing R;
    R.init(ring_mem, rfull);
    // a key is a candidate when its first digit is >= g: for x > 0 the key is x's bit
    // pattern, so the test is x >= the float whose bit pattern is g << 21
    const float t = __uint_as_float(min(g, 1023u) << 21);
    auto is_cand = [&](float v) { return g == 0u || (g < 1024u && v >= t); };
    const int64_t a = aligned_from(x, i0, i1);
    const int64_t nv = (i1 - a) >> 2, b = a + 4 * nv;
    // the keys outside the aligned middle, taken by thread 0 from the last down
    auto side = [&](int64_t lo, int64_t hi) {
      if (threadIdx.x == 0) {
        uint32_t f = fill;
        bool ov = over;
        for (int64_t i = hi - 1; i >= lo && !ov; --i) {
          const float v = x[i];
          if (!is_cand(v)) continue;
          if (f == 0u) {
            ov = true;
            break;
          }
          --f;
          P[f] = (int32_t)i;
          K[f] = score_key(v);
        }
        sm.res[0] = f;
        sm.res[1] = ov ? 1u : 0u;
      }
      __syncthreads();
      fill = sm.res[0];
      over = sm.res[1] != 0u;
      __syncthreads();
    };
    side(b, i1);
    constexpr int kPerWarp = kGroups / kWarps;   // groups of a ring chunk per warp, in order
    const bool ok = ring_pass(R, reinterpret_cast<const unsigned char*>(x + a), nullptr, nv * 16,
                              true, [&](const unsigned char* st, const unsigned char*,
                                        int64_t off, uint32_t bytes) {
      if (over) return;   // the same in every thread
      const int ng = (int)(bytes / 16);
      const float4* v4 = reinterpret_cast<const float4*>(st);
      uint32_t cmu[kPerWarp / 32];
      uint32_t wc = 0;
#pragma unroll
      for (int u = 0; u < kPerWarp / 32; ++u) {
        const int j = warp * kPerWarp + u * 32 + lane;
        uint32_t cm = 0u;
        if (j < ng) {
          const float4 v = v4[j];
          if (is_cand(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w))))
            cm = (is_cand(v.x) ? 1u : 0u) | (is_cand(v.y) ? 2u : 0u) |
                 (is_cand(v.z) ? 4u : 0u) | (is_cand(v.w) ? 8u : 0u);
        }
        cmu[u] = cm;
        wc += __popc(cm);
      }
      wc = warp_sum_u(wc);
      if (lane == 0) sm.scr[warp] = wc;
      __syncthreads();
      uint32_t c = lane < kWarps ? sm.scr[lane] : 0u, ci = c;
#pragma unroll
      for (int d = 1; d < kWarps; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, ci, d);
        if (lane >= d) ci += y;
      }
      const uint32_t T = __shfl_sync(0xFFFFFFFFu, ci, kWarps - 1);
      const uint32_t before = __shfl_sync(0xFFFFFFFFu, ci - c, warp);
      if (T == 0u) return;
      if (T > fill) {
        over = true;
        return;
      }
      uint32_t o = fill - T + before;
#pragma unroll
      for (int u = 0; u < kPerWarp / 32; ++u) {
        const int j = warp * kPerWarp + u * 32 + lane;
        const uint32_t nc = __popc(cmu[u]);
        uint32_t incl = nc;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
          if (lane >= d) incl += y;
        }
        if (cmu[u]) {
          const float4 v = v4[j];
          const float vs[4] = {v.x, v.y, v.z, v.w};
          uint32_t q = o + incl - nc;
          const int64_t i = a + off / 4 + 4 * (int64_t)j;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            if ((cmu[u] >> cc) & 1u) {
              P[q] = (int32_t)(i + cc);
              K[q] = score_key(vs[cc]);
              ++q;
            }
        }
        o += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      fill -= T;
    });
    if (!ok) {
      if (threadIdx.x == 0) raise_dev(hdr, DEV_WAIT_TIMEOUT, 0xA20u);
      over = true;
    }
    if (!over) side(i0, a);
  }
  if (threadIdx.x == 0) {
    ufill[seg * nch + blockIdx.x] = fill;
    if (over) atomicOr(&uover[seg], 1u);
  }
  if (!last_of_layer(done + seg, (uint32_t)nch, &sm.flag)) return;

  // ---- the last CTA of the layer: tau, keq and the per-head counts
  for (int i = threadIdx.x; i < 2 * Hkv; i += kThreads) sm.cnt[i] = 0u;
  const bool overflow = __ldcg(&uover[seg]) != 0u;
  if (threadIdx.x == 0) {
    uint32_t s0 = 0;
    for (int c = 0; c < nch; ++c) {
      sm.cstart[c] = s0;
      s0 += (uint32_t)UC - __ldcg(&ufill[seg * nch + c]);
    }
    sm.cstart[nch] = s0;
  }
  __syncthreads();
  uint32_t tau = 0xFFFFFFFFu, keq = 0u;   // no key equals 0xFFFFFFFF
  if (Bp > 0) {
    const uint32_t U = sm.cstart[nch];
    // union entry t lives in chunk region c (cstart[c] <= t < cstart[c + 1]) at offset
    // UC - (its region's length) + (t - cstart[c])
    auto where = [&](uint32_t t) -> int64_t {
      int lo = 0, hi = nch;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm.cstart[mid] <= t) lo = mid; else hi = mid;
      }
      return (seg * nch + lo) * UC + (UC - (int64_t)(sm.cstart[lo + 1] - sm.cstart[lo])) +
             (int64_t)(t - sm.cstart[lo]);
    };
    auto tally = [&](int64_t pos, uint32_t k) {
      const int h = (int)(pos / C);
      if (k > tau) atomicAdd(&sm.cnt[2 * h], 1u);
      else if (k == tau) atomicAdd(&sm.cnt[2 * h + 1], 1u);
    };
    if (!overflow && U <= (uint32_t)(kRingBytes / 4)) {
      // the union's keys, gathered into the (idle) ring memory, 4 loads in flight per thread
      uint32_t* Ub = reinterpret_cast<uint32_t*>(ring_mem);
      for (uint32_t tb = 0; tb < U; tb += 4 * kThreads) {
        uint32_t kk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t t = tb + u * kThreads + threadIdx.x;
          kk[u] = t < U ? __ldcg(ukey + where(t)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t t = tb + u * kThreads + threadIdx.x;
          if (t < U) Ub[t] = kk[u];
        }
      }
      __syncthreads();
      auto each = [&](auto&& fn) {
        for (uint32_t tb = 0; tb < U; tb += kThreads) {
          const uint32_t t = tb + threadIdx.x;
          fn(t < U ? Ub[t] : 0u, t < U);
        }
      };
      radix_tau(sm, (uint32_t)Bp, g, each);
      tau = sm.res[0];
      keq = sm.res[1];
      for (uint32_t t = threadIdx.x; t < U; t += kThreads) {
        const uint32_t k = Ub[t];
        if (k >= tau) tally(__ldcg(upos + where(t)), k);
      }
    } else if (!overflow) {
      // a union longer than the ring memory: read from L2, 8 keys per thread in flight
      auto each = [&](auto&& fn) {
        for (uint32_t tb = 0; tb < U; tb += 8 * kThreads) {
          uint32_t kk[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t t = tb + u * kThreads + threadIdx.x;
            kk[u] = t < U ? __ldcg(ukey + where(t)) : 0u;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) fn(kk[u], tb + u * kThreads + threadIdx.x < U);
        }
      };
      radix_tau(sm, (uint32_t)Bp, g, each);
      tau = sm.res[0];
      keq = sm.res[1];
      for (uint32_t t = threadIdx.x; t < U; t += kThreads) {
        const int64_t e = where(t);
        const uint32_t k = __ldcg(ukey + e);
        if (k >= tau) tally(__ldcg(upos + e), k);
      }
    } else {
      // every key of the layer
      auto each = [&](auto&& fn) {
        for (int64_t ib = 0; ib < N; ib += kThreads) {
          const int64_t i = ib + threadIdx.x;
          fn(i < N ? score_key(x[i]) : 0u, i < N);
        }
      };
      radix_tau(sm, (uint32_t)Bp, 0u, each);
      tau = sm.res[0];
      keq = sm.res[1];
      for (int64_t i = threadIdx.x; i < N; i += kThreads) {
        const uint32_t k = score_key(x[i]);
        if (k >= tau) tally(i, k);
      }
    }
  }
  __syncthreads();
  // f_g: keys above tau in head g, plus tau-equal keys in (head, position) order; then the
  // safeguard blend in exact integers and the largest remainders (ties to the lower head)
  if (threadIdx.x == 0) {
    const int64_t den = (int64_t)ad * Hkv;
    int64_t left_eq = (int64_t)keq, fsum = 0, flo = 0;
    for (int h = 0; h < Hkv; ++h) {
      const int64_t eqh = sm.cnt[2 * h + 1];
      const int64_t take = left_eq < eqh ? left_eq : eqh;
      left_eq -= take;
      const int64_t f = (int64_t)sm.cnt[2 * h] + take;
      fsum += f;
      const int64_t X = (int64_t)an * Bp + (int64_t)(ad - an) * Hkv * f;
      sm.b.sBg[h] = (int32_t)(X / den);
      sm.b.srem[h] = X % den;
      flo += sm.b.sBg[h];
    }
    if (fsum != Bp) raise_dev(hdr, DEV_SELECT, (unsigned)seg);
    sm.sleft = Bp - flo;
  }
  __syncthreads();
  for (int h = threadIdx.x; h < Hkv; h += kThreads) {
    const int64_t rh = sm.b.srem[h];
    int64_t before = 0;
    for (int m = 0; m < Hkv; ++m)
      if (sm.b.srem[m] > rh || (sm.b.srem[m] == rh && m < h)) ++before;
    head_budget[seg * Hkv + h] = sm.b.sBg[h] + (before < sm.sleft ? 1 : 0) + w;
  }
}

// ---------------------------------------------------------------------------------------

AllocPlan alloc_plan(const Shape& s) {
  AllocPlan p{};
  const int64_t S = s.segments();
  const int64_t N = (int64_t)s.Hkv * (s.C() > 0 ? s.C() : 1);
  // one wave of kMinBlocks CTAs per SM over all layers, at least one ring stage per CTA
  int64_t nch = (int64_t)num_sms() * kMinBlocks / (S > 0 ? S : 1);
  const int64_t maxch = cdiv(N, (int64_t)kRingStage / 4);
  if (nch > maxch) nch = maxch;
  if (nch > kMaxChunks) nch = kMaxChunks;
  if (nch < 1) nch = 1;
  nch = cdiv(N, chunk_len(N, (int)nch));   // no empty chunk
  p.nchunkE = (int)nch;
  // a layer's union holds min(N, kUnionPerLayer) keys, split evenly over its CTAs
  const int64_t ucap = N < kUnionPerLayer ? N : kUnionPerLayer;
  p.union_per_cta = cdiv(ucap, nch) + 4;
  size_t off = kWsHeader;
  p.off_bprime = off;
  off += align_up((size_t)S * sizeof(int64_t), 256);
  p.off_epart = off;
  off += align_up((size_t)S * nch * sizeof(double2), 256);
  p.off_gbin = off;
  off += align_up((size_t)S * sizeof(uint32_t), 256);
  p.off_ufill = off;
  off += align_up((size_t)S * nch * sizeof(uint32_t), 256);
  p.off_zero = off;   // cleared by every call: done counters, overflow flags, histograms
  off += align_up((size_t)S * sizeof(uint32_t), 256);
  off += align_up((size_t)S * sizeof(uint32_t), 256);
  off += align_up((size_t)S * kBins * sizeof(uint32_t), 256);
  p.off_union = off;
  off += align_up((size_t)S * nch * p.union_per_cta * sizeof(int32_t), 256);
  off += align_up((size_t)S * nch * p.union_per_cta * sizeof(uint32_t), 256);
  p.off_end = off;
  return p;
}

cudaError_t launch_allocate(const Shape& s, const float* scores, const int64_t* budget,
                            int entropy_mode, uint32_t an, uint32_t ad, int32_t* layer_budget,
                            int32_t* head_budget, char* ws, const AllocPlan& p,
                            cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t S = s.segments();
  if (S <= 0) return cudaSuccess;
  const int C = s.C();
  const int64_t N = (int64_t)s.Hkv * C;
  const int nch = p.nchunkE;
  const int64_t UC = p.union_per_cta;
  int64_t* bprime = reinterpret_cast<int64_t*>(ws + p.off_bprime);
  double2* part = reinterpret_cast<double2*>(ws + p.off_epart);
  uint32_t* gbin = reinterpret_cast<uint32_t*>(ws + p.off_gbin);
  uint32_t* ufill = reinterpret_cast<uint32_t*>(ws + p.off_ufill);
  char* z = ws + p.off_zero;
  uint32_t* done = reinterpret_cast<uint32_t*>(z);
  z += align_up((size_t)S * sizeof(uint32_t), 256);
  uint32_t* uover = reinterpret_cast<uint32_t*>(z);
  z += align_up((size_t)S * sizeof(uint32_t), 256);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(z);
  int32_t* upos = reinterpret_cast<int32_t*>(ws + p.off_union);
  uint32_t* ukey = reinterpret_cast<uint32_t*>(
      ws + p.off_union + align_up((size_t)S * nch * UC * sizeof(int32_t), 256));
  // counters, flags and histograms start at zero
  cudaError_t e = cudaMemsetAsync(ws + p.off_zero, 0, p.off_union - p.off_zero, st);
  if (e != cudaSuccess) return e;
  static bool opted = false;   // the sweeps' rings are dynamic shared memory above 48 KB
  if (!opted) {
    const void* ks[3] = {(const void*)alloc_sweep1<true>, (const void*)alloc_sweep1<false>,
                         (const void*)alloc_sweep2};
    for (const void* k : ks) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (e != cudaSuccess) return e;
    }
    opted = true;
  }
  const dim3 sweep((unsigned)nch, (unsigned)S);
  if (entropy_mode)
    alloc_sweep1<true><<<sweep, kThreads, kRingBytes, st>>>(scores, N, nch, part, ghist, hdr);
  else
    alloc_sweep1<false><<<sweep, kThreads, kRingBytes, st>>>(scores, N, nch, part, ghist, hdr);
  alloc_bound<<<(unsigned)S, kThreads, 0, st>>>(part, nch, s.L, s.Hkv, s.n, s.w, C, budget,
                                                entropy_mode, layer_budget, bprime, ghist, gbin,
                                                hdr);
  alloc_sweep2<<<sweep, kThreads, kRingBytes, st>>>(scores, s.Hkv, C, nch, gbin, bprime, upos,
                                                    ukey, ufill, uover, UC, done, s.w, an, ad,
                                                    head_budget, hdr);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace kv
