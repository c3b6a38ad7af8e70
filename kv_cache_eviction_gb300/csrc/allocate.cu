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
//     position order, per CTA (a region as long as the CTA's chunk: it cannot overflow,
//     whatever the budget).  The layer's CTAs then find tau and the tau-equal quota with an
//     exact radix select (11/11/10 bits) over their lists, waiting for one another at
//     bounded barriers (the launch is cooperative), count each head's keys above and at tau,
//     and the layer's first CTA blends the head budgets.
// Consecutive sweeps walk their chunks in opposite directions, so the second starts on the
// part of the scores the first left in L2.
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
  int64_t cap[kMaxLayers];   // most selectable rows the layer can keep
  double red_d[kWarps];
  long long red_i[kWarps];
  int64_t mine;
};
// layer_cap (nullable) [B][L]: the most rows (window included) layer l may keep; the
// layer's selectable share is capped at it as well as at Hkv * C.  With caps, a total that
// the layers cannot hold together leaves every layer at its cap.
__device__ int64_t lava_layer_share(SplitSmem& sm, const double2* part, int nch, int L, int Hkv,
                                    int n, int w, int C, int64_t total, int b, int lme,
                                    const int32_t* layer_cap, WsHeader* hdr) {
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
    int64_t cl = (int64_t)Hkv * C;
    if (layer_cap != nullptr) {
      const int64_t given = (int64_t)layer_cap[(int64_t)b * L + l] - (int64_t)w * Hkv;
      cl = given < 0 ? 0 : given < cl ? given : cl;
    }
    sm.cap[l] = cl;
  }
  long long capsum = 0;
  for (int l = threadIdx.x; l < L; l += blockDim.x) capsum += sm.cap[l];
  capsum = block_sum_ll(capsum, sm.red_i);   // also a barrier: every cap is in place
  int64_t R = total - (int64_t)L * w * Hkv;
  if (R < 0 || (layer_cap == nullptr && R > (int64_t)capsum)) {
    if (threadIdx.x == 0 && lme == 0) raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)b);
    R = R < 0 ? 0 : (int64_t)capsum;
  }
  if (R >= (int64_t)capsum) {   // the layers keep all they can
    __syncthreads();
    return sm.cap[lme];
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
    long long nover = 0, capped = 0;
    for (int l = threadIdx.x; l < L; l += blockDim.x) {
      if (sm.sel[l] >= 0) continue;
      const double q = esum > 0.0 ? (double)rem * sm.e[l] / esum : (double)rem / (double)active;
      sm.frac[l] = q;
      if (q > (double)sm.cap[l]) {
        ++nover;
        capped += sm.cap[l];
      }
    }
    nover = block_sum_ll(nover, sm.red_i);
    capped = block_sum_ll(capped, sm.red_i);
    if (nover == 0 || active == 0) break;
    for (int l = threadIdx.x; l < L; l += blockDim.x)
      if (sm.sel[l] < 0 && sm.frac[l] > (double)sm.cap[l]) sm.sel[l] = sm.cap[l];
    rem -= (int64_t)capped;
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
            const int64_t* __restrict__ budget, int entropy, const int32_t* __restrict__ layer_cap,
            int32_t* __restrict__ layer_budget,
            int64_t* __restrict__ bprime, const uint32_t* __restrict__ ghist,
            uint32_t* __restrict__ gbin, WsHeader* hdr) {
  __shared__ SplitSmem sm;
  __shared__ uint32_t scr[40], res[2];
  const int64_t seg = blockIdx.x;
  const int64_t N = (int64_t)Hkv * C;
  int64_t Bp;
  if (entropy) {
    const int b = (int)(seg / L), lme = (int)(seg - (int64_t)b * L);
    Bp = lava_layer_share(sm, part, nch, L, Hkv, n, w, C, budget[b], b, lme, layer_cap, hdr);
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
// Sweep 2: the union of keys with first digit >= g, then the exact select over it by all
// the CTAs of the layer
// ---------------------------------------------------------------------------------------

struct Sweep2Smem {
  union {
    uint32_t hist[kBins];          // the radix passes
    struct {                       // then the blend
      int64_t srem[kMaxHeads];
      int32_t sBg[kMaxHeads];
    } b;
  };
  uint32_t scr[40], res[2];
  uint32_t cnt[2 * kMaxHeads];     // this CTA's per-head counts: above tau, equal to tau
  uint32_t ok;
};

// Barrier of the CTAs of one layer (co-resident: the kernel is a cooperative launch): the
// call's k-th barrier completes when the layer's counter reaches k * nch.  Writes before it
// (fenced) are visible after it.  The wait is bounded (1 s); a CTA that gives up records
// DEV_WAIT_TIMEOUT and waits no more (its layer's results are then invalid).
__device__ void layer_barrier(uint32_t* ctr, uint32_t target, uint32_t* ok, WsHeader* hdr) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    if (*ok) {
      const uint64_t t0 = ptx::globaltimer();
      while (ptx::ld_acquire_u32(ctr) < target) {
        if (ptx::globaltimer() - t0 > 1000000000ull) {
          raise_dev(hdr, DEV_WAIT_TIMEOUT, 0xA30u);
          *ok = 0u;
          break;
        }
        __nanosleep(64);
      }
    }
  }
  __syncthreads();
}

// Grid (chunks, layers of this launch), a cooperative launch (every CTA resident).  Each CTA
// walks its chunk backwards (the tail keys, the ring's chunks last to first, the head keys),
// listing its candidates from the end of its own region, so [fill, UC) holds them in
// ascending position order; UC is the chunk's length, so a region cannot overflow.  Then
// the layer's CTAs run three radix passes over their regions (each pass: shared-memory
// histogram, added into the layer's global histogram of that pass, a layer barrier, the
// pick repeated in every CTA), count their keys above and at tau per head into the layer's
// counters, and after a last barrier the layer's first CTA blends the head budgets.
__global__ void __launch_bounds__(kThreads, kMinBlocks)
alloc_sweep2(const float* __restrict__ scores, int Hkv, int C, int nch, int64_t seg0,
             const uint32_t* __restrict__ gbin, const int64_t* __restrict__ bprime,
             int32_t* __restrict__ upos, uint32_t* __restrict__ ukey, int64_t UC,
             uint32_t* __restrict__ lhist /*[S][3][kBins]*/, uint32_t* __restrict__ hcnt,
             uint32_t* __restrict__ lbar, int w, uint32_t an, uint32_t ad,
             int32_t* __restrict__ head_budget, WsHeader* hdr) {
  __shared__ Sweep2Smem sm;
  __shared__ uint64_t rfull[kRingStages];
  extern __shared__ __align__(128) unsigned char ring_mem[];
  const int64_t seg = seg0 + blockIdx.y;
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
  if (threadIdx.x == 0) sm.ok = 1u;
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
        for (int64_t i = hi - 1; i >= lo; --i) {
          const float v = x[i];
          if (!is_cand(v)) continue;
          --f;
          P[f] = (int32_t)i;
          K[f] = score_key(v);
        }
        sm.res[0] = f;
      }
      __syncthreads();
      fill = sm.res[0];
      __syncthreads();
    };
    side(b, i1);
    constexpr int kPerWarp = kGroups / kWarps;   // groups of a ring chunk per warp, in order
    const bool ok = ring_pass(R, reinterpret_cast<const unsigned char*>(x + a), nullptr, nv * 16,
                              true, [&](const unsigned char* st, const unsigned char*,
                                        int64_t off, uint32_t bytes) {
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
      if (T == 0u) return;   // the same in every thread
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
    if (!ok && threadIdx.x == 0) {
      raise_dev(hdr, DEV_WAIT_TIMEOUT, 0xA20u);
      sm.ok = 0u;
    }
    side(i0, a);
  }

  // ---- the exact select over the layer's union (every CTA of the layer takes part)
  for (int i = threadIdx.x; i < 2 * Hkv; i += kThreads) sm.cnt[i] = 0u;
  const int nu = (int)(UC - fill);   // this CTA's candidates: P/K[fill, UC)
  uint32_t* bar = lbar + seg;
  uint32_t tau = 0xFFFFFFFFu, keq = 0u;   // no key equals 0xFFFFFFFF
  if (Bp > 0) {
    uint32_t prefix = 0, mask = 0, krem = (uint32_t)Bp;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int nb = pass == 2 ? 1024 : 2048;
      for (int i = threadIdx.x; i < nb; i += kThreads) sm.hist[i] = 0u;
      __syncthreads();
      for (int tb = 0; tb < nu; tb += 8 * kThreads) {
        uint32_t kk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int tt = tb + u * kThreads + (int)threadIdx.x;
          kk[u] = tt < nu ? K[fill + tt] : 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const bool in = tb + u * kThreads + (int)threadIdx.x < nu &&
                          (pass == 0 ? (kk[u] >> 21) >= g : (kk[u] & mask) == prefix);
          hist_add_runs(sm.hist, in ? (kk[u] >> sh) & (uint32_t)(nb - 1) : kNoBin);
        }
      }
      __syncthreads();
      uint32_t* G = lhist + (seg * 3 + pass) * kBins;
      for (int i = threadIdx.x; i < nb; i += kThreads) {
        const uint32_t c = sm.hist[i];
        if (c) atomicAdd(&G[i], c);
      }
      layer_barrier(bar, (uint32_t)(pass + 1) * (uint32_t)nch, &sm.ok, hdr);
      for (int i = threadIdx.x; i < nb; i += kThreads) sm.hist[i] = __ldcg(G + i);
      __syncthreads();
      block_pick<kThreads>(sm.hist, nb, krem, sm.scr, sm.res);
      __syncthreads();
      prefix |= sm.res[0] << sh;
      mask |= (uint32_t)(nb - 1) << sh;
      krem = sm.res[1];
      __syncthreads();
    }
    tau = prefix;
    keq = krem;
    // this CTA's keys above and at tau, per head (every such key is a candidate)
    for (int tt = threadIdx.x; tt < nu; tt += kThreads) {
      const uint32_t k = K[fill + tt];
      if (k < tau) continue;
      const int h = (int)(P[fill + tt] / C);
      atomicAdd(&sm.cnt[2 * h + (k > tau ? 0 : 1)], 1u);
    }
    __syncthreads();
    uint32_t* Hc = hcnt + seg * 2 * Hkv;
    for (int i = threadIdx.x; i < 2 * Hkv; i += kThreads)
      if (sm.cnt[i]) atomicAdd(&Hc[i], sm.cnt[i]);
    layer_barrier(bar, 4u * (uint32_t)nch, &sm.ok, hdr);
    if (blockIdx.x != 0) return;
    for (int i = threadIdx.x; i < 2 * Hkv; i += kThreads) sm.cnt[i] = __ldcg(Hc + i);
    __syncthreads();
  } else if (blockIdx.x != 0) {
    return;
  }
  // ---- the layer's first CTA: f_g = keys above tau in head g plus tau-equal keys in (head,
  // position) order; the safeguard blend in exact integers and the largest remainders (ties
  // to the lower head)
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
    sm.scr[0] = (uint32_t)(Bp - flo);
  }
  __syncthreads();
  const int64_t left = sm.scr[0];
  for (int h = threadIdx.x; h < Hkv; h += kThreads) {
    const int64_t rh = sm.b.srem[h];
    int64_t before = 0;
    for (int m = 0; m < Hkv; ++m)
      if (sm.b.srem[m] > rh || (sm.b.srem[m] == rh && m < h)) ++before;
    head_budget[seg * Hkv + h] = sm.b.sBg[h] + (before < left ? 1 : 0) + w;
  }
}

// ---------------------------------------------------------------------------------------

// CTAs of alloc_sweep2 that can be resident at once (its cooperative launch needs them all).
static int64_t sweep2_resident() {
  static std::atomic<int> slot[kMaxDevices];
  const int occ = per_device(slot, []() {
    int n = 0;
    if (cudaFuncSetAttribute(alloc_sweep2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRingBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, alloc_sweep2, kThreads,
                                                      kRingBytes) != cudaSuccess ||
        n < 1)
      n = 1;
    return n;
  });
  return (int64_t)occ * num_sms();
}

AllocPlan alloc_plan(const Shape& s) {
  AllocPlan p{};
  const int64_t S = s.segments();
  const int64_t N = (int64_t)s.Hkv * (s.C() > 0 ? s.C() : 1);
  // one wave over all layers (or, with more layers than resident CTAs, one CTA per layer and
  // several launches), at least one ring stage per CTA
  int64_t nch = sweep2_resident() / (S > 0 ? S : 1);
  const int64_t maxch = cdiv(N, (int64_t)kRingStage / 4);
  if (nch > maxch) nch = maxch;
  if (nch > kMaxChunks) nch = kMaxChunks;
  if (nch < 1) nch = 1;
  nch = cdiv(N, chunk_len(N, (int)nch));   // no empty chunk
  p.nchunkE = (int)nch;
  p.union_per_cta = chunk_len(N, (int)nch);   // a chunk's candidates fit in its region
  size_t off = kWsHeader;
  p.off_bprime = off;
  off += align_up((size_t)S * sizeof(int64_t), 256);
  p.off_epart = off;
  off += align_up((size_t)S * nch * sizeof(double2), 256);
  p.off_gbin = off;
  off += align_up((size_t)S * sizeof(uint32_t), 256);
  p.off_zero = off;   // cleared by every call: barriers, histograms, per-head counts
  off += align_up((size_t)S * sizeof(uint32_t), 256);
  off += align_up((size_t)S * kBins * sizeof(uint32_t), 256);
  off += align_up((size_t)S * 3 * kBins * sizeof(uint32_t), 256);
  off += align_up((size_t)S * 2 * s.Hkv * sizeof(uint32_t), 256);
  p.off_union = off;
  off += align_up((size_t)S * nch * p.union_per_cta * sizeof(int32_t), 256);
  off += align_up((size_t)S * nch * p.union_per_cta * sizeof(uint32_t), 256);
  p.off_end = off;
  return p;
}

cudaError_t launch_allocate(const Shape& s, const float* scores, const int64_t* budget,
                            int entropy_mode, const int32_t* layer_cap, uint32_t an, uint32_t ad,
                            int32_t* layer_budget, int32_t* head_budget, char* ws,
                            const AllocPlan& p, cudaStream_t st) {
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
  char* z = ws + p.off_zero;
  uint32_t* lbar = reinterpret_cast<uint32_t*>(z);
  z += align_up((size_t)S * sizeof(uint32_t), 256);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(z);
  z += align_up((size_t)S * kBins * sizeof(uint32_t), 256);
  uint32_t* lhist = reinterpret_cast<uint32_t*>(z);
  z += align_up((size_t)S * 3 * kBins * sizeof(uint32_t), 256);
  uint32_t* hcnt = reinterpret_cast<uint32_t*>(z);
  int32_t* upos = reinterpret_cast<int32_t*>(ws + p.off_union);
  uint32_t* ukey = reinterpret_cast<uint32_t*>(
      ws + p.off_union + align_up((size_t)S * nch * UC * sizeof(int32_t), 256));
  // barriers, histograms and counts start at zero
  cudaError_t e = cudaMemsetAsync(ws + p.off_zero, 0, p.off_union - p.off_zero, st);
  if (e != cudaSuccess) return e;
  // the sweeps' rings are dynamic shared memory above 48 KB: opted in once per device
  static std::atomic<int> opted[kMaxDevices];
  const int ok = per_device(opted, []() {
    const void* ks[3] = {(const void*)alloc_sweep1<true>, (const void*)alloc_sweep1<false>,
                         (const void*)alloc_sweep2};
    for (const void* k : ks)
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes) !=
          cudaSuccess)
        return 0;
    return 1;
  });
  if (!ok) return cudaErrorInvalidConfiguration;
  const dim3 sweep((unsigned)nch, (unsigned)S);
  if (entropy_mode)
    alloc_sweep1<true><<<sweep, kThreads, kRingBytes, st>>>(scores, N, nch, part, ghist, hdr);
  else
    alloc_sweep1<false><<<sweep, kThreads, kRingBytes, st>>>(scores, N, nch, part, ghist, hdr);
  alloc_bound<<<(unsigned)S, kThreads, 0, st>>>(part, nch, s.L, s.Hkv, s.n, s.w, C, budget,
                                                entropy_mode, layer_cap, layer_budget, bprime,
                                                ghist, gbin, hdr);
  count_launches(2);
  // sweep 2 is a cooperative launch (the CTAs of a layer wait for one another), over as many
  // layers at a time as can be resident
  const int64_t per_launch = sweep2_resident() / nch > 0 ? sweep2_resident() / nch : 1;
  for (int64_t s0 = 0; s0 < S; s0 += per_launch) {
    const int64_t sb = S - s0 < per_launch ? S - s0 : per_launch;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)nch, (unsigned)sb);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kRingBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, alloc_sweep2, scores, s.Hkv, C, nch, s0,
                           (const uint32_t*)gbin, (const int64_t*)bprime, upos, ukey, UC, lhist,
                           hcnt, lbar, s.w, an, ad, head_budget, hdr);
    if (e != cudaSuccess) return e;
    count_launches(1);
  }
  return cudaGetLastError();
}

// Per-layer sums of the head budgets of a model-wide selection (one thread per segment).
__global__ void layer_sums(const int32_t* __restrict__ head_budget, int64_t segments, int Hkv,
                           int32_t* __restrict__ layer_budget) {
  const int64_t seg = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (seg >= segments) return;
  int64_t t = 0;
  for (int g = 0; g < Hkv; ++g) t += head_budget[seg * Hkv + g];
  layer_budget[seg] = (int32_t)t;
}

cudaError_t launch_layer_sums(const int32_t* head_budget, int64_t segments, int Hkv,
                              int32_t* layer_budget, cudaStream_t st) {
  if (segments <= 0) return cudaSuccess;
  layer_sums<<<(unsigned)cdiv(segments, (int64_t)256), 256, 0, st>>>(head_budget, segments, Hkv,
                                                                     layer_budget);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace kv
