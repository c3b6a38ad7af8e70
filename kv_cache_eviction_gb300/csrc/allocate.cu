// Per-head budgets of every (sequence, layer).
//
// Ada-KV Algorithm 1: concatenate the heads' scores, take the layer-wide top B', count how
// many of them each head owns (f_g).  Ada-KV Algorithm 2, safeguard: blend f_g with the
// uniform share B'/Hkv, exact integers, alpha on the uniform side.  LAVa, uncertainty-based
// layer budgets: each layer's share of the sequence's total is proportional to the entropy
// of its normalised scores.
//
// The layer-wide top-B' is a radix select on the fp32 bit patterns (no sort): three
// passes of 11/11/10 bits, each a histogram over every layer at once (many CTAs per layer,
// shared-memory counts merged into per-layer global bins), then a sweep that counts, per
// head, the keys above the threshold and the keys equal to it.  Each sweep is one wave of
// CTAs reading 16-byte vectors; the last CTA of a layer to finish picks the digit of the
// pass (or, after the count, blends the head budgets), so no launch is spent on per-layer
// bookkeeping.  Consecutive sweeps walk their chunks in opposite directions, so each one
// starts on the part of the scores the previous one left in L2.
#include "kv_internal.cuh"

namespace kv {

namespace {
constexpr int kThreads = 256;
constexpr int kMinBlocks = 6;    // resident CTAs per SM the sweeps are sized for
constexpr int kU = 4;            // 16-byte loads in flight per thread per step
constexpr int kBins = 2048;
constexpr int kMaxHeads = 256;

struct RadixState {          // one per (sequence, layer)
  uint32_t prefix, mask;     // resolved high bits of the threshold key
  uint32_t krem;             // keys still to take from the current prefix class
  uint32_t active;           // 0 when B' == 0 (nothing to select)
};

__device__ __forceinline__ int pass_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__device__ __forceinline__ int pass_bins(int pass) { return pass == 2 ? 1024 : 2048; }

// Visits the keys x[i0, i1): fn(value, ok, i) is called the same number of times by every
// thread of the block (warp votes inside fn stay convergent); ok is false for padding, i is
// the key's index.  The
// 16-byte aligned middle is read as float4, kU vectors in flight per thread; `rev` walks
// the steps from the end of the range.
template <typename Fn>
__device__ __forceinline__ void sweep_keys(const float* __restrict__ x, int64_t i0, int64_t i1,
                                           bool rev, Fn&& fn) {
  const uintptr_t addr = reinterpret_cast<uintptr_t>(x + i0);
  int64_t a = i0 + (int64_t)(((16u - (uint32_t)(addr & 15u)) & 15u) >> 2);
  if (a > i1) a = i1;
  const int64_t nv = (i1 - a) >> 2;
  const int64_t b = a + nv * 4;
  {
    const int64_t ih = i0 + threadIdx.x, it = b + threadIdx.x;
    const bool okh = ih < a, okt = it < i1;
    const float xh = okh ? x[ih] : 0.0f, xt = okt ? x[it] : 0.0f;
    fn(xh, okh, ih);
    fn(xt, okt, it);
  }
  const float4* xv = reinterpret_cast<const float4*>(x + a);
  const int64_t step = (int64_t)kU * blockDim.x;
  const int64_t nsteps = cdiv(nv, step);
  for (int64_t s = 0; s < nsteps; ++s) {
    const int64_t base = (rev ? nsteps - 1 - s : s) * step + threadIdx.x;
    float4 v[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int64_t j = base + (int64_t)k * blockDim.x;
      v[k] = j < nv ? xv[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int64_t j = base + (int64_t)k * blockDim.x;
      const bool ok = j < nv;
      const int64_t i = a + 4 * j;
      fn(v[k].x, ok, i);
      fn(v[k].y, ok, i + 1);
      fn(v[k].z, ok, i + 2);
      fn(v[k].w, ok, i + 3);
    }
  }
}

// Keys per CTA of a layer: a multiple of 4, so the chunks of an aligned layer are aligned.
__device__ __forceinline__ int64_t chunk_len(int64_t N, int nch) {
  return cdiv(cdiv(N, nch), 4) * 4;
}

// True in every thread of the CTA that is the n-th and last of its layer to get here; its
// reads of the other CTAs' atomics come after a fence.  The counter is left at zero.
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

// The digit of pass `pass` that holds the krem-th largest key of the layer (bins counted
// from the top) and krem's rank inside it; G is the layer's global histogram, which is
// cleared for the next pass.  All threads call it; scr holds >= 34 words.
__device__ void pick_digit(uint32_t* G, int pass, uint32_t krem, uint32_t* scr, WsHeader* hdr,
                           unsigned seg, uint32_t& bin_out, uint32_t& kr_out) {
  const int nb = pass_bins(pass);
  const int per = nb / (int)blockDim.x;   // 8 or 4
  uint32_t c[kBins / kThreads];
  uint32_t local = 0;
#pragma unroll
  for (int q = 0; q < kBins / kThreads; ++q) {
    c[q] = q < per ? __ldcg(G + nb - 1 - ((int)threadIdx.x * per + q)) : 0u;
    local += c[q];
  }
  if (threadIdx.x == 0) { scr[32] = 0u; scr[33] = 0u; }
  uint32_t total;
  const uint32_t incl = block_incl_scan(local, scr, &total);   // ends with a barrier
  const uint32_t excl = incl - local;
  if (excl < krem && krem <= incl) {
    uint32_t acc = excl;
#pragma unroll
    for (int q = 0; q < kBins / kThreads; ++q) {
      if (q < per && acc < krem) {
        if (acc + c[q] >= krem) {
          scr[32] = (uint32_t)(nb - 1 - ((int)threadIdx.x * per + q));
          scr[33] = krem - acc;
        }
        acc += c[q];
      }
    }
  }
  if (threadIdx.x == 0 && krem > total) raise_dev(hdr, DEV_SELECT, seg);
  for (int i = threadIdx.x; i < nb; i += blockDim.x) G[i] = 0u;
  __syncthreads();
  bin_out = scr[32];
  kr_out = scr[33];
  __syncthreads();
}

__device__ __forceinline__ void advance(RadixState& r, int pass, uint32_t bin, uint32_t kr) {
  r.prefix |= bin << pass_shift(pass);
  r.mask |= (uint32_t)(pass_bins(pass) - 1) << pass_shift(pass);
  r.krem = kr;
}

__device__ __forceinline__ void merge_hist(const uint32_t* hist, uint32_t* G, int nb) {
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    const uint32_t c = hist[i];
    if (c) atomicAdd(&G[i], c);
  }
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

// LAVa entropy mode, first sweep: the first digit's histogram (it does not depend on B', so
// it is taken before the layer budgets exist) and per-CTA partial sums of s and s*ln(s)
// (float terms, float runs of 16 added into fp64).
__global__ void __launch_bounds__(kThreads, kMinBlocks)
entropy_hist(const float* __restrict__ scores, int64_t N, int nch, double2* __restrict__ part,
             uint32_t* __restrict__ ghist) {
  __shared__ uint32_t hist[kBins];
  __shared__ double sa[kThreads / 32], sb[kThreads / 32];
  const int64_t seg = blockIdx.y;
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0u;
  __syncthreads();
  const int64_t per = chunk_len(N, nch);
  const int64_t i0 = min(N, blockIdx.x * per), i1 = min(N, i0 + per);
  double a = 0.0, b = 0.0;
  float ra = 0.f, rb = 0.f;
  int terms = 0;
  sweep_keys(scores + seg * N, i0, i1, false, [&](float x, bool ok, int64_t) {
    hist_add_runs(hist, ok ? (score_key(x) >> 21) : 0xFFFFFFFFu);
    if (ok && x > 0.0f) {
      ra += x;
      rb += x * (__log2f(x) * 0.69314718055994531f);
    }
    if (++terms == 16) {
      a += (double)ra;
      b += (double)rb;
      ra = rb = 0.f;
      terms = 0;
    }
  });
  a += (double)ra;
  b += (double)rb;
  a = warp_sum_d(a);
  b = warp_sum_d(b);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sa[warp] = a; sb[warp] = b; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double ta = 0.0, tb = 0.0;
    for (int i = 0; i < kThreads / 32; ++i) { ta += sa[i]; tb += sb[i]; }
    part[seg * nch + blockIdx.x] = make_double2(ta, tb);
  }
  merge_hist(hist, ghist + seg * kBins, kBins);
}

// One CTA per (sequence, layer): e_l of every layer of the sequence, the capped
// proportional split of R = total - L*w*Hkv with floors and largest remainders (ties to the
// lower layer), then this layer's first digit from the histogram of the entropy sweep.  The
// split is the same in every CTA of a sequence (same inputs, same order); each thread owns
// the layers l = tid (mod blockDim), sums over the active layers are block reductions and
// the largest remainders are ranks every thread counts for its own layers.
constexpr int kMaxLayers = 1024;
__global__ void __launch_bounds__(kThreads)
layer_budgets(const double2* __restrict__ part, int nch, int L, int Hkv, int n, int w, int C,
              const int64_t* __restrict__ total, int32_t* __restrict__ layer_budget,
              int64_t* __restrict__ bprime, RadixState* __restrict__ st,
              uint32_t* __restrict__ ghist, WsHeader* hdr) {
  __shared__ double e[kMaxLayers], frac[kMaxLayers];
  __shared__ int64_t sel[kMaxLayers];   // -1: active; >= 0: capped at that value
  __shared__ double red_d[kThreads / 32];
  __shared__ long long red_i[kThreads / 32];
  __shared__ uint32_t scr[34];
  __shared__ int64_t mine;
  const int64_t seg = blockIdx.x;
  const int b = (int)(seg / L), lme = (int)(seg - (int64_t)b * L);
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
    e[l] = el > 0.0 ? el : 0.0;
    sel[l] = -1;
  }
  const int64_t cap = (int64_t)Hkv * C;
  int64_t R = total[b] - (int64_t)L * w * Hkv;
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
      if (sel[l] < 0) { es += e[l]; ++na; }
    const double esum = block_sum_dbl(es, red_d);
    const long long active = block_sum_ll(na, red_i);
    long long nover = 0;
    for (int l = threadIdx.x; l < L; l += blockDim.x) {
      if (sel[l] >= 0) continue;
      const double q = esum > 0.0 ? (double)rem * e[l] / esum : (double)rem / (double)active;
      frac[l] = q;
      if (q > (double)cap) ++nover;
    }
    nover = block_sum_ll(nover, red_i);
    if (nover == 0 || active == 0) break;
    for (int l = threadIdx.x; l < L; l += blockDim.x)
      if (sel[l] < 0 && frac[l] > (double)cap) sel[l] = cap;
    rem -= (int64_t)nover * cap;
  }
  long long used = 0;
  for (int l = threadIdx.x; l < L; l += blockDim.x) {
    if (sel[l] >= 0) continue;
    const double f = floor(frac[l]);
    frac[l] -= f;                  // keep only the fractional part
    sel[l] = -2 - (int64_t)f;      // active: the floor is stored as -2 - floor
    used += (long long)f;
  }
  const int64_t left = rem - (int64_t)block_sum_ll(used, red_i);   // also a barrier
  // largest remainders: an active layer gets one more unit when fewer than `left` active
  // layers precede it in (fraction desc, layer asc) order
  if (lme % blockDim.x == threadIdx.x) {
    int64_t v = sel[lme];
    if (v <= -2) {
      const double fl = frac[lme];
      int64_t before = 0;
      for (int m = 0; m < L; ++m)
        if (sel[m] <= -2 && (frac[m] > fl || (frac[m] == fl && m < lme))) ++before;
      v = (-2 - v) + (before < left ? 1 : 0);
    }
    bprime[seg] = v;
    layer_budget[seg] = (int32_t)(v + (int64_t)w * Hkv);
    mine = v;
  }
  __syncthreads();
  const int64_t Bp = mine;
  RadixState r{0u, 0u, (uint32_t)Bp, Bp > 0 ? 1u : 0u};
  uint32_t bin, kr;
  pick_digit(ghist + seg * kBins, 0, r.krem, scr, hdr, (unsigned)seg, bin, kr);
  if (threadIdx.x == 0) {
    if (r.active) advance(r, 0, bin, kr);
    st[seg] = r;
  }
}

// Histogram of the pass's digit over the keys that match the resolved prefix; the last CTA
// of the layer picks the digit.  Pass 0 without the entropy sweep also takes B' from the
// per-layer budget (range-checked) and sets up the layer's state.
__global__ void __launch_bounds__(kThreads, kMinBlocks)
radix_hist(const float* __restrict__ scores, int64_t N, int nch, int pass,
           const int64_t* __restrict__ budget, int Hkv, int w, int32_t* __restrict__ layer_budget,
           int64_t* __restrict__ bprime, RadixState* __restrict__ st,
           uint32_t* __restrict__ ghist, uint32_t* __restrict__ done, WsHeader* hdr) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t scr[34];
  __shared__ uint32_t flag;
  const int64_t seg = blockIdx.y;
  RadixState r{0u, 0u, 0u, 1u};
  if (pass > 0) {
    r = st[seg];
    if (!r.active) return;   // no CTA of this layer takes part
  }
  const int sh = pass_shift(pass), nb = pass_bins(pass);
  for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0u;
  __syncthreads();
  const int64_t per = chunk_len(N, nch);
  const int64_t i0 = min(N, blockIdx.x * per), i1 = min(N, i0 + per);
  sweep_keys(scores + seg * N, i0, i1, (pass & 1) != 0, [&](float x, bool ok, int64_t) {
    uint32_t bin = 0xFFFFFFFFu;
    if (ok) {
      const uint32_t key = score_key(x);
      if ((key & r.mask) == r.prefix) bin = (key >> sh) & (uint32_t)(nb - 1);
    }
    hist_add_runs(hist, bin);
  });
  __syncthreads();
  uint32_t* G = ghist + seg * kBins;
  merge_hist(hist, G, nb);
  if (!last_of_layer(done + seg, (uint32_t)nch, &flag)) return;
  if (pass == 0) {
    int64_t Bp = budget[seg] - (int64_t)w * Hkv;
    if (Bp < 0 || Bp > N) {
      if (threadIdx.x == 0) raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)seg);
      Bp = Bp < 0 ? 0 : N;
    }
    r.krem = (uint32_t)Bp;
    r.active = Bp > 0 ? 1u : 0u;
    if (threadIdx.x == 0) {
      bprime[seg] = Bp;
      layer_budget[seg] = (int32_t)(Bp + (int64_t)w * Hkv);
    }
  }
  uint32_t bin, kr;
  pick_digit(G, pass, r.krem, scr, hdr, (unsigned)seg, bin, kr);
  if (threadIdx.x == 0) {
    if (r.active) advance(r, pass, bin, kr);
    st[seg] = r;
  }
}

// Thread 0 of the last CTA of a layer: f_g from the per-head counts (tau-equal keys in head
// order), each head's floor of the blend in sBg and its remainder in srem; returns the units
// left for the largest remainders.  The counts are left zeroed for the next call.
__device__ __noinline__ int64_t blend_floors(int64_t left_eq, uint32_t* Cg, int Hkv, int64_t Bp,
                                             uint32_t an, uint32_t ad, int32_t* sBg,
                                             int64_t* srem, WsHeader* hdr, unsigned seg) {
  const int64_t den = (int64_t)ad * Hkv;
  int64_t fsum = 0, flo = 0;
  for (int g = 0; g < Hkv; ++g) {
    const int64_t eqg = __ldcg(Cg + 2 * g + 1);
    const int64_t take = left_eq < eqg ? left_eq : eqg;
    left_eq -= take;
    const int64_t f = (int64_t)__ldcg(Cg + 2 * g) + take;
    Cg[2 * g] = 0u;
    Cg[2 * g + 1] = 0u;
    fsum += f;
    const int64_t X = (int64_t)an * Bp + (int64_t)(ad - an) * Hkv * f;
    sBg[g] = (int32_t)(X / den);
    srem[g] = X % den;
    flo += sBg[g];
  }
  if (fsum != Bp) raise_dev(hdr, DEV_SELECT, seg);
  return Bp - flo;
}

// Per-head counts of keys above the threshold and equal to it; the last CTA of the layer
// then forms f_g (keys above tau in head g, plus tau-equal keys in (head, position) order)
// and the safeguard blend in exact integers.
__global__ void __launch_bounds__(kThreads, kMinBlocks)
radix_count(const float* __restrict__ scores, int Hkv, int C, int nch,
            const RadixState* __restrict__ st, const int64_t* __restrict__ bprime,
            uint32_t* __restrict__ counts /*[S][Hkv][2]*/, uint32_t* __restrict__ done, int w,
            uint32_t an, uint32_t ad, int32_t* __restrict__ head_budget, WsHeader* hdr) {
  __shared__ uint32_t cnt[2 * kMaxHeads];
  __shared__ int64_t srem[kMaxHeads];
  __shared__ int32_t sBg[kMaxHeads];
  __shared__ int64_t sleft;
  __shared__ uint32_t flag;
  const int64_t seg = blockIdx.y;
  const RadixState r = st[seg];
  const int64_t N = (int64_t)Hkv * C;
  uint32_t* Cg = counts + seg * 2 * Hkv;
  if (r.active) {
    const uint32_t tau = r.prefix;
    for (int i = threadIdx.x; i < 2 * Hkv; i += blockDim.x) cnt[i] = 0u;
    __syncthreads();
    const int64_t per = chunk_len(N, nch);
    const int64_t i0 = min(N, blockIdx.x * per), i1 = min(N, i0 + per);
    // one sub-sweep per head the chunk meets (walked from the last, like the steps)
    const float* S = scores + seg * N;
    if (i1 > i0) {
      const int h0 = (int)(i0 / C), h1 = (int)((i1 - 1) / C);
      for (int h = h1; h >= h0; --h) {
        const int64_t a = max(i0, (int64_t)h * C), b = min(i1, (int64_t)(h + 1) * C);
        uint32_t gt = 0, eq = 0;
        sweep_keys(S, a, b, true, [&](float x, bool ok, int64_t) {
          const uint32_t key = score_key(x);
          gt += (ok && key > tau) ? 1u : 0u;
          eq += (ok && key == tau) ? 1u : 0u;
        });
        gt = warp_sum_u(gt);
        eq = warp_sum_u(eq);
        if ((threadIdx.x & 31) == 0) {
          if (gt) atomicAdd(&cnt[2 * h], gt);
          if (eq) atomicAdd(&cnt[2 * h + 1], eq);
        }
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * Hkv; i += blockDim.x)
      if (cnt[i]) atomicAdd(&Cg[i], cnt[i]);
  }
  if (!last_of_layer(done + seg, (uint32_t)nch, &flag)) return;
  const int64_t Bp = bprime[seg];
  if (threadIdx.x == 0)
    sleft = blend_floors(r.active ? (int64_t)r.krem : 0, Cg, Hkv, Bp, an, ad, sBg, srem, hdr,
                         (unsigned)seg);
  __syncthreads();
  // largest remainders (ties to the lower head): a head gets one more unit when fewer than
  // `left` heads precede it in (remainder desc, head asc) order
  for (int g = threadIdx.x; g < Hkv; g += blockDim.x) {
    const int64_t rg = srem[g];
    int64_t before = 0;
    for (int m = 0; m < Hkv; ++m)
      if (srem[m] > rg || (srem[m] == rg && m < g)) ++before;
    head_budget[seg * Hkv + g] = sBg[g] + (before < sleft ? 1 : 0) + w;
  }
}

AllocPlan alloc_plan(const Shape& s) {
  AllocPlan p{};
  const int64_t S = s.segments();
  const int64_t N = (int64_t)s.Hkv * (s.C() > 0 ? s.C() : 1);
  // one wave of kMinBlocks CTAs per SM over all layers, at least one full step per CTA
  int64_t nch = (int64_t)num_sms() * kMinBlocks / (S > 0 ? S : 1);
  const int64_t maxch = cdiv(N, (int64_t)kU * 4 * kThreads);
  if (nch > maxch) nch = maxch;
  if (nch < 1) nch = 1;
  p.nchunkE = (int)nch;
  size_t off = kWsHeader;
  p.off_bprime = off;
  off += align_up((size_t)S * sizeof(int64_t), 256);
  p.off_epart = off;
  off += align_up((size_t)S * p.nchunkE * sizeof(double2), 256);
  p.off_e = off;
  off += align_up((size_t)S * sizeof(uint32_t), 256);
  p.off_scratch = off;   // radix state, histograms, per-head counts
  off += align_up((size_t)S * sizeof(RadixState), 256);
  off += align_up((size_t)S * kBins * sizeof(uint32_t), 256);
  off += align_up((size_t)S * 2 * kMaxHeads * sizeof(uint32_t), 256);
  p.off_end = off;
  return p;
}

cudaError_t launch_allocate(const Shape& s, const float* scores, const int64_t* budget,
                            int entropy_mode, uint32_t an, uint32_t ad, int32_t* layer_budget,
                            int32_t* head_budget, char* ws, const AllocPlan& p,
                            cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t S = s.segments();
  const int C = s.C();
  const int64_t N = (int64_t)s.Hkv * C;
  int64_t* bprime = reinterpret_cast<int64_t*>(ws + p.off_bprime);
  uint32_t* done = reinterpret_cast<uint32_t*>(ws + p.off_e);
  char* sc = ws + p.off_scratch;
  RadixState* rst = reinterpret_cast<RadixState*>(sc);
  sc += align_up((size_t)S * sizeof(RadixState), 256);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(sc);
  sc += align_up((size_t)S * kBins * sizeof(uint32_t), 256);
  uint32_t* counts = reinterpret_cast<uint32_t*>(sc);
  // counters, histograms and counts start at zero; the kernels leave them zeroed behind them
  cudaError_t e = cudaMemsetAsync(done, 0, p.off_end - p.off_e, st);
  if (e != cudaSuccess) return e;
  const int nch = p.nchunkE;
  const dim3 sweep((unsigned)nch, (unsigned)S);
  if (entropy_mode) {
    double2* part = reinterpret_cast<double2*>(ws + p.off_epart);
    entropy_hist<<<sweep, kThreads, 0, st>>>(scores, N, nch, part, ghist);
    layer_budgets<<<(unsigned)S, kThreads, 0, st>>>(part, nch, s.L, s.Hkv, s.n, s.w, C, budget,
                                                    layer_budget, bprime, rst, ghist, hdr);
    count_launches(2);
  } else {
    radix_hist<<<sweep, kThreads, 0, st>>>(scores, N, nch, 0, budget, s.Hkv, s.w, layer_budget,
                                           bprime, rst, ghist, done, hdr);
    count_launches(1);
  }
  for (int pass = 1; pass < 3; ++pass)
    radix_hist<<<sweep, kThreads, 0, st>>>(scores, N, nch, pass, budget, s.Hkv, s.w,
                                           layer_budget, bprime, rst, ghist, done, hdr);
  radix_count<<<sweep, kThreads, 0, st>>>(scores, s.Hkv, C, nch, rst, bprime, counts, done, s.w,
                                          an, ad, head_budget, hdr);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace kv
