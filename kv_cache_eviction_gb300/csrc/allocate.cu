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
// shared-memory counts merged into per-layer global bins) followed by a
// small kernel that picks the digit holding the B'-th largest key.  A last pass counts,
// per head, the keys above the threshold and the keys equal to it.
#include "kv_internal.cuh"

namespace kv {

namespace {
constexpr int kThreads = 256;
constexpr int kBins = 2048;
constexpr int kMaxHeads = 256;

struct RadixState {          // one per (sequence, layer)
  uint32_t prefix, mask;     // resolved high bits of the threshold key
  uint32_t krem;             // keys still to take from the current prefix class
  uint32_t active;           // 0 when B' == 0 (nothing to select)
};

__device__ __forceinline__ int pass_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__device__ __forceinline__ int pass_bins(int pass) { return pass == 2 ? 1024 : 2048; }
}  // namespace

// LAVa entropy mode: the first histogram sweep also forms the per-chunk partial sums of s
// and s*ln(s) (float terms, float runs of 64 added into fp64).  The first digit's
// histogram does not depend on B', so it can be taken before the layer budgets exist.
__global__ void __launch_bounds__(kThreads)
entropy_hist(const float* __restrict__ scores, int64_t N, int nch, double2* __restrict__ part,
             uint32_t* __restrict__ ghist) {
  __shared__ uint32_t hist[kBins];
  __shared__ double sa[kThreads / 32], sb[kThreads / 32];
  const int64_t seg = blockIdx.y;
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0u;
  __syncthreads();
  const int64_t per = cdiv(N, nch);
  const int64_t i0 = blockIdx.x * per, i1 = min(N, i0 + per);
  const float* S = scores + seg * N;
  // 8 keys per thread per step, all loaded before any is used (latency hiding); the step
  // count is the same for every lane so the warp votes stay convergent
  constexpr int U = 8;
  const int64_t step = (int64_t)U * blockDim.x;
  double a = 0.0, b = 0.0;
  float ra = 0.f, rb = 0.f;
  for (int64_t base = i0; base < i1; base += step) {
    float x[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t i = base + (int64_t)k * blockDim.x + threadIdx.x;
      x[k] = i < i1 ? S[i] : -1.0f;   // -1: no key
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      hist_add_runs(hist, x[k] >= 0.0f ? (score_key(x[k]) >> 21) : 0xFFFFFFFFu);
      if (x[k] > 0.0f) {
        ra += x[k];
        rb += x[k] * (__log2f(x[k]) * 0.69314718055994531f);
      }
    }
    a += (double)ra;
    b += (double)rb;
    ra = rb = 0.f;
  }
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
  uint32_t* G = ghist + seg * kBins;
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (hist[i]) atomicAdd(&G[i], hist[i]);
}

// One CTA per sequence: e_l for every layer in parallel, then the capped proportional split
// of R = total - L*w*Hkv with floors and largest remainders (ties to the lower layer).  The
// split works on shared-memory copies (L <= kMaxLayers).
constexpr int kMaxLayers = 1024;
__global__ void __launch_bounds__(kThreads)
layer_budgets(const double2* __restrict__ part, int nch, int L, int Hkv, int n, int w, int C,
              const int64_t* __restrict__ total, int32_t* __restrict__ layer_budget,
              int64_t* __restrict__ bprime, WsHeader* hdr) {
  __shared__ double e[kMaxLayers], quota[kMaxLayers];
  __shared__ int64_t sel[kMaxLayers];
  const int b = blockIdx.x;
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
    sel[l] = -1;                    // -1: active (not yet capped)
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t cap = (int64_t)Hkv * C;
    int64_t R = total[b] - (int64_t)L * w * Hkv;
    if (R < 0 || R > (int64_t)L * cap) {
      raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)b);
      R = R < 0 ? 0 : (int64_t)L * cap;
    }
    int64_t rem = R;
    int active = L;
    for (;;) {
      double esum = 0.0;
      for (int l = 0; l < L; ++l) if (sel[l] < 0) esum += e[l];
      bool any_over = false;
      for (int l = 0; l < L; ++l) {
        if (sel[l] >= 0) continue;
        quota[l] = esum > 0.0 ? (double)rem * e[l] / esum : (double)rem / (double)active;
        if (quota[l] > (double)cap) any_over = true;
      }
      if (!any_over || active == 0) break;
      for (int l = 0; l < L; ++l) {
        if (sel[l] < 0 && quota[l] > (double)cap) {
          sel[l] = cap;
          rem -= cap;
          --active;
        }
      }
    }
    int64_t used = 0;
    for (int l = 0; l < L; ++l) {
      if (sel[l] >= 0) continue;
      const double f = floor(quota[l]);
      quota[l] -= f;                // keep only the fractional part
      sel[l] = -2 - (int64_t)f;     // still active: the floor is stored as -2 - floor
      used += (int64_t)f;
    }
    for (int64_t left = rem - used; left > 0; --left) {
      int best = -1;
      for (int l = 0; l < L; ++l) {
        if (sel[l] > -2) continue;  // capped or already given its extra unit
        if (best < 0 || quota[l] > quota[best]) best = l;
      }
      if (best < 0) break;
      sel[best] = (-2 - sel[best]) + 1;
    }
    for (int l = 0; l < L; ++l)
      if (sel[l] <= -2) sel[l] = -2 - sel[l];
  }
  __syncthreads();
  for (int l = threadIdx.x; l < L; l += blockDim.x) {
    bprime[(int64_t)b * L + l] = sel[l];
    layer_budget[(int64_t)b * L + l] = (int32_t)(sel[l] + (int64_t)w * Hkv);
  }
}

// B' of every (sequence, layer) and the initial radix state.
__global__ void radix_init(const int64_t* __restrict__ budget, const int64_t* __restrict__ bprime_in,
                           int64_t S, int Hkv, int C, int w, int32_t* __restrict__ layer_budget,
                           int64_t* __restrict__ bprime, RadixState* __restrict__ st,
                           WsHeader* hdr) {
  const int64_t seg = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (seg >= S) return;
  const int64_t N = (int64_t)Hkv * C;
  int64_t Bp;
  if (bprime_in) {
    Bp = bprime_in[seg];
  } else {
    Bp = budget[seg] - (int64_t)w * Hkv;
    if (Bp < 0 || Bp > N) {
      raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)seg);
      Bp = Bp < 0 ? 0 : N;
    }
    layer_budget[seg] = (int32_t)(Bp + (int64_t)w * Hkv);
  }
  bprime[seg] = Bp;
  RadixState r;
  r.prefix = 0;
  r.mask = 0;
  r.krem = (uint32_t)Bp;
  r.active = Bp > 0 ? 1u : 0u;
  st[seg] = r;
}

// Histogram of the current digit over the keys that match the resolved prefix.
__global__ void __launch_bounds__(kThreads)
radix_hist(const float* __restrict__ scores, int64_t N, int nch, const RadixState* __restrict__ st,
           uint32_t* __restrict__ ghist, int pass) {
  __shared__ uint32_t hist[kBins];
  const int64_t seg = blockIdx.y;
  const RadixState r = st[seg];
  if (!r.active) return;
  const int sh = pass_shift(pass), nb = pass_bins(pass);
  for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0u;
  __syncthreads();
  const int64_t per = cdiv(N, nch);
  const int64_t i0 = blockIdx.x * per, i1 = min(N, i0 + per);
  const float* S = scores + seg * N;
  // 8 keys per thread per step, loaded before use; uniform step count (convergent votes)
  constexpr int U = 8;
  const int64_t step = (int64_t)U * blockDim.x;
  for (int64_t base = i0; base < i1; base += step) {
    float x[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t i = base + (int64_t)k * blockDim.x + threadIdx.x;
      x[k] = i < i1 ? S[i] : -1.0f;
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      uint32_t bin = 0xFFFFFFFFu;
      if (x[k] >= 0.0f) {
        const uint32_t key = score_key(x[k]);
        if ((key & r.mask) == r.prefix) bin = (key >> sh) & (uint32_t)(nb - 1);
      }
      hist_add_runs(hist, bin);
    }
  }
  __syncthreads();
  uint32_t* G = ghist + seg * kBins;
  for (int i = threadIdx.x; i < nb; i += blockDim.x)
    if (hist[i]) atomicAdd(&G[i], hist[i]);
}

// One CTA per (sequence, layer): picks the digit that holds the krem-th largest key and
// clears the histogram for the next pass.
__global__ void __launch_bounds__(1024)
radix_pick(RadixState* __restrict__ st, uint32_t* __restrict__ ghist, int pass) {
  __shared__ uint32_t scratch[32];
  __shared__ uint32_t res[2];
  const int64_t seg = blockIdx.x;
  RadixState r = st[seg];
  uint32_t* G = ghist + seg * kBins;
  const int nb = pass_bins(pass), sh = pass_shift(pass);
  if (!r.active) {
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) G[i] = 0u;
    return;
  }
  const int per = nb / (int)blockDim.x;   // bins per thread, counted from the top
  uint32_t local = 0;
  for (int q = 0; q < per; ++q) local += G[nb - 1 - (threadIdx.x * per + q)];
  uint32_t total;
  const uint32_t incl = block_incl_scan(local, scratch, &total);
  const uint32_t excl = incl - local;
  if (excl < r.krem && r.krem <= incl) {
    uint32_t acc = excl;
    for (int q = 0; q < per; ++q) {
      const int bin = nb - 1 - (threadIdx.x * per + q);
      const uint32_t c = G[bin];
      if (acc + c >= r.krem) {
        res[0] = (uint32_t)bin;
        res[1] = r.krem - acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) G[i] = 0u;
  if (threadIdx.x == 0) {
    r.prefix |= res[0] << sh;
    r.mask |= (uint32_t)(nb - 1) << sh;
    r.krem = res[1];
    st[seg] = r;
  }
}

// Per-head counts of keys above the threshold and equal to it.
__global__ void __launch_bounds__(kThreads)
radix_count(const float* __restrict__ scores, int Hkv, int C, int nch,
            const RadixState* __restrict__ st, uint32_t* __restrict__ counts /*[S][Hkv][2]*/) {
  __shared__ uint32_t cnt[2 * kMaxHeads];
  const int64_t seg = blockIdx.y;
  const RadixState r = st[seg];
  if (!r.active) return;
  const int64_t N = (int64_t)Hkv * C;
  const uint32_t tau = r.prefix;
  for (int i = threadIdx.x; i < 2 * Hkv; i += blockDim.x) cnt[i] = 0u;
  __syncthreads();
  const int64_t per = cdiv(N, nch);
  const int64_t i0 = blockIdx.x * per, i1 = min(N, i0 + per);
  const float* S = scores + seg * N;
  // coalesced sweep, 8 keys per thread per step loaded before use; a thread's keys
  // advance by blockDim, so its head changes rarely
  constexpr int U = 8;
  const int64_t step = (int64_t)U * blockDim.x;
  int head = -1;
  int64_t next = 0;   // first key index of the next head
  uint32_t gt = 0, eq = 0;
  for (int64_t base = i0; base < i1; base += step) {
    float x[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t i = base + (int64_t)k * blockDim.x + threadIdx.x;
      x[k] = i < i1 ? S[i] : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t i = base + (int64_t)k * blockDim.x + threadIdx.x;
      if (i >= i1) break;
      if (i >= next) {
        if (head >= 0) {
          if (gt) atomicAdd(&cnt[2 * head], gt);
          if (eq) atomicAdd(&cnt[2 * head + 1], eq);
        }
        head = (int)(i / C);
        next = (int64_t)(head + 1) * C;
        gt = eq = 0;
      }
      const uint32_t key = score_key(x[k]);
      gt += key > tau;
      eq += key == tau;
    }
  }
  if (head >= 0) {
    if (gt) atomicAdd(&cnt[2 * head], gt);
    if (eq) atomicAdd(&cnt[2 * head + 1], eq);
  }
  __syncthreads();
  uint32_t* Cg = counts + seg * 2 * Hkv;
  for (int i = threadIdx.x; i < 2 * Hkv; i += blockDim.x)
    if (cnt[i]) atomicAdd(&Cg[i], cnt[i]);
}

// f_g = keys above tau in head g, plus tau-equal keys in (head, position) order; then the
// safeguard blend in exact integers.  One thread per (sequence, layer).
__global__ void alloc_blend(const RadixState* __restrict__ st, const int64_t* __restrict__ bprime,
                            uint32_t* __restrict__ counts, int64_t S, int Hkv, int C, int w,
                            uint32_t an, uint32_t ad, int32_t* __restrict__ head_budget,
                            WsHeader* hdr) {
  const int64_t seg = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (seg >= S) return;
  const RadixState r = st[seg];
  const int64_t Bp = bprime[seg];
  uint32_t* Cg = counts + seg * 2 * Hkv;
  const int64_t den = (int64_t)ad * Hkv;
  int64_t left_eq = r.active ? (int64_t)r.krem : 0, fsum = 0, flo = 0;
  int64_t rem[kMaxHeads];
  int32_t Bg[kMaxHeads];
  for (int g = 0; g < Hkv; ++g) {
    int64_t f = 0;
    if (r.active) {
      const int64_t eqg = Cg[2 * g + 1];
      int64_t take = left_eq < eqg ? left_eq : eqg;
      left_eq -= take;
      f = (int64_t)Cg[2 * g] + take;
    }
    Cg[2 * g] = 0u;          // counts are left zeroed for the next call
    Cg[2 * g + 1] = 0u;
    fsum += f;
    const int64_t X = (int64_t)an * Bp + (int64_t)(ad - an) * Hkv * f;
    Bg[g] = (int32_t)(X / den);
    rem[g] = X % den;
    flo += Bg[g];
  }
  if (fsum != Bp) raise_dev(hdr, DEV_SELECT, (unsigned)seg);
  for (int64_t left = Bp - flo; left > 0; --left) {
    int best = -1;
    for (int g = 0; g < Hkv; ++g) {
      if (rem[g] < 0) continue;
      if (best < 0 || rem[g] > rem[best]) best = g;
    }
    if (best < 0) break;
    Bg[best] += 1;
    rem[best] = -1;
  }
  for (int g = 0; g < Hkv; ++g) head_budget[seg * Hkv + g] = Bg[g] + w;
}

AllocPlan alloc_plan(const Shape& s) {
  AllocPlan p{};
  const int64_t S = s.segments();
  const int64_t N = (int64_t)s.Hkv * (s.C() > 0 ? s.C() : 1);
  // enough CTAs to cover the GPU about four times over, at least 8K keys each
  int64_t nch = cdiv((int64_t)num_sms() * 4, S > 0 ? S : 1);
  const int64_t maxch = cdiv(N, 8192);
  if (nch > maxch) nch = maxch;
  if (nch < 1) nch = 1;
  p.nchunkE = (int)nch;
  size_t off = kWsHeader;
  p.off_bprime = off;
  off += align_up((size_t)S * sizeof(int64_t), 256);
  p.off_epart = off;
  off += align_up((size_t)S * p.nchunkE * sizeof(double2), 256);
  p.off_e = off;
  off += align_up((size_t)S * 2 * sizeof(double), 256);
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
  char* sc = ws + p.off_scratch;
  RadixState* rst = reinterpret_cast<RadixState*>(sc);
  sc += align_up((size_t)S * sizeof(RadixState), 256);
  uint32_t* ghist = reinterpret_cast<uint32_t*>(sc);
  sc += align_up((size_t)S * kBins * sizeof(uint32_t), 256);
  uint32_t* counts = reinterpret_cast<uint32_t*>(sc);
  // histograms and counts start at zero; the kernels leave them zeroed behind them
  cudaError_t e = cudaMemsetAsync(ghist, 0,
                                  (size_t)(reinterpret_cast<char*>(counts) -
                                           reinterpret_cast<char*>(ghist)) +
                                      (size_t)S * 2 * kMaxHeads * sizeof(uint32_t),
                                  st);
  if (e != cudaSuccess) return e;
  const int nch = p.nchunkE;
  const unsigned sb = (unsigned)cdiv(S, 128);
  if (entropy_mode) {
    double2* part = reinterpret_cast<double2*>(ws + p.off_epart);
    entropy_hist<<<dim3(nch, (unsigned)S), kThreads, 0, st>>>(scores, N, nch, part, ghist);
    layer_budgets<<<s.B, kThreads, 0, st>>>(part, nch, s.L, s.Hkv, s.n, s.w, C, budget,
                                            layer_budget, bprime, hdr);
    radix_init<<<sb, 128, 0, st>>>(nullptr, bprime, S, s.Hkv, C, s.w, layer_budget, bprime, rst,
                                   hdr);
    count_launches(3);
  } else {
    radix_init<<<sb, 128, 0, st>>>(budget, nullptr, S, s.Hkv, C, s.w, layer_budget, bprime, rst,
                                   hdr);
    radix_hist<<<dim3(nch, (unsigned)S), kThreads, 0, st>>>(scores, N, nch, rst, ghist, 0);
    count_launches(2);
  }
  for (int pass = 0; pass < 3; ++pass) {
    if (pass > 0) {
      radix_hist<<<dim3(nch, (unsigned)S), kThreads, 0, st>>>(scores, N, nch, rst, ghist, pass);
      count_launches(1);
    }
    radix_pick<<<(unsigned)S, 1024, 0, st>>>(rst, ghist, pass);
    count_launches(1);
  }
  radix_count<<<dim3(nch, (unsigned)S), kThreads, 0, st>>>(scores, s.Hkv, C, nch, rst, counts);
  alloc_blend<<<sb, 128, 0, st>>>(rst, bprime, counts, S, s.Hkv, C, s.w, an, ad, head_budget, hdr);
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace kv
