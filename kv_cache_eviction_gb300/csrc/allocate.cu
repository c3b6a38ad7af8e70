// Per-head budgets of every (sequence, layer).
//
// Ada-KV Algorithm 1: concatenate the heads' scores, take the layer-wide top
// B', count how many of them each head owns (f_g).  Ada-KV Algorithm 2,
// safeguard: blend f_g with the uniform share B'/Hkv, exact integers, alpha on
// the uniform side.  LAVa, uncertainty-based layer budgets: each layer's share
// of the sequence's total is proportional to the entropy of its normalised
// scores.
#include "kv_internal.cuh"
#include "radix_select.cuh"

namespace kv {

namespace {
constexpr int kSelThreads = 1024;
constexpr int kMaxHeads = 256;
constexpr int kEntThreads = 256;
}

// Per-chunk partial sums of s and s*ln(s) (fp64 accumulation).
__global__ void __launch_bounds__(kEntThreads)
entropy_partial(const float* __restrict__ scores, int64_t N, int nch,
                double2* __restrict__ part) {
  const int64_t seg = blockIdx.y;
  const int64_t per = cdiv(N, nch);
  const int64_t i0 = blockIdx.x * per, i1 = min(N, i0 + per);
  const float* S = scores + seg * N;
  double a = 0.0, b = 0.0;
  for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const float x = S[i];
    if (x > 0.0f) {
      a += (double)x;
      b += (double)x * (double)logf(x);
    }
  }
  a = warp_sum_d(a);
  b = warp_sum_d(b);
  __shared__ double sa[kEntThreads / 32], sb[kEntThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sa[warp] = a; sb[warp] = b; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double ta = 0.0, tb = 0.0;
    for (int i = 0; i < kEntThreads / 32; ++i) { ta += sa[i]; tb += sb[i]; }
    part[seg * nch + blockIdx.x] = make_double2(ta, tb);
  }
}

// One thread per sequence: e_l, then the capped proportional split of
// R = total - L*w*Hkv with floors and largest remainders (ties to the lower layer).
__global__ void layer_budgets(const double2* __restrict__ part, int nch, int L, int Hkv, int n,
                              int w, int C, const int64_t* __restrict__ total,
                              int32_t* __restrict__ layer_budget, int64_t* __restrict__ bprime,
                              double* __restrict__ scratch, WsHeader* hdr) {
  if (threadIdx.x != 0) return;
  const int b = blockIdx.x;
  double* e = scratch + (int64_t)b * L * 2;
  double* quota = e + L;
  int64_t* sel = bprime + (int64_t)b * L;
  for (int l = 0; l < L; ++l) {
    double S = 0.0, T = 0.0;
    const double2* p = part + ((int64_t)b * L + l) * nch;
    for (int c = 0; c < nch; ++c) { S += p[c].x; T += p[c].y; }
    double el = 0.0;
    if (S > 0.0) el = (log(S) - T / S) / ((double)Hkv * (double)n);
    e[l] = el > 0.0 ? el : 0.0;
  }
  const int64_t cap = (int64_t)Hkv * C;
  int64_t R = total[b] - (int64_t)L * w * Hkv;
  if (R < 0 || R > (int64_t)L * cap) {
    raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)b);
    R = R < 0 ? 0 : (int64_t)L * cap;
  }
  // sel[l] = -1 marks an active (not yet capped) layer.
  for (int l = 0; l < L; ++l) sel[l] = -1;
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
    quota[l] -= f;                  // keep only the fractional part
    sel[l] = -2 - (int64_t)f;       // still marked active: floor stored as -2 - floor
    used += (int64_t)f;
  }
  int64_t left = rem - used;
  for (; left > 0; --left) {
    int best = -1;
    for (int l = 0; l < L; ++l) {
      if (sel[l] > -2) continue;    // capped or already bumped
      if (best < 0 || quota[l] > quota[best]) best = l;
    }
    if (best < 0) break;
    sel[best] = (-2 - sel[best]) + 1;   // floor + 1, now final
  }
  for (int l = 0; l < L; ++l) {
    if (sel[l] <= -2) sel[l] = -2 - sel[l];
    layer_budget[(int64_t)b * L + l] = (int32_t)(sel[l] + (int64_t)w * Hkv);
  }
}

// One CTA per (sequence, layer): layer-wide threshold, per-head counts, blend.
__global__ void __launch_bounds__(kSelThreads)
alloc_select(const float* __restrict__ scores, int Hkv, int C, int w,
             const int64_t* __restrict__ budget, const int64_t* __restrict__ bprime_in,
             uint32_t an, uint32_t ad, int32_t* __restrict__ layer_budget,
             int32_t* __restrict__ head_budget, WsHeader* hdr) {
  __shared__ RadixSmem rs;
  __shared__ uint32_t gt[kMaxHeads], eq[kMaxHeads];
  __shared__ int64_t X[kMaxHeads];
  __shared__ int32_t Bg[kMaxHeads];
  __shared__ unsigned int red[2][32];
  const int64_t seg = blockIdx.x;
  const int64_t N = (int64_t)Hkv * C;
  const float* S = scores + seg * N;
  int64_t Bp;
  if (bprime_in) {
    Bp = bprime_in[seg];
  } else {
    Bp = budget[seg] - (int64_t)w * Hkv;
    if (Bp < 0 || Bp > N) {
      if (threadIdx.x == 0) raise_dev(hdr, DEV_BUDGET_RANGE, (unsigned)seg);
      Bp = Bp < 0 ? 0 : N;
    }
    if (threadIdx.x == 0) layer_budget[seg] = (int32_t)(Bp + (int64_t)w * Hkv);
  }
  uint32_t tau, keq;
  block_topk_threshold<kSelThreads>(N, Bp, [&](int64_t i) { return score_key(S[i]); }, rs, tau,
                                    keq);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int g = 0; g < Hkv; ++g) {
    unsigned int cg = 0, ce = 0;
    const float* Sg = S + (int64_t)g * C;
    for (int64_t j = threadIdx.x; j < C; j += kSelThreads) {
      const uint32_t key = score_key(Sg[j]);
      cg += key > tau;
      ce += key == tau;
    }
    cg = warp_sum_u(cg);
    ce = warp_sum_u(ce);
    if (lane == 0) { red[0][warp] = cg; red[1][warp] = ce; }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned int a = 0, b = 0;
      for (int i = 0; i < kSelThreads / 32; ++i) { a += red[0][i]; b += red[1][i]; }
      gt[g] = a;
      eq[g] = b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // f_g: all keys above tau, plus tau-equal keys in (head, position) order.
    int64_t left_eq = keq, fsum = 0;
    const int64_t den = (int64_t)ad * Hkv;
    int64_t flo = 0;
    for (int g = 0; g < Hkv; ++g) {
      int64_t take = left_eq < (int64_t)eq[g] ? left_eq : (int64_t)eq[g];
      if (take < 0) take = 0;
      left_eq -= take;
      const int64_t f = (int64_t)gt[g] + take;
      fsum += f;
      X[g] = (int64_t)an * Bp + (int64_t)(ad - an) * Hkv * f;
      Bg[g] = (int32_t)(X[g] / den);
      flo += Bg[g];
      X[g] = X[g] % den;   // remainder
    }
    if (fsum != Bp) raise_dev(hdr, DEV_SELECT, (unsigned)seg);
    for (int64_t left = Bp - flo; left > 0; --left) {
      int best = -1;
      for (int g = 0; g < Hkv; ++g) {
        if (X[g] < 0) continue;
        if (best < 0 || X[g] > X[best]) best = g;
      }
      if (best < 0) break;
      Bg[best] += 1;
      X[best] = -1;
    }
    for (int g = 0; g < Hkv; ++g) head_budget[seg * Hkv + g] = Bg[g] + w;
  }
}

AllocPlan alloc_plan(const Shape& s) {
  AllocPlan p{};
  const int64_t S = s.segments();
  const int64_t N = (int64_t)s.Hkv * (s.C() > 0 ? s.C() : 1);
  p.nchunkE = (int)(N / 65536 + 1);
  if (p.nchunkE > 64) p.nchunkE = 64;
  size_t off = kWsHeader;
  p.off_bprime = off;
  off += align_up((size_t)S * sizeof(int64_t), 256);
  p.off_epart = off;
  off += align_up((size_t)S * p.nchunkE * sizeof(double2), 256);
  p.off_e = off;
  off += align_up((size_t)S * 2 * sizeof(double), 256);
  p.off_scratch = off;
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
  int64_t* bprime = reinterpret_cast<int64_t*>(ws + p.off_bprime);
  if (entropy_mode) {
    double2* part = reinterpret_cast<double2*>(ws + p.off_epart);
    double* scratch = reinterpret_cast<double*>(ws + p.off_e);
    entropy_partial<<<dim3(p.nchunkE, (unsigned)S), kEntThreads, 0, st>>>(
        scores, (int64_t)s.Hkv * C, p.nchunkE, part);
    layer_budgets<<<s.B, 32, 0, st>>>(part, p.nchunkE, s.L, s.Hkv, s.n, s.w, C, budget,
                                      layer_budget, bprime, scratch, hdr);
    count_launches(2);
  }
  alloc_select<<<(unsigned)S, kSelThreads, 0, st>>>(scores, s.Hkv, C, s.w,
                                                    entropy_mode ? nullptr : budget,
                                                    entropy_mode ? bprime : nullptr, an, ad,
                                                    layer_budget, head_budget, hdr);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace kv
