// Observation-window scoring on CUDA cores (any w, fp32 or bf16), plus the
// LAVa value-norm factor and the CriticalKV projected-value norm.
//
// Ada-KV (Algorithm 2, scoring steps): window softmax over the causal rows,
// window mean, max-pool, GQA group mean.  LAVa (Definition 1; GQA adaptation):
// scale by max_k ||V[k]||_1, group max.  CriticalKV (key designs): the row
// norm ||(V W^O)_j||_1.
//
// Two passes over K: pass 1 finds each window row's log-sum-exp over every key
// it can see (online max/sum per chunk, then a combine); pass 2 recomputes the
// logits of the candidate keys, forms exp(z - lse), averages over the window
// rows, pools and reduces over the query-head group.  Logits are kept in the
// log2 domain: z2 = (q.k) * scale * log2(e).
#include <cstdlib>
#include <cstring>

#include "kv_internal.cuh"

namespace kv {

namespace {
constexpr int kThreads = 256;     // 8 warps
constexpr int kMaxRowsPerWarp = 32;  // G*w <= 256
constexpr int kMaxG = 8;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
score_pass1_simt(const T* __restrict__ q_win, const T* __restrict__ k, int n, int w, int d, int R,
                 int chunk, int nchunk, float c2, float2* __restrict__ part) {
  extern __shared__ float sm[];
  const int dp = d + 1;
  float* Qs = sm;            // [R][d]
  float* Ks = sm + R * d;    // [32][d+1]
  const int64_t unit = blockIdx.y;
  const int ch = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* Q = q_win + unit * (int64_t)R * d;
  const T* K = k + unit * (int64_t)n * d;
  for (int i = threadIdx.x; i < R * d; i += blockDim.x) Qs[i] = to_f(Q[i]);
  const int j0 = ch * chunk, j1 = min(n, j0 + chunk);
  const int nr = (R - warp + 7) / 8;
  float m[kMaxRowsPerWarp], l[kMaxRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kMaxRowsPerWarp; ++i) { m[i] = -INFINITY; l[i] = 0.f; }
  for (int jt = j0; jt < j1; jt += 32) {
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * d; i += blockDim.x) {
      const int r = i / d, c = i - r * d, j = jt + r;
      Ks[r * dp + c] = (j < j1) ? to_f(K[(int64_t)j * d + c]) : 0.f;
    }
    __syncthreads();
    const int j = jt + lane;
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
      if (i < nr) {
        const int row = warp + 8 * i;
        const int t = row % w;
        const float* qr = Qs + row * d;
        const float* kr = Ks + lane * dp;
        float acc = 0.f;
        for (int c = 0; c < d; ++c) acc = fmaf(qr[c], kr[c], acc);
        const float z = (j < j1 && j <= n - w + t) ? acc * c2 : -INFINITY;
        const float mn = fmaxf(m[i], warp_max(z));
        if (mn != -INFINITY) {
          const float se = warp_sum(exp2f(z - mn));
          l[i] = l[i] * exp2f(m[i] - mn) + se;
          m[i] = mn;
        }
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i)
      if (i < nr) part[(unit * nchunk + ch) * R + warp + 8 * i] = make_float2(m[i], l[i]);
  }
}

// lse2[unit][row] = log2 sum_j exp2(z2[row, j]) from the per-chunk (max, sum) pairs.
__global__ void score_lse_combine(const float2* __restrict__ part, int nchunk, int R,
                                  float* __restrict__ lse2) {
  const int64_t unit = blockIdx.x;
  for (int row = threadIdx.x; row < R; row += blockDim.x) {
    float M = -INFINITY;
    for (int c = 0; c < nchunk; ++c) M = fmaxf(M, part[(unit * nchunk + c) * R + row].x);
    float S = 0.f;
    for (int c = 0; c < nchunk; ++c) {
      const float2 p = part[(unit * nchunk + c) * R + row];
      if (p.x != -INFINITY) S += p.y * exp2f(p.x - M);
    }
    lse2[unit * R + row] = M + log2f(S);
  }
}

// TERMS = 0: the KV head's score (window mean, pool, group mean or max, V-bar factor) into
// scores[unit][C].  TERMS = 1: every query head's pooled window mean, TERMS = 2: every query
// head's sqrt(sum_t P[t, j]^2) (no pooling: pool = 1), into scores[unit][G][C].
template <typename T, int TERMS = 0>
__global__ void __launch_bounds__(kThreads)
score_pass2_simt(const T* __restrict__ q_win, const T* __restrict__ k,
                 const float* __restrict__ lse2, const float* __restrict__ vbar, int n, int w,
                 int d, int G, int pool, int group_max, int chunk2, float c2,
                 float* __restrict__ scores) {
  extern __shared__ float sm[];
  const int R = G * w, dp = d + 1, C = n - w, r = pool / 2, ext = chunk2 + 2 * r;
  float* Qs = sm;                 // [R][d]
  float* Ks = Qs + R * d;         // [32][d+1]
  float* Ls = Ks + 32 * dp;       // [R]
  float* red = Ls + R;            // [8][G][32]
  float* As = red + 8 * G * 32;   // [G][ext] window means of candidates [e0, e1)
  const int64_t unit = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = blockIdx.x * chunk2, c1 = min(C, c0 + chunk2);
  const int e0 = max(0, c0 - r), e1 = min(C, c1 + r);
  const T* Q = q_win + unit * (int64_t)R * d;
  const T* K = k + unit * (int64_t)n * d;
  for (int i = threadIdx.x; i < R * d; i += blockDim.x) Qs[i] = to_f(Q[i]);
  for (int i = threadIdx.x; i < R; i += blockDim.x) Ls[i] = lse2[unit * R + i];
  const float inv_w = 1.0f / (float)w;
  const int nr = (R - warp + 7) / 8;
  for (int jt = e0; jt < e1; jt += 32) {
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * d; i += blockDim.x) {
      const int rr = i / d, c = i - rr * d, j = jt + rr;
      Ks[rr * dp + c] = (j < e1) ? to_f(K[(int64_t)j * d + c]) : 0.f;
    }
    __syncthreads();
    float accq[kMaxG];
#pragma unroll
    for (int q = 0; q < kMaxG; ++q) accq[q] = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxRowsPerWarp; ++i) {
      if (i < nr) {
        const int row = warp + 8 * i;
        const int ql = row / w;
        const float* qr = Qs + row * d;
        const float* kr = Ks + lane * dp;
        float acc = 0.f;
        for (int c = 0; c < d; ++c) acc = fmaf(qr[c], kr[c], acc);
        float p = exp2f(acc * c2 - Ls[row]);
        if (TERMS == 2) p *= p;
#pragma unroll
        for (int q = 0; q < kMaxG; ++q) accq[q] += (q == ql) ? p : 0.f;
      }
    }
    for (int q = 0; q < G; ++q) red[(warp * G + q) * 32 + lane] = accq[q];
    __syncthreads();
    if (warp == 0) {
      const int j = jt + lane;
      for (int q = 0; q < G; ++q) {
        float s = 0.f;
        for (int ww = 0; ww < 8; ++ww) s += red[(ww * G + q) * 32 + lane];
        if (j < e1) As[q * ext + (j - e0)] = TERMS == 2 ? sqrtf(s) : s * inv_w;
      }
    }
  }
  __syncthreads();
  if (TERMS != 0) {
    for (int idx = threadIdx.x; idx < G * (c1 - c0); idx += blockDim.x) {
      const int q = idx / (c1 - c0), j = c0 + (idx - q * (c1 - c0));
      const int lo = max(0, j - r), hi = min(C - 1, j + r);
      float pm = -INFINITY;
      for (int jj = lo; jj <= hi; ++jj) pm = fmaxf(pm, As[q * ext + (jj - e0)]);
      scores[(unit * G + q) * C + j] = pm;
    }
    return;
  }
  const float vb = vbar ? vbar[unit] : 1.0f;
  for (int j = c0 + threadIdx.x; j < c1; j += blockDim.x) {
    const int lo = max(0, j - r), hi = min(C - 1, j + r);
    float gv = group_max ? -INFINITY : 0.f;
    for (int q = 0; q < G; ++q) {
      float pm = -INFINITY;
      for (int jj = lo; jj <= hi; ++jj) pm = fmaxf(pm, As[q * ext + (jj - e0)]);
      gv = group_max ? fmaxf(gv, pm) : gv + pm;
    }
    if (!group_max) gv = gv / (float)G;
    if (vbar) gv = gv * vb;
    scores[unit * C + j] = gv;
  }
}

// vbar[unit] = max over rows of ||V[row]||_1 (float bits, atomicMax on non-negative floats).
template <typename T>
__global__ void __launch_bounds__(kThreads)
vbar_simt(const T* __restrict__ v, int n, int d, int rows_per_cta, unsigned int* __restrict__ vbar_bits) {
  const int64_t unit = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = blockIdx.x * rows_per_cta, r1 = min(n, r0 + rows_per_cta);
  const T* V = v + unit * (int64_t)n * d;
  float mx = 0.f;
  for (int row = r0 + warp; row < r1; row += 8) {
    float s = 0.f;
    for (int c = lane; c < d; c += 32) s += fabsf(to_f(V[(int64_t)row * d + c]));
    mx = fmaxf(mx, warp_sum(s));
  }
  __shared__ float wm[8];
  if (lane == 0) wm[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = wm[0];
    for (int i = 1; i < 8; ++i) m = fmaxf(m, wm[i]);
    atomicMax(&vbar_bits[unit], __float_as_uint(m));
  }
}

// crit[unit][j] = sum_e | sum_c V[j][c] * W_O[l][g][c][e] |  for j < C.
template <typename T>
__global__ void __launch_bounds__(kThreads)
crit_norm_simt(const T* __restrict__ v, const T* __restrict__ w_o, int L, int Hkv, int n, int C,
               int d, int D, float* __restrict__ crit) {
  extern __shared__ float sm[];
  float* Vs = sm;            // [32][d]
  float* Ws = Vs + 32 * d;   // [d][64]
  const int64_t unit = blockIdx.y;
  const int g = (int)(unit % Hkv);
  const int l = (int)((unit / Hkv) % L);
  const int j0 = blockIdx.x * 32;
  const T* V = v + unit * (int64_t)n * d;
  const T* W = w_o + ((int64_t)l * Hkv + g) * (int64_t)d * D;
  for (int i = threadIdx.x; i < 32 * d; i += blockDim.x) {
    const int rr = i / d, c = i - rr * d;
    Vs[i] = (j0 + rr < C) ? to_f(V[(int64_t)(j0 + rr) * d + c]) : 0.f;
  }
  const int row = threadIdx.x >> 3, cg = threadIdx.x & 7;
  float part = 0.f;
  for (int e0 = 0; e0 < D; e0 += 64) {
    __syncthreads();
    for (int i = threadIdx.x; i < d * 64; i += blockDim.x) {
      const int c = i >> 6, e = i & 63;
      Ws[i] = (e0 + e < D) ? to_f(W[(int64_t)c * D + e0 + e]) : 0.f;
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    for (int c = 0; c < d; ++c) {
      const float x = Vs[row * d + c];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = fmaf(x, Ws[c * 64 + cg * 8 + u], acc[u]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (e0 + cg * 8 + u < D) part += fabsf(acc[u]);
  }
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  part += __shfl_xor_sync(0xffffffffu, part, 4);
  if (cg == 0 && j0 + row < C) crit[unit * C + j0 + row] = part;
}

// ---------------------------------------------------------------------------
// tcgen05 path (score_tc.cu)
// ---------------------------------------------------------------------------
bool score_tc_supported(const Shape& s);
size_t score_tc_ws(const Shape& s, int mode);
cudaError_t launch_score_tc(const Shape& s, int mode, int group, const void* q_win,
                            const void* k, const void* v, float* scores, char* ws,
                            cudaStream_t st, int terms = 0);
bool crit_tc_supported(const Shape& s, int D);
cudaError_t launch_crit_tc(const Shape& s, const void* v, const void* w_o, int D, float* crit,
                           char* ws, cudaStream_t st);

// KVEVICT_SCORE_PATH=simt forces the CUDA-core kernels (tests compare the two paths).
static bool simt_forced() {
  const char* e = std::getenv("KVEVICT_SCORE_PATH");
  return e != nullptr && std::strcmp(e, "simt") == 0;
}

ScorePlan score_plan(const Shape& s, int mode) {
  ScorePlan p{};
  p.path = score_tc_supported(s) ? 1 : 0;
  const int64_t units = s.units();
  const int R = s.R();
  p.chunk1 = 512;
  p.nchunk1 = (int)cdiv(s.n, p.chunk1);
  p.chunk2 = 512;
  p.nchunk2 = (int)cdiv(s.C() > 0 ? s.C() : 1, p.chunk2);
  size_t off = kWsHeader;
  p.off_part = off;
  off += align_up((size_t)units * p.nchunk1 * R * sizeof(float2), 256);
  p.off_lse = off;
  off += align_up((size_t)units * R * sizeof(float), 256);
  p.off_vbar = off;
  off += align_up((size_t)units * sizeof(float), 256);
  p.off_end = off;
  // the workspace covers either path, whichever runs
  const size_t tc = score_tc_ws(s, mode);
  if (tc > p.off_end) p.off_end = tc;
  return p;
}

template <typename T>
static cudaError_t launch_score_simt_t(const Shape& s, int mode, int group, const T* q_win,
                                       const T* k, const T* v, float* scores, char* ws,
                                       const ScorePlan& p, cudaStream_t st) {
  const int R = s.R(), d = s.d, n = s.n, w = s.w, C = s.C();
  const int64_t units = s.units();
  const float c2 = (1.0f / sqrtf((float)d)) * 1.4426950408889634f;
  float2* part = reinterpret_cast<float2*>(ws + p.off_part);
  float* lse2 = reinterpret_cast<float*>(ws + p.off_lse);
  float* vbar = reinterpret_cast<float*>(ws + p.off_vbar);
  const size_t sm1 = (size_t)(R * d + 32 * (d + 1)) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(score_pass1_simt<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  score_pass1_simt<T><<<dim3(p.nchunk1, (unsigned)units), kThreads, sm1, st>>>(
      q_win, k, n, w, d, R, p.chunk1, p.nchunk1, c2, part);
  score_lse_combine<<<(unsigned)units, 128, 0, st>>>(part, p.nchunk1, R, lse2);
  count_launches(2);
  const float* vb = nullptr;
  if (mode == KV_SCORE_LAVA) {
    e = cudaMemsetAsync(vbar, 0, (size_t)units * sizeof(float), st);
    if (e != cudaSuccess) return e;
    const int rows = 256;
    vbar_simt<T><<<dim3((unsigned)cdiv(n, rows), (unsigned)units), kThreads, 0, st>>>(
        v, n, d, rows, reinterpret_cast<unsigned int*>(vbar));
    count_launches(1);
    vb = vbar;
  }
  if (C > 0) {
    const int G = s.G(), r = s.pool / 2;
    const size_t sm2 = (size_t)(R * d + 32 * (d + 1) + R + 8 * G * 32 + G * (p.chunk2 + 2 * r)) *
                       sizeof(float);
    e = cudaFuncSetAttribute(score_pass2_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm2);
    if (e != cudaSuccess) return e;
    score_pass2_simt<T><<<dim3(p.nchunk2, (unsigned)units), kThreads, sm2, st>>>(
        q_win, k, lse2, vb, n, w, d, G, s.pool, group == KV_GROUP_MAX, p.chunk2, c2, scores);
    count_launches(1);
  }
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_terms_simt_t(const Shape& s, int kind, const T* q_win, const T* k,
                                      float* terms, char* ws, const ScorePlan& p,
                                      cudaStream_t st) {
  const int R = s.R(), d = s.d, n = s.n, w = s.w, C = s.C();
  const int64_t units = s.units();
  const float c2 = (1.0f / sqrtf((float)d)) * 1.4426950408889634f;
  float2* part = reinterpret_cast<float2*>(ws + p.off_part);
  float* lse2 = reinterpret_cast<float*>(ws + p.off_lse);
  const size_t sm1 = (size_t)(R * d + 32 * (d + 1)) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(score_pass1_simt<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  score_pass1_simt<T><<<dim3(p.nchunk1, (unsigned)units), kThreads, sm1, st>>>(
      q_win, k, n, w, d, R, p.chunk1, p.nchunk1, c2, part);
  score_lse_combine<<<(unsigned)units, 128, 0, st>>>(part, p.nchunk1, R, lse2);
  count_launches(2);
  if (C > 0) {
    const int G = s.G();
    const int pool = kind == KV_TERMS_L2 ? 1 : s.pool, r = pool / 2;
    const size_t sm2 = (size_t)(R * d + 32 * (d + 1) + R + 8 * G * 32 + G * (p.chunk2 + 2 * r)) *
                       sizeof(float);
    auto kern = kind == KV_TERMS_L2 ? score_pass2_simt<T, 2> : score_pass2_simt<T, 1>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
    if (e != cudaSuccess) return e;
    kern<<<dim3(p.nchunk2, (unsigned)units), kThreads, sm2, st>>>(
        q_win, k, lse2, nullptr, n, w, d, G, pool, 0, p.chunk2, c2, terms);
    count_launches(1);
  }
  return cudaGetLastError();
}

cudaError_t launch_window_terms(const Shape& s, int kind, const void* q_win, const void* k,
                                float* terms, char* ws, const ScorePlan& p, cudaStream_t st) {
  // the tcgen05 kernel where the shape allows (its P2 epilogue forms every query head's
  // window sums anyway), the CUDA-core kernels otherwise
  if (p.path == 1 && !simt_forced())
    return launch_score_tc(s, KV_SCORE_ADA, KV_GROUP_MEAN, q_win, k, nullptr, terms, ws, st,
                           kind == KV_TERMS_L2 ? 2 : 1);
  if (s.dtype == KV_BF16)
    return launch_terms_simt_t<__nv_bfloat16>(s, kind, (const __nv_bfloat16*)q_win,
                                              (const __nv_bfloat16*)k, terms, ws, p, st);
  return launch_terms_simt_t<float>(s, kind, (const float*)q_win, (const float*)k, terms, ws, p,
                                    st);
}

template <typename T>
static cudaError_t launch_crit_simt_t(const Shape& s, const T* v, const T* w_o, int D,
                                      float* crit, cudaStream_t st) {
  const int C = s.C();
  if (C <= 0) return cudaSuccess;
  const size_t sm = (size_t)(32 * s.d + s.d * 64) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(crit_norm_simt<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  crit_norm_simt<T><<<dim3((unsigned)cdiv(C, 32), (unsigned)s.units()), kThreads, sm, st>>>(
      v, w_o, s.L, s.Hkv, s.n, C, s.d, D, crit);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_score(const Shape& s, int mode, int group, const void* q_win, const void* k,
                         const void* v, const void* w_o, int D, float* scores, float* crit,
                         char* ws, const ScorePlan& p, cudaStream_t st) {
  cudaError_t e;
  if (p.path == 1) {
    e = launch_score_tc(s, mode, group, q_win, k, v, scores, ws, st);
  } else if (s.dtype == KV_BF16) {
    e = launch_score_simt_t<__nv_bfloat16>(s, mode, group, (const __nv_bfloat16*)q_win,
                                           (const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
                                           scores, ws, p, st);
  } else {
    e = launch_score_simt_t<float>(s, mode, group, (const float*)q_win, (const float*)k,
                                   (const float*)v, scores, ws, p, st);
  }
  if (e != cudaSuccess || mode != KV_SCORE_CRITICAL) return e;
  return launch_crit_norm(s, v, w_o, D, crit, ws, st);
}

cudaError_t launch_crit_norm(const Shape& s, const void* v, const void* w_o, int D, float* crit,
                             char* ws, cudaStream_t st) {
  if (crit_tc_supported(s, D) && !simt_forced())
    return launch_crit_tc(s, v, w_o, D, crit, ws, st);
  if (s.dtype == KV_BF16)
    return launch_crit_simt_t<__nv_bfloat16>(s, (const __nv_bfloat16*)v,
                                             (const __nv_bfloat16*)w_o, D, crit, st);
  return launch_crit_simt_t<float>(s, (const float*)v, (const float*)w_o, D, crit, st);
}

}  // namespace kv
