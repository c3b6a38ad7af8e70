// The step after the tcgen05 window-scoring kernel.
//
// LAVa: the score of key j is the pooled window mean times max_k ||V[k]||_1 over the unit's
// candidate keys, a factor known only once every range of the unit has been through the
// main kernel, which therefore writes unscaled scores.  SnapKV-style pooling: a key within
// pool/2 of a boundary between two CTAs' ranges needs window means from both sides; the main
// kernel leaves halo copies of the means next to each boundary and the keys are pooled here.
#include "kv_internal.cuh"

namespace kv {

namespace {
constexpr int kFixThreads = 256;
constexpr int kFixU = 4;   // 16-byte vectors in flight per thread
}

// Grid (chunks, units).  A CTA scales its chunk of the unit's keys, then rewrites the
// boundary keys that fall inside the chunk (pooled from the halos, then scaled).
__global__ void __launch_bounds__(kFixThreads)
score_tc_fixup(const float* __restrict__ halo, const float* __restrict__ vbar, int Pg, int Tu,
               int C, int G, int r, int group_max, int terms, int per,
               float* __restrict__ scores) {
  const int64_t u = blockIdx.y;
  const int c0 = min(C, (int)blockIdx.x * per), c1 = min(C, c0 + per);
  // terms: every query head's pooled mean, scores[u][G][C]
  float* S = scores + u * (int64_t)C * (terms ? G : 1);
  float vb = 1.0f;
  if (vbar) {
    vb = vbar[u];
    const uintptr_t addr = reinterpret_cast<uintptr_t>(S + c0);
    const int a = min(c1, c0 + (int)(((16u - (uint32_t)(addr & 15u)) & 15u) >> 2));
    const int nv = (c1 - a) >> 2;
    const int b = a + 4 * nv;
    if (c0 + (int)threadIdx.x < a) S[c0 + threadIdx.x] *= vb;
    if (b + (int)threadIdx.x < c1) S[b + threadIdx.x] *= vb;
    float4* xv = reinterpret_cast<float4*>(S + a);
    for (int j0 = threadIdx.x; j0 < nv; j0 += kFixU * kFixThreads) {
      float4 x[kFixU];
#pragma unroll
      for (int k = 0; k < kFixU; ++k) {
        const int j = j0 + k * kFixThreads;
        x[k] = j < nv ? xv[j] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kFixU; ++k) {
        const int j = j0 + k * kFixThreads;
        if (j < nv) xv[j] = make_float4(x[k].x * vb, x[k].y * vb, x[k].z * vb, x[k].w * vb);
      }
    }
    __syncthreads();
  }
  const int R4 = 4 * r;
  for (int idx = threadIdx.x; idx < (Pg - 1) * 2 * r; idx += blockDim.x) {
    const int bnd = idx / (2 * r) + 1;
    const int b = (int)(((int64_t)bnd * Tu) / Pg) * 128;
    if (b >= C) continue;
    const int j = b - r + idx % (2 * r);
    if (j < c0 || j >= c1) continue;   // another CTA's key (or outside the unit)
    const int lo = max(0, j - r), hi = min(C - 1, j + r);
    const float* Hl = halo + (u * Pg + bnd - 1) * (int64_t)G * R4;
    const float* Hr = halo + (u * Pg + bnd) * (int64_t)G * R4;
    float gv = group_max ? -INFINITY : 0.f;
    for (int q = 0; q < G; ++q) {
      float pm = -INFINITY;
      for (int jj = lo; jj <= hi; ++jj) {
        const float x = jj < b ? Hl[q * R4 + 2 * r + (jj - (b - 2 * r))] : Hr[q * R4 + (jj - b)];
        pm = fmaxf(pm, x);
      }
      if (terms) S[(int64_t)q * C + j] = pm;
      gv = group_max ? fmaxf(gv, pm) : gv + pm;
    }
    if (terms) continue;
    if (!group_max) gv = gv / (float)G;
    if (vbar) gv = gv * vb;
    S[j] = gv;
  }
}

cudaError_t launch_score_fixup(const float* halo, const float* vbar, int64_t units, int Pg,
                               int Tu, int C, int G, int r, int group_max, int terms,
                               float* scores, cudaStream_t st) {
  if (units <= 0 || C <= 0) return cudaSuccess;
  // scaling: about eight CTAs per SM, at least 4K keys each; boundary keys only: one CTA
  int64_t nch = 1;
  if (vbar) {
    nch = cdiv((int64_t)num_sms() * 8, units);
    const int64_t maxch = cdiv(C, 4096);
    if (nch > maxch) nch = maxch;
    if (nch < 1) nch = 1;
  }
  const int per = (int)(cdiv(cdiv(C, nch), 4) * 4);
  nch = cdiv(C, per);
  score_tc_fixup<<<dim3((unsigned)nch, (unsigned)units), kFixThreads, 0, st>>>(
      halo, vbar, Pg, Tu, C, G, r, group_max, terms, per, scores);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace kv
