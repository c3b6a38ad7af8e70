// One decode step of attention over the flat cache.
//
// Ada-KV formal model: the new token's k, v are appended to its head's cache,
// then A = softmax(q K^T / sqrt(d)) and o = A V per query head; the flat layout
// with uneven per-head lengths is read as variable-length (cu_seqlens-style)
// attention.  Flash-decoding: every (sequence, layer, KV head) is split into
// `splits` row ranges whose partial (max, sum, o) are merged by a combine
// kernel; the G query heads of a KV head share one read of its K/V rows.
#include "kv_internal.cuh"

namespace kv {

namespace {
constexpr int kThreads = 256;
constexpr int kTile = 64;
constexpr int kMaxG = 8;
constexpr int kMaxOut = 4;   // G*d / kThreads outputs per thread (G*d <= 1024)
}

// Append k_new / v_new at row cu + lens of every head (one warp per head).
__global__ void decode_append(const char* __restrict__ kn, const char* __restrict__ vn,
                              char* __restrict__ kf, char* __restrict__ vf,
                              const int64_t* __restrict__ cu, int32_t* __restrict__ lens,
                              int64_t H, int Hkv, int row_bytes, int64_t cap, WsHeader* hdr) {
  const int64_t h = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= H) return;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g], end = cu[seg * (Hkv + 1) + g + 1];
  const int len = lens[h];
  if (base + len >= end || base + len >= cap) {
    if (lane == 0) raise_dev(hdr, DEV_NO_RESERVE, (unsigned)h);
    return;
  }
  const int vecs = row_bytes >> 4;
  const int64_t row = base + len;
  for (int c = lane; c < vecs; c += 32) {
    reinterpret_cast<uint4*>(kf + row * row_bytes)[c] =
        reinterpret_cast<const uint4*>(kn + h * row_bytes)[c];
    reinterpret_cast<uint4*>(vf + row * row_bytes)[c] =
        reinterpret_cast<const uint4*>(vn + h * row_bytes)[c];
  }
  __syncwarp();
  if (lane == 0) lens[h] = len + 1;
}

// Partial attention of one row range of one KV head for its G query heads.
// part[(unit*splits + split)] = { m[G], l[G], o[G][d] } in log2 units.
template <typename T>
__global__ void __launch_bounds__(kThreads)
decode_partial(const T* __restrict__ q, const T* __restrict__ kf, const T* __restrict__ vf,
               const int64_t* __restrict__ cu, const int32_t* __restrict__ lens, int Hkv, int G,
               int d, int splits, int64_t cap, float c2, float* __restrict__ part) {
  extern __shared__ float sm[];
  const int dp = d + 1;
  float* Qs = sm;                       // [G][d]
  float* Ks = Qs + G * d;               // [kTile][d+1]
  float* Vs = Ks + kTile * dp;          // [kTile][d]
  float* Ps = Vs + kTile * d;           // [G][kTile]
  float* Ms = Ps + G * kTile;           // [G] running max
  float* Ls = Ms + kMaxG;               // [G] running sum
  float* As = Ls + kMaxG;               // [G] rescale of this tile
  const int64_t unit = blockIdx.y;
  const int split = blockIdx.x;
  const int64_t seg = unit / Hkv;
  const int g = (int)(unit - seg * Hkv);
  const int Hq = Hkv * G;
  const int64_t base = cu[seg * (Hkv + 1) + g];
  // rows past the flat buffer are never read
  const int64_t room = cap - base;
  const int len = (int)max((int64_t)0, min((int64_t)lens[unit], room));
  const int per = (len + splits - 1) / splits;
  const int r0 = split * per, r1 = min(len, r0 + per);
  const T* Q = q + (seg * Hq + (int64_t)g * G) * d;
  for (int i = threadIdx.x; i < G * d; i += kThreads) Qs[i] = to_f(Q[i]);
  if (threadIdx.x < kMaxG) { Ms[threadIdx.x] = -INFINITY; Ls[threadIdx.x] = 0.f; }
  const int nout = G * d;
  float o[kMaxOut];
#pragma unroll
  for (int u = 0; u < kMaxOut; ++u) o[u] = 0.f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t0 = r0; t0 < r1; t0 += kTile) {
    __syncthreads();
    for (int i = threadIdx.x; i < kTile * d; i += kThreads) {
      const int rr = i / d, c = i - rr * d;
      const int r = t0 + rr;
      float kv = 0.f, vv = 0.f;
      if (r < r1) {
        kv = to_f(kf[(base + r) * d + c]);
        vv = to_f(vf[(base + r) * d + c]);
      }
      Ks[rr * dp + c] = kv;
      Vs[rr * d + c] = vv;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * kTile; i += kThreads) {
      const int qq = i / kTile, rr = i - qq * kTile;
      float acc = 0.f;
      const float* qr = Qs + qq * d;
      const float* kr = Ks + rr * dp;
      for (int c = 0; c < d; ++c) acc = fmaf(qr[c], kr[c], acc);
      Ps[i] = (t0 + rr < r1) ? acc * c2 : -INFINITY;
    }
    __syncthreads();
    if (warp < G) {
      float* pr = Ps + warp * kTile;
      float mx = -INFINITY;
      for (int rr = lane; rr < kTile; rr += 32) mx = fmaxf(mx, pr[rr]);
      mx = warp_max(mx);
      const float mold = Ms[warp];
      const float mnew = fmaxf(mold, mx);
      float s = 0.f;
      for (int rr = lane; rr < kTile; rr += 32) {
        const float p = exp2f(pr[rr] - mnew);
        pr[rr] = p;
        s += p;
      }
      s = warp_sum(s);
      if (lane == 0) {
        const float a = exp2f(mold - mnew);
        As[warp] = a;
        Ls[warp] = Ls[warp] * a + s;
        Ms[warp] = mnew;
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kMaxOut; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      if (idx < nout) {
        const int qq = idx / d, c = idx - qq * d;
        const float* pr = Ps + qq * kTile;
        float acc = o[u] * As[qq];
        for (int rr = 0; rr < kTile; ++rr) acc = fmaf(pr[rr], Vs[rr * d + c], acc);
        o[u] = acc;
      }
    }
  }
  __syncthreads();
  float* P = part + (unit * splits + split) * (int64_t)G * (d + 2);
  if (threadIdx.x < G) {
    P[threadIdx.x] = Ms[threadIdx.x];
    P[G + threadIdx.x] = Ls[threadIdx.x];
  }
#pragma unroll
  for (int u = 0; u < kMaxOut; ++u) {
    const int idx = threadIdx.x + u * kThreads;
    if (idx < nout) P[2 * G + idx] = o[u];
  }
}

template <typename T>
__global__ void decode_combine(const float* __restrict__ part, int splits, int Hkv, int G, int d,
                               T* __restrict__ out) {
  const int64_t unit = blockIdx.x;
  const int64_t seg = unit / Hkv;
  const int g = (int)(unit - seg * Hkv);
  const int Hq = Hkv * G;
  const int64_t stride = (int64_t)G * (d + 2);
  for (int idx = threadIdx.x; idx < G * d; idx += blockDim.x) {
    const int qq = idx / d;
    float M = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, part[(unit * splits + sp) * stride + qq]);
    float Lsum = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < splits; ++sp) {
        const float* P = part + (unit * splits + sp) * stride;
        const float m = P[qq];
        if (m == -INFINITY) continue;
        const float a = exp2f(m - M);
        Lsum += P[G + qq] * a;
        O += P[2 * G + idx] * a;
      }
    }
    const float val = Lsum > 0.f ? O / Lsum : 0.f;
    out[(seg * Hq + (int64_t)g * G) * d + idx] = from_f<T>(val);
  }
}

DecodePlan decode_plan(const Shape& s) {
  DecodePlan p{};
  const int64_t units = s.units();
  int64_t sp = cdiv((int64_t)num_sms() * 8, units > 0 ? units : 1);
  if (sp < 1) sp = 1;
  if (sp > 64) sp = 64;
  p.splits = (int)sp;
  size_t off = kWsHeader;
  p.off_part = off;
  off += align_up((size_t)units * p.splits * s.G() * (s.d + 2) * sizeof(float), 256);
  p.off_end = off;
  return p;
}

template <typename T>
static cudaError_t launch_decode_t(const Shape& s, const T* q, void* kf, void* vf,
                                   const int64_t* cu, int32_t* lens, int64_t cap, float scale,
                                   T* out, char* ws, const DecodePlan& p, cudaStream_t st) {
  const int G = s.G(), d = s.d;
  const int64_t units = s.units();
  float* part = reinterpret_cast<float*>(ws + p.off_part);
  const size_t sm = (size_t)(G * d + kTile * (d + 1) + kTile * d + G * kTile + 3 * kMaxG) *
                    sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(decode_partial<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const float c2 = scale * 1.4426950408889634f;
  decode_partial<T><<<dim3(p.splits, (unsigned)units), kThreads, sm, st>>>(
      q, (const T*)kf, (const T*)vf, cu, lens, s.Hkv, G, d, p.splits, cap, c2, part);
  decode_combine<T><<<(unsigned)units, 256, 0, st>>>(part, p.splits, s.Hkv, G, d, out);
  count_launches(2);
  return cudaGetLastError();
}

cudaError_t launch_decode(const Shape& s, const void* q, const void* kn, const void* vn,
                          void* kf, void* vf, const int64_t* cu, int32_t* lens, int64_t cap,
                          float scale, void* out, char* ws, const DecodePlan& p,
                          cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t H = s.units();
  if (kn != nullptr) {
    const int warps = 8;
    decode_append<<<(unsigned)cdiv(H, warps), warps * 32, 0, st>>>(
        (const char*)kn, (const char*)vn, (char*)kf, (char*)vf, cu, lens, H, s.Hkv,
        s.d * s.esize(), cap, hdr);
    count_launches(1);
  }
  if (s.dtype == KV_BF16)
    return launch_decode_t<__nv_bfloat16>(s, (const __nv_bfloat16*)q, kf, vf, cu, lens, cap,
                                          scale, (__nv_bfloat16*)out, ws, p, st);
  return launch_decode_t<float>(s, (const float*)q, kf, vf, cu, lens, cap, scale, (float*)out,
                                ws, p, st);
}

}  // namespace kv
