// One decode step of attention over the flat cache when its heads are short.
//
// Ada-KV formal model: the new token's k, v are appended to its head's cache, then
// A = softmax(q K^T / sqrt(d)) and o = A V per query head, over the uneven per-head lengths
// of the flat layout.
//
// With a few hundred rows per head, the row-balanced split of decode.cu is a chain of
// latencies (a prep kernel, a chunk map, a merge kernel) around very little data.  Here
// one CTA of 4 warps takes one KV head: the warps split the head's rows evenly, each
// streams its rows through its own ring of bulk copies (3 stages, 16 rows each), the new
// token's row is read straight from k_new / v_new, the warps' (max, sum, o) are merged in
// shared memory, and the CTA finally appends the new row and bumps the head's length.  One
// launch, no partials in global memory.  Rows of 256 bytes (bf16 d = 128, fp32 d = 64):
// 16 lanes per row, two rows per warp step.
#include "kv_internal.cuh"
#include "tc_ptx.cuh"

namespace kv {

namespace {
constexpr int kHWarps = 4;
constexpr int kHThreads = kHWarps * 32;
constexpr int kHStages = 3;
constexpr int kHRows = 16;                   // rows per ring stage
constexpr int kHRowBytes = 256;
constexpr int kHStageBytes = kHRows * kHRowBytes;

// Every warp's stages start on a 128-byte boundary (bulk copies need 16-byte aligned shared
// memory destinations; the barriers would otherwise leave warps 1..3 at an 8-byte offset).
struct __align__(128) HeadWarpSmem {
  unsigned char st[kHStages][2][kHStageBytes];   // [stage][K, V]
  uint64_t full[kHStages];
};
static_assert(sizeof(HeadWarpSmem) % 128 == 0, "per-warp stages stay 128-byte aligned");
struct HeadSmem {
  HeadWarpSmem w[kHWarps];
};

__device__ __forceinline__ void unpack_row16(const uint4& r, float2 (&f)[4]) {   // bf16 x 8
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
}
__device__ __forceinline__ void unpack_row16(const uint4& r, float2 (&f)[2]) {   // fp32 x 4
  f[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
  f[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
}
__device__ __forceinline__ uint4 pack_row16(const float (&o)[8], __nv_bfloat16) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 pack_row16(const float (&o)[4], float) {
  return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                    __float_as_uint(o[3]));
}
}  // namespace

// GM: the group size rounded up to 1, 2, 4 or 8 (register arrays); G <= GM is the real one.
template <typename T, int GM>
__global__ void __launch_bounds__(kHThreads, 2)
decode_head(const T* __restrict__ q, const T* __restrict__ kn, const T* __restrict__ vn,
            T* __restrict__ kf, T* __restrict__ vf, const int64_t* __restrict__ cu,
            int32_t* __restrict__ lens, int64_t cap, T* __restrict__ out, int Hkv, int G,
            float c2, WsHeader* hdr) {
  constexpr int VE = 16 / (int)sizeof(T);    // elements per 16-byte lane slice
  constexpr int V2 = VE / 2;                 // fp32 pairs per slice
  constexpr int D = kHRowBytes / (int)sizeof(T);
  extern __shared__ __align__(128) unsigned char dsm_raw[];
  HeadSmem& S = *reinterpret_cast<HeadSmem*>(dsm_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  HeadWarpSmem& ws = S.w[warp];
  const int half = lane >> 4, ci = lane & 15;
  const int64_t h = blockIdx.x;
  const int64_t seg = h / Hkv;
  const int g0 = (int)(h - seg * Hkv);
  const int GD = G * D;

  if (lane == 0) {
    for (int s = 0; s < kHStages; ++s) ptx::mbar_init(&ws.full[s], 1);
    ptx::fence_mbar_init();
  }
  // this lane's slices of the G query rows, scaled into the exp2 domain
  float2 qf[GM][V2];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    float2 f[V2];
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (g < G) raw = *reinterpret_cast<const uint4*>(q + h * GD + g * D + ci * VE);
    unpack_row16(raw, f);
#pragma unroll
    for (int e = 0; e < V2; ++e) qf[g][e] = ptx::fmul2(f[e], make_float2(c2, c2));
  }
  const int64_t base = cu[seg * (Hkv + 1) + g0], end = cu[seg * (Hkv + 1) + g0 + 1];
  const int len = lens[h];
  const int64_t e = end < cap ? end : cap;
  // rows read from the flat buffer, and whether the new row is appended (and attended to)
  int64_t nflat = 0;
  bool app = false;
  if (e > base && base >= 0) {
    nflat = len > 0 ? (int64_t)len : 0;
    if (nflat > e - base) nflat = e - base;
    app = kn != nullptr && len >= 0 && base + len < end && base + len < cap;
  }
  if (threadIdx.x == 0) {
    if (end > cap) raise_dev(hdr, DEV_FLAT_CAPACITY, (unsigned)h);
    if (kn != nullptr && !app) raise_dev(hdr, DEV_NO_RESERVE, (unsigned)h);
  }
  const int64_t R = nflat + (app ? 1 : 0);
  const int64_t r0 = R * warp / kHWarps, r1 = R * (warp + 1) / kHWarps;
  const int64_t f0 = r0, f1 = r1 < nflat ? r1 : nflat;   // this warp's flat rows
  const int nitems = f1 > f0 ? (int)((f1 - f0 + kHRows - 1) / kHRows) : 0;
  __syncwarp();

  auto issue = [&](int it) {
    if (lane == 0) {
      const int s = it % kHStages;
      const int64_t row = base + f0 + (int64_t)it * kHRows;
      const int64_t nr = (f1 - (f0 + (int64_t)it * kHRows)) < kHRows
                             ? f1 - (f0 + (int64_t)it * kHRows) : kHRows;
      const uint32_t bytes = (uint32_t)(nr * kHRowBytes);
      ptx::mbar_arrive_expect_tx(&ws.full[s], 2u * bytes);
      ptx::bulk_load(ws.st[s][0], reinterpret_cast<const char*>(kf) + row * kHRowBytes, bytes,
                     &ws.full[s]);
      ptx::bulk_load(ws.st[s][1], reinterpret_cast<const char*>(vf) + row * kHRowBytes, bytes,
                     &ws.full[s]);
    }
  };
  int issued = 0;   // items whose copies have been issued (the same in every lane)
  for (; issued < nitems && issued < kHStages; ++issued) issue(issued);

  float mrun[GM], lrun[GM];
  float2 o[GM][V2];
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    mrun[g] = -INFINITY;
    lrun[g] = 0.f;
#pragma unroll
    for (int e2 = 0; e2 < V2; ++e2) o[g][e2] = make_float2(0.f, 0.f);
  }
  // two rows per step (one per half-warp): k, v slices of this lane's row, ok = row exists
  auto step = [&](const uint4& kr, const uint4& vr, bool ok) {
    float2 kfv[V2], vfv[V2];
    unpack_row16(kr, kfv);
    unpack_row16(vr, vfv);
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      float2 a = make_float2(0.f, 0.f);
#pragma unroll
      for (int e2 = 0; e2 < V2; ++e2) a = ptx::ffma2(qf[g][e2], kfv[e2], a);
      float sc = a.x + a.y;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sc += __shfl_xor_sync(0xFFFFFFFFu, sc, off);
      if (!ok) sc = -INFINITY;
      const float so = __shfl_xor_sync(0xFFFFFFFFu, sc, 16);   // the other half's row
      const float mn = fmaxf(mrun[g], fmaxf(sc, so));
      const float mu = mn == -INFINITY ? 0.f : mn;
      const float al = ptx::ex2(mrun[g] - mu);
      const float p = ptx::ex2(sc - mu), po = ptx::ex2(so - mu);
      mrun[g] = mn;
      lrun[g] = lrun[g] * al + p + po;
#pragma unroll
      for (int e2 = 0; e2 < V2; ++e2)
        o[g][e2] = ptx::ffma2(make_float2(p, p), vfv[e2],
                              ptx::fmul2(o[g][e2], make_float2(al, al)));
    }
  };

  bool okw = true;
  int consumed = 0;   // items read (their stage may be reused)
  for (int it = 0; it < nitems && okw; ++it) {
    const int s = it % kHStages;
    const bool landed = ptx::mbar_wait(&ws.full[s], (uint32_t)((it / kHStages) & 1));
    if (__any_sync(0xFFFFFFFFu, !landed)) {
      okw = false;
      if (lane == 0) raise_dev(hdr, DEV_WAIT_TIMEOUT, 0x600u + (unsigned)s);
      break;
    }
    const int64_t rb = f0 + (int64_t)it * kHRows;
    const int nr = (int)((f1 - rb) < kHRows ? f1 - rb : kHRows);
    {
      const unsigned char* Ks = ws.st[s][0];
      const unsigned char* Vs = ws.st[s][1];
      for (int r = 0; r < nr; r += 2) {
        const int row = r + half;
        const bool ok = row < nr;
        uint4 kr = make_uint4(0u, 0u, 0u, 0u), vr = kr;
        if (ok) {
          kr = *reinterpret_cast<const uint4*>(Ks + row * kHRowBytes + ci * 16);
          vr = *reinterpret_cast<const uint4*>(Vs + row * kHRowBytes + ci * 16);
        }
        step(kr, vr, ok);
      }
    }
    __syncwarp();   // every lane is done with stage s
    consumed = it + 1;
    if (issued < nitems) issue(issued++);
  }
  if (!okw && lane == 0) {
    // a wait gave up: let the copies issued and not yet read land before the memory is reused
    for (int it = consumed; it < issued; ++it)
      (void)ptx::mbar_wait(&ws.full[it % kHStages], (uint32_t)((it / kHStages) & 1),
                           20000000ull);
  }
  // the new row, in the warp whose range holds it
  if (app && r0 <= nflat && nflat < r1) {
    uint4 kr = make_uint4(0u, 0u, 0u, 0u), vr = kr;
    if (half == 0) {
      kr = *reinterpret_cast<const uint4*>(kn + h * D + ci * VE);
      vr = *reinterpret_cast<const uint4*>(vn + h * D + ci * VE);
    }
    step(kr, vr, half == 0);
  }
  // this warp's (max, sum, o): the two half-warps' o hold different rows' terms
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int e2 = 0; e2 < V2; ++e2) {
      o[g][e2].x += __shfl_xor_sync(0xFFFFFFFFu, o[g][e2].x, 16);
      o[g][e2].y += __shfl_xor_sync(0xFFFFFFFFu, o[g][e2].y, 16);
    }
  __syncthreads();   // every warp is done with its ring: its memory holds the partials now
  float* part = reinterpret_cast<float*>(dsm_raw);   // [warp][g][2 + D]
  const int pstride = 2 + D;
  if (half == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        float* P = part + (warp * GM + g) * pstride;
        if (ci == 0) {
          P[0] = mrun[g];
          P[1] = lrun[g];
        }
#pragma unroll
        for (int e2 = 0; e2 < V2; ++e2) {
          P[2 + ci * VE + 2 * e2] = o[g][e2].x;
          P[2 + ci * VE + 2 * e2 + 1] = o[g][e2].y;
        }
      }
    }
  }
  __syncthreads();
  // merge the warps' partials: thread t writes 16 bytes of one query row
  for (int idx = threadIdx.x; idx < G * (D / VE); idx += kHThreads) {
    const int g = idx / (D / VE), sl = idx - g * (D / VE);
    float M = -INFINITY;
    for (int w = 0; w < kHWarps; ++w) M = fmaxf(M, part[(w * GM + g) * pstride]);
    const float mu = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    float acc[VE];
#pragma unroll
    for (int x = 0; x < VE; ++x) acc[x] = 0.f;
    for (int w = 0; w < kHWarps; ++w) {
      const float* P = part + (w * GM + g) * pstride;
      const float sc = ptx::ex2(P[0] - mu);
      L += P[1] * sc;
#pragma unroll
      for (int x = 0; x < VE; ++x) acc[x] += P[2 + sl * VE + x] * sc;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int x = 0; x < VE; ++x) acc[x] *= inv;
    *reinterpret_cast<uint4*>(out + h * GD + g * D + sl * VE) = pack_row16(acc, T());
  }
  // append the new row (no warp read its slot) and count it
  if (app && warp == 0) {
    const int64_t row = base + len;
    if (lane < 16) {
      reinterpret_cast<uint4*>(kf + row * D)[ci] =
          reinterpret_cast<const uint4*>(kn + h * D)[ci];
      reinterpret_cast<uint4*>(vf + row * D)[ci] =
          reinterpret_cast<const uint4*>(vn + h * D)[ci];
    }
    if (lane == 0) lens[h] = len + 1;
  }
}

// cap = 0: the row size and group alone decide (a forced choice)
bool decode_head_supported(const Shape& s, int64_t cap) {
  const int64_t H = s.units();
  return s.d * s.esize() == kHRowBytes && s.G() <= 8 && H > 0 && cap / H <= kDecodeHeadRowsMax;
}

// One instantiation: its shared-memory opt-in once (each kernel needs its own), then the
// launch, one CTA per KV head.
template <typename T, int GM>
static cudaError_t launch_head_t(const Shape& s, const void* q, const void* kn, const void* vn,
                                 void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                 int64_t cap, float c2, void* out, WsHeader* hdr,
                                 cudaStream_t st) {
  const size_t smem = sizeof(HeadSmem);
  static const cudaError_t opted = cudaFuncSetAttribute(
      decode_head<T, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (opted != cudaSuccess) return opted;
  decode_head<T, GM><<<(unsigned)s.units(), kHThreads, smem, st>>>(
      (const T*)q, (const T*)kn, (const T*)vn, (T*)kf, (T*)vf, cu, lens, cap, (T*)out, s.Hkv,
      s.G(), c2, hdr);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_decode_head(const Shape& s, const void* q, const void* kn, const void* vn,
                               void* kf, void* vf, const int64_t* cu, int32_t* lens,
                               int64_t cap, float scale, void* out, WsHeader* hdr,
                               cudaStream_t st) {
  const float c2 = scale * 1.4426950408889634f;
  const int G = s.G();
  const int GM = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
#define KV_HEAD_CASE(T, M)                                                                 \
  return launch_head_t<T, M>(s, q, kn, vn, kf, vf, cu, lens, cap, c2, out, hdr, st)
  if (s.dtype == KV_BF16) {
    switch (GM) {
      case 1: KV_HEAD_CASE(__nv_bfloat16, 1);
      case 2: KV_HEAD_CASE(__nv_bfloat16, 2);
      case 4: KV_HEAD_CASE(__nv_bfloat16, 4);
      default: KV_HEAD_CASE(__nv_bfloat16, 8);
    }
  }
  switch (GM) {
    case 1: KV_HEAD_CASE(float, 1);
    case 2: KV_HEAD_CASE(float, 2);
    case 4: KV_HEAD_CASE(float, 4);
    default: KV_HEAD_CASE(float, 8);
  }
#undef KV_HEAD_CASE
}

}  // namespace kv
