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
// launch (a programmatic dependent of the call before it), no partials in global memory.
// Rows of 256 bytes (bf16 d = 128, fp32 d = 64):
// 16 lanes per row, tiles of 32 scores per warp (RowTileAttn).
#include "decode_rows16.cuh"

namespace kv {

namespace {
using namespace r16;
constexpr int kHWarps = 4;
constexpr int kHThreads = kHWarps * 32;
constexpr int kHStages = kStages;
constexpr int kHRows = kStageRows;
constexpr int kHRowBytes = kRowBytes;

struct HeadSmem {
  WarpRing w[kHWarps];
};
}  // namespace

// GM: the group size rounded up to 2, 4 or 8 (register arrays); G <= GM is the real one.
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
  WarpRing& ws = S.w[warp];
  const int half = lane >> 4, ci = lane & 15;
  const int64_t h = blockIdx.x;
  const int64_t seg = h / Hkv;
  const int g0 = (int)(h - seg * Hkv);
  const int GD = G * D;

  if (lane == 0) {
    for (int s = 0; s < kHStages; ++s) ptx::mbar_init(&ws.full[s], 1);
    ptx::fence_mbar_init();
  }
  // a programmatic dependent launch: the next call on the stream may start launching, and
  // nothing of the previous one is read or written before it is done
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  // this lane's slices of the G query rows, scaled into the exp2 domain
  using Att = RowTileAttn<T, GM>;
  Att att;
  {
    uint4 qr[GM];
    load_q<T, GM>(q, h, G, ci, qr);
    att.begin(qr, c2);
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
    for (int b = 0; b < nr; b += Att::kRows) {
      uint4 kr[Att::U], vr[Att::U];
      load_tile<Att>(ws.st[s][0], ws.st[s][1], b, nr, kr, vr);
      att.tile(kr, vr, nr - b, ws.red, ws.pbuf);
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
    uint4 kr[Att::U], vr[Att::U];
#pragma unroll
    for (int u = 0; u < Att::U; ++u) {
      kr[u] = make_uint4(0u, 0u, 0u, 0u);
      vr[u] = kr[u];
    }
    if (half == 0) {
      kr[0] = *reinterpret_cast<const uint4*>(kn + h * D + ci * VE);
      vr[0] = *reinterpret_cast<const uint4*>(vn + h * D + ci * VE);
    }
    att.tile(kr, vr, 1, ws.red, ws.pbuf);
  }
  // this warp's (max, sum, o): the two half-warps' o hold different rows' terms
  att.finish();
  __syncthreads();   // every warp is done with its ring: its memory holds the partials now
  float* part = reinterpret_cast<float*>(dsm_raw);   // [warp][g][2 + D]
  const int pstride = 2 + D;
  if (half == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        float* P = part + (warp * GM + g) * pstride;
        if (ci == 0) {
          P[0] = att.m[g];
          P[1] = att.l[g];
        }
#pragma unroll
        for (int e2 = 0; e2 < V2; ++e2) {
          P[2 + ci * VE + 2 * e2] = att.o[g][e2].x;
          P[2 + ci * VE + 2 * e2 + 1] = att.o[g][e2].y;
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

// One instantiation: its shared-memory opt-in once per device (each kernel needs its own),
// then the launch, one CTA per KV head.
template <typename T, int GM>
static cudaError_t launch_head_t(const Shape& s, const void* q, const void* kn, const void* vn,
                                 void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                 int64_t cap, float c2, void* out, WsHeader* hdr,
                                 cudaStream_t st) {
  const size_t smem = sizeof(HeadSmem);
  static std::atomic<int> opted[kMaxDevices];
  if (!per_device(opted, [&]() {
        return cudaFuncSetAttribute(decode_head<T, GM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem) == cudaSuccess ? 1 : 0;
      }))
    return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)s.units());
  cfg.blockDim = dim3(kHThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_head<T, GM>, (const T*)q, (const T*)kn,
                                           (const T*)vn, (T*)kf, (T*)vf, cu, lens, cap, (T*)out,
                                           s.Hkv, s.G(), c2, hdr);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

cudaError_t launch_decode_head(const Shape& s, const void* q, const void* kn, const void* vn,
                               void* kf, void* vf, const int64_t* cu, int32_t* lens,
                               int64_t cap, float scale, void* out, WsHeader* hdr,
                               cudaStream_t st) {
  const float c2 = scale * 1.4426950408889634f;
  const int G = s.G();
  const int GM = G <= 2 ? 2 : G <= 4 ? 4 : 8;   // tiles of 32 scores: GM >= 2
#define KV_HEAD_CASE(T, M)                                                                 \
  return launch_head_t<T, M>(s, q, kn, vn, kf, vf, cu, lens, cap, c2, out, hdr, st)
  if (s.dtype == KV_BF16) {
    switch (GM) {
      case 2: KV_HEAD_CASE(__nv_bfloat16, 2);
      case 4: KV_HEAD_CASE(__nv_bfloat16, 4);
      default: KV_HEAD_CASE(__nv_bfloat16, 8);
    }
  }
  switch (GM) {
    case 2: KV_HEAD_CASE(float, 2);
    case 4: KV_HEAD_CASE(float, 4);
    default: KV_HEAD_CASE(float, 8);
  }
#undef KV_HEAD_CASE
}

}  // namespace kv
