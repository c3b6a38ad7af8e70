// Pieces shared by the decode kernels that read rows of 256 bytes (bf16 d = 128, fp32
// d = 64): a warp's ring of bulk-copy stages, and the online softmax of one warp over tiles
// of rows.  Lane (half, ci) holds the 16-byte slice ci of the tile's rows of parity `half`,
// and slice ci of every query row's q and o.
#pragma once

#include "kv_internal.cuh"
#include "tc_ptx.cuh"

namespace kv {
namespace r16 {

constexpr int kRowBytes = 256;
constexpr int kStages = 3;
constexpr int kStageRows = 16;                   // rows per ring stage
constexpr int kStageBytes = kStageRows * kRowBytes;
// Partial of one (piece, head) in global or shared memory: max[8], sum[8] (G <= 8 used),
// then o[G][d]; 16 floats of head keep every o row 16-byte aligned.
constexpr int kPartHead = 16;

constexpr int kRedFloats = 576;   // tile transpose buffer (the largest, GM = 2)

// Every warp's stages start on a 128-byte boundary (bulk copies need 16-byte aligned shared
// memory destinations; the barriers would otherwise leave warps 1..3 at an 8-byte offset).
struct __align__(128) WarpRing {
  unsigned char st[kStages][2][kStageBytes];   // [stage][K, V]
  float red[kRedFloats];                       // RowTileAttn: partial dot products
  float2 pbuf[32];                             // RowTileAttn: softmax numerators
  uint64_t full[kStages];
};
static_assert(sizeof(WarpRing) % 128 == 0, "per-warp stages stay 128-byte aligned");

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

// Launch attribute of a programmatic dependent launch: the kernel may start while the one
// before it on the stream finishes, and waits (griddepcontrol.wait) before touching memory.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a{};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Slice ci of the query rows g < G of KV head h (zeros for g >= G).
template <typename T, int GM>
__device__ __forceinline__ void load_q(const T* __restrict__ q, int64_t h, int G, int ci,
                                       uint4 (&qr)[GM]) {
  constexpr int D = kRowBytes / (int)sizeof(T);
  constexpr int VE = 16 / (int)sizeof(T);
#pragma unroll
  for (int g = 0; g < GM; ++g) {
    qr[g] = make_uint4(0u, 0u, 0u, 0u);
    if (g < G) qr[g] = *reinterpret_cast<const uint4*>(q + (h * G + g) * D + ci * VE);
  }
}

// Running (max, sum, o) of GM query rows over the rows seen so far, in the exp2 domain
// (q is scaled by softmax scale * log2 e), over tiles of 2U rows (U = 16 / GM row pairs):
// lane (half, ci) computes the partial dot products of its slice with the query rows for
// each of its half's U rows;
// a transpose through shared memory leaves lane (vrow = lane / GM, gj = lane % GM) with the
// 16 partials of row vrow and query gj, whose sum is that row's score.  One maximum per
// query and tile, one exponential per lane for the numerators (shared back through shared
// memory) and a rescale of o only when a query's maximum grows: per row, a fraction of the
// shuffles and exponentials that reducing each row's dot product across its 16 lanes would
// take.
template <typename T, int GM>
struct RowTileAttn {
  static_assert(GM == 2 || GM == 4 || GM == 8, "tiles of 32 scores");
  static constexpr int VE = 16 / (int)sizeof(T);
  static constexpr int V2 = VE / 2;
  static constexpr int D = kRowBytes / (int)sizeof(T);
  static constexpr int U = 16 / GM;              // row pairs per tile
  static constexpr int kRows = 2 * U;            // rows per tile
  static constexpr int kRedStride = 17 * GM;     // floats per row (padding: no bank conflicts)
  static_assert(kRows * kRedStride <= kRedFloats, "transpose buffer");
  float2 qf[GM][V2];
  float2 o[GM][V2];
  float m[GM];   // running maximum per query (the same in every lane)
  float l[GM];   // after finish(): the sum per query
  float mj, lj;  // query gj = lane % GM: maximum at the last rescale, and this lane's sum

  __device__ __forceinline__ void begin(const uint4 (&qr)[GM], float c2) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      float2 f[V2];
      unpack_row16(qr[g], f);
#pragma unroll
      for (int e = 0; e < V2; ++e) {
        qf[g][e] = ptx::fmul2(f[e], make_float2(c2, c2));
        o[g][e] = make_float2(0.f, 0.f);
      }
      m[g] = -INFINITY;
    }
    mj = -INFINITY;
    lj = 0.f;
  }

  // One tile: kr[u], vr[u] are this lane's slices of tile row 2u + half; rows at or past
  // nvalid are masked (their slices may hold anything finite).
  __device__ __forceinline__ void tile(const uint4 (&kr)[U], const uint4 (&vr)[U], int nvalid,
                                       float* red, float2* pbuf) {
    const int lane = threadIdx.x & 31, half = lane >> 4, ci = lane & 15;
    const int gj = lane % GM, vrow = lane / GM;
    float sc[U][GM];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float2 f[V2];
      unpack_row16(kr[u], f);
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < V2; ++e) a = ptx::ffma2(qf[g][e], f[e], a);
        sc[u][g] = a.x + a.y;
      }
    }
    // [tile row][lane slice][query]
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float* dst = red + (2 * u + half) * kRedStride + ci * GM;
      if constexpr (GM == 2) {
        *reinterpret_cast<float2*>(dst) = make_float2(sc[u][0], sc[u][1]);
      } else {
#pragma unroll
        for (int g = 0; g < GM; g += 4)
          *reinterpret_cast<float4*>(dst + g) =
              make_float4(sc[u][g], sc[u][g + 1], sc[u][g + 2], sc[u][g + 3]);
      }
    }
    __syncwarp();
    float s0 = 0.f, s1 = 0.f;
    const float* src = red + vrow * kRedStride + gj;
#pragma unroll
    for (int t = 0; t < 16; t += 2) {
      s0 += src[t * GM];
      s1 += src[(t + 1) * GM];
    }
    float sj = s0 + s1;
    if (vrow >= nvalid) sj = -INFINITY;
    float mx = sj;
#pragma unroll
    for (int off = GM; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      const float mt = __shfl_sync(0xFFFFFFFFu, mx, g);
      if (mt > m[g]) {   // the same in every lane
        const float a = ptx::ex2(m[g] - mt);
        m[g] = mt;
#pragma unroll
        for (int e = 0; e < V2; ++e) o[g][e] = ptx::fmul2(o[g][e], make_float2(a, a));
        if (g == gj) {
          lj *= a;
          mj = mt;
        }
      }
    }
    const float pj = ptx::ex2(sj - (mj == -INFINITY ? 0.f : mj));
    lj += pj;
    pbuf[lane] = make_float2(pj, pj);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float2 pv[GM];
#pragma unroll
      for (int g = 0; g < GM; g += 2) {
        const float4 t = *reinterpret_cast<const float4*>(pbuf + (2 * u + half) * GM + g);
        pv[g] = make_float2(t.x, t.y);
        pv[g + 1] = make_float2(t.z, t.w);
      }
      float2 f[V2];
      unpack_row16(vr[u], f);
#pragma unroll
      for (int g = 0; g < GM; ++g)
#pragma unroll
        for (int e = 0; e < V2; ++e) o[g][e] = ptx::ffma2(pv[g], f[e], o[g][e]);
    }
  }

  // After the last tile: l per query, and o summed over the two half-warps (both halves
  // hold the sum).
  __device__ __forceinline__ void finish() {
    float ls = lj;
#pragma unroll
    for (int off = GM; off < 32; off <<= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, off);
#pragma unroll
    for (int g = 0; g < GM; ++g) l[g] = __shfl_sync(0xFFFFFFFFu, ls, g);
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
      for (int e = 0; e < V2; ++e) {
        o[g][e].x += __shfl_xor_sync(0xFFFFFFFFu, o[g][e].x, 16);
        o[g][e].y += __shfl_xor_sync(0xFFFFFFFFu, o[g][e].y, 16);
      }
  }
};

// Tile rows [b, b + kRows) of a stage of n rows: this lane's slices (zeros past n).
template <typename A>
__device__ __forceinline__ void load_tile(const unsigned char* Ks, const unsigned char* Vs, int b,
                                          int n, uint4 (&kr)[A::U], uint4 (&vr)[A::U]) {
  const int lane = threadIdx.x & 31, half = lane >> 4, ci = lane & 15;
#pragma unroll
  for (int u = 0; u < A::U; ++u) {
    const int r = b + 2 * u + half;
    kr[u] = make_uint4(0u, 0u, 0u, 0u);
    vr[u] = kr[u];
    if (r < n) {
      kr[u] = *reinterpret_cast<const uint4*>(Ks + r * kRowBytes + ci * 16);
      vr[u] = *reinterpret_cast<const uint4*>(Vs + r * kRowBytes + ci * 16);
    }
  }
}

}  // namespace r16
}  // namespace kv
