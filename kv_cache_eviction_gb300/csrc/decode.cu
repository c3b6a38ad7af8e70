// One decode step of attention over the flat cache: the entry point that picks one of three
// kernels (one CTA per head in decode_head.cu, the one-launch split of decode_split.cu, or
// the row-balanced split below, for many long heads).
//
// Ada-KV formal model: the new token's k, v are appended to its head's cache,
// then A = softmax(q K^T / sqrt(d)) and o = A V per query head; the flat layout
// with uneven per-head lengths is read as variable-length (cu_seqlens-style)
// attention.
//
// Work split (flash-decoding over the flat buffer, balanced by rows, not by heads):
// the flat row range [0, cap) is cut into equal chunks of C rows, whatever heads they
// hold.  Per-head lengths are very uneven after head-adaptive allocation, so a head-major
// split would leave a few workers with most of the rows.  Every warp is an independent
// worker: it takes a chunk from an atomic queue, streams the chunk's K/V rows through its
// own two-stage shared-memory ring (bulk copies, one mbarrier per stage), and keeps the
// online-softmax state of one head in registers.  A head inside one chunk is finished by
// that warp; a head spanning several chunks leaves one partial (max, sum, o) per chunk,
// merged by a third kernel (merging in the workers, behind a fence and a ticket, stalls
// them for longer than the other warps of an SM can cover).  No barrier ties the warps of
// a CTA together.
//
//   decode_prep     one warp per head: append k_new / v_new, lens += 1, write
//                   chunk -> first head into a map, clear the chunk queue.
//   decode_attn     persistent CTAs (as many as fit), every warp a worker.
//   decode_combine  heads that span several chunks: merges their partials.
// The second and third kernels are programmatic dependents of the one before.
#include <cstdlib>
#include <cstring>

#include "kv_internal.cuh"
#include "tc_ptx.cuh"

namespace kv {

namespace {
constexpr int kPrepWarps = 8;
constexpr int kWarps = 4;                  // workers per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kStageBytes = 4096;          // K (and again V) bytes per ring stage per warp
constexpr int kItemsPerChunkMin = 4;       // a chunk holds at least this many full stages
constexpr int kRedFloats = 8 * (16 * 4 + 4);   // transpose buffer per warp (floats)
// Partial of one (chunk, head): max[8], sum[8] (G <= 8 used), then o[G][d]; 16 floats of
// head keep every o row 16-byte aligned whatever G is.
constexpr int kPartHead = 16;

struct WarpSmem {
  unsigned char stage[2][2][kStageBytes];  // [stage][K, V]
  float red[kRedFloats];                   // [row step][lane slice][query] partial dots
  float2 pbuf[32];                         // softmax numerators, one per lane
  uint64_t full[2];
};
struct DecSmem {
  WarpSmem w[kWarps];
};

// 16 bytes of one row as fp32 pairs (elements 2i, 2i+1 in .x, .y).
__device__ __forceinline__ void unpack16(const uint4& r, float2 (&f)[4]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
}
__device__ __forceinline__ void unpack16(const uint4& r, float2 (&f)[2]) {
  f[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
  f[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
}
// One lane slice of the output, o * inv, as 16 bytes of the output type.
__device__ __forceinline__ uint4 pack16(const float2 (&o)[4], float inv, __nv_bfloat16) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(o[i].x * inv, o[i].y * inv);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 pack16(const float2 (&o)[2], float inv, float) {
  return make_uint4(__float_as_uint(o[0].x * inv), __float_as_uint(o[0].y * inv),
                    __float_as_uint(o[1].x * inv), __float_as_uint(o[1].y * inv));
}

__device__ __forceinline__ int64_t shfl64(int64_t v, int src) {
  return (int64_t)__shfl_sync(0xFFFFFFFFu, (long long)v, src);
}
}  // namespace

// Append, chunk map and queue reset; one warp per head.
__global__ void decode_prep(const char* __restrict__ kn, const char* __restrict__ vn,
                            char* __restrict__ kf, char* __restrict__ vf,
                            const int64_t* __restrict__ cu, int32_t* __restrict__ lens,
                            uint32_t* __restrict__ map, uint32_t* __restrict__ work,
                            char* __restrict__ out, int64_t H, int Hkv, int row_bytes,
                            int out_bytes, int64_t cap, int64_t C, int64_t nchunks,
                            WsHeader* hdr) {
  ptx::griddep_launch_dependents();
  const int64_t h = (int64_t)blockIdx.x * kPrepWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= H) return;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g], end = cu[seg * (Hkv + 1) + g + 1];
  const int len = lens[h];
  if (kn != nullptr) {
    const int64_t row = base + len;
    if (len < 0 || row >= end || row >= cap) {
      if (lane == 0) raise_dev(hdr, DEV_NO_RESERVE, (unsigned)h);
    } else {
      for (int c = lane; c < (row_bytes >> 4); c += 32) {
        reinterpret_cast<uint4*>(kf + row * row_bytes)[c] =
            reinterpret_cast<const uint4*>(kn + h * row_bytes)[c];
        reinterpret_cast<uint4*>(vf + row * row_bytes)[c] =
            reinterpret_cast<const uint4*>(vn + h * row_bytes)[c];
      }
      if (lane == 0) lens[h] = len + 1;
    }
  }
  if (lane == 0) {
    if (h == 0) *work = 0u;
    if (end > cap) raise_dev(hdr, DEV_FLAT_CAPACITY, (unsigned)h);
  }
  const int64_t e = end < cap ? end : cap;
  if (e <= base || base < 0) {
    // no row of this head can be read: its output is zero
    for (int c = lane; c < (out_bytes >> 4); c += 32)
      reinterpret_cast<uint4*>(out + h * out_bytes)[c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  // chunks whose first row lies in this head's extent start their walk here
  for (int64_t c = cdiv(base, C) + lane; c < nchunks && c * C < e; c += 32)
    map[c] = (uint32_t)h;
}

// Row steps per warp iteration: with 16 lanes per row, U * GM = 16 puts the iteration's
// 2 * U * GM partial dot products one per lane after the shared-memory transpose.
template <int GM>
struct DecU {
  static constexpr int value = GM >= 8 ? 2 : 4;
};

// GM: the group size rounded up to 1, 2, 4 or 8 (register arrays); G <= GM is the real one.
// LPRT: lanes per row when fixed at compile time (0: derived from d at run time).
template <typename T, int GM, int LPRT>
__global__ void __launch_bounds__(kThreads, GM >= 8 ? 2 : 3)
decode_attn(const T* __restrict__ q, const T* __restrict__ kf, const T* __restrict__ vf,
            const int64_t* __restrict__ cu, const int32_t* __restrict__ lens,
            const uint32_t* __restrict__ map, uint32_t* __restrict__ work,
            float* __restrict__ part, T* __restrict__ out, int64_t H, int Hkv, int G, int d,
            int64_t cap, int64_t C, int64_t nchunks, float c2, WsHeader* hdr) {
  constexpr int VE = 16 / (int)sizeof(T);       // elements per 16-byte lane slice
  constexpr int V2 = VE / 2;                    // fp32 pairs per slice
  constexpr int U = DecU<GM>::value;            // row steps per warp iteration
  // Dot-product reduction across the lanes of a row: through shared memory (one sum per
  // lane) when the iteration holds exactly 32 of them, else by butterfly shuffles.
  constexpr bool kXpose = LPRT == 16 && U * GM == 16;
  constexpr int kRedStride = 16 * GM + 4;       // floats per row step (padding: no conflicts)
  static_assert(!kXpose || 2 * U * kRedStride <= kRedFloats, "transpose buffer");
  extern __shared__ __align__(128) unsigned char dsm_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WarpSmem& ws = reinterpret_cast<DecSmem*>(dsm_raw)->w[warp];

  const int row_bytes = d * (int)sizeof(T);
  const int CPR = d / VE;                       // 16-byte slices per row
  int LPR = 1;
  while (LPR < CPR) LPR <<= 1;                  // lanes per row
  if (LPRT > 0) LPR = LPRT;
  const int RPS = 32 / LPR;                     // rows per warp step
  const int ci = lane & (LPR - 1), rg = lane / LPR;
  const bool act = ci < CPR;
  const int Ct = kStageBytes / row_bytes;       // rows per stage
  const int GD = G * d;
  const int64_t pstride = kPartHead + (int64_t)GD; // floats per partial
  // transpose path: this lane's reduced value is (row step vrow = lane / GM, query gj)
  const int gj = lane % GM, vrow = lane / GM;

  if (lane == 0) {
    ptx::mbar_init(&ws.full[0], 1);
    ptx::mbar_init(&ws.full[1], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  // the merge kernel may start launching; it waits for this grid before reading anything
  ptx::griddep_launch_dependents();
  // everything below reads what decode_prep wrote
  ptx::griddep_wait();
  const int64_t S = H / Hkv;
  const int64_t total = cu[S * (Hkv + 1) - 1];
  const int64_t nworkers = (int64_t)gridDim.x * kWarps;

  uint32_t phase = 0;                           // bit s: parity of the next wait on full[s]
  bool abort_ = false;                          // a wait gave up: no more waits or copies
  int64_t c = (int64_t)blockIdx.x * kWarps + warp;
  while (c < nchunks && c * C < total) {
    const int64_t R0 = c * C;
    const int64_t R1 = (R0 + C < cap) ? R0 + C : cap;
    // the next chunk is claimed now and used when this one is done
    uint32_t claim = 0;
    if (lane == 0) claim = atomicAdd(work, 1u);
    const int64_t h0 = (int64_t)map[c];
    for (int64_t hstart = h0; h0 < H;) {
      // piece table: lane i holds head hstart + i's rows in this chunk
      const int64_t h = hstart + lane;
      bool in_range = false, inc = false, single = false;
      int64_t lo = 0, hi = 0, slot = 0;
      if (h < H) {
        const int64_t seg = h / Hkv;
        const int g = (int)(h - seg * Hkv);
        const int64_t base = cu[seg * (Hkv + 1) + g], end = cu[seg * (Hkv + 1) + g + 1];
        const int64_t len = lens[h];
        const int64_t e = end < cap ? end : cap;
        in_range = base < R1;
        inc = in_range && e > base && base >= 0 && e > R0;
        lo = base > R0 ? base : R0;
        hi = base + (len > 0 ? len : 0);
        if (hi > e) hi = e;
        if (hi > R1) hi = R1;
        if (hi < lo) hi = lo;
        single = inc && base / C == (e - 1) / C;
        slot = c + h;
        if (inc && hi > lo) {
          const char* qh = reinterpret_cast<const char*>(q + h * GD);
          for (int off = 0; off < GD * (int)sizeof(T); off += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qh + off));
        }
      }
      const uint32_t pmask = __ballot_sync(0xFFFFFFFFu, inc);
      const uint32_t smask = __ballot_sync(0xFFFFFFFFu, single);
      const bool more = (__ballot_sync(0xFFFFFFFFu, in_range) >> 31) & 1u;

      // producer cursor (lane 0 issues; every lane tracks it): piece lane pl, first row px
      uint32_t prem = pmask;
      int pl = prem ? __ffs(prem) - 1 : 32;
      int64_t px = shfl64(lo, pl & 31);
      int issued = 0;
      auto issue_next = [&]() {
        if (pl >= 32) return;
        const int64_t phi = shfl64(hi, pl);
        const int64_t nr = (px + Ct < phi) ? (int64_t)Ct : phi - px;
        if (lane == 0 && !abort_) {
          const int s = issued & 1;
          const uint32_t bytes = (uint32_t)(nr * row_bytes);
          ptx::mbar_arrive_expect_tx(&ws.full[s], 2u * bytes);
          if (bytes) {
            ptx::bulk_load(ws.stage[s][0], reinterpret_cast<const char*>(kf) + px * row_bytes,
                           bytes, &ws.full[s]);
            ptx::bulk_load(ws.stage[s][1], reinterpret_cast<const char*>(vf) + px * row_bytes,
                           bytes, &ws.full[s]);
          }
        }
        ++issued;
        if (px + nr >= phi) {
          prem &= prem - 1u;
          pl = prem ? __ffs(prem) - 1 : 32;
          px = shfl64(lo, pl & 31);
        } else {
          px += nr;
        }
      };
      issue_next();
      issue_next();

      // consumer: the same sequence, two items behind
      uint32_t crem = pmask;
      int cl = crem ? __ffs(crem) - 1 : 32;
      int64_t cx = shfl64(lo, cl & 31);
      float2 qf[GM][V2], o[GM][V2];
      float mrun[GM], lrun[GM];
      float mj = -INFINITY, lj = 0.f;           // transpose path: state of query gj
      for (int k = 0; cl < 32; ++k) {
        const int s = k & 1;
        const int64_t clo = shfl64(lo, cl), chi = shfl64(hi, cl), ch = shfl64(h, cl);
        const int64_t nr = (cx + Ct < chi) ? (int64_t)Ct : chi - cx;
        const bool first = cx == clo, last = cx + nr >= chi;
        if (first && chi > clo) {
          const T* qh = q + ch * GD;
#pragma unroll
          for (int g = 0; g < GM; ++g) {
            float2 f[V2];
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (act && g < G) raw = *reinterpret_cast<const uint4*>(qh + g * d + ci * VE);
            unpack16(raw, f);
#pragma unroll
            for (int e = 0; e < V2; ++e) {
              qf[g][e] = ptx::fmul2(f[e], make_float2(c2, c2));
              o[g][e] = make_float2(0.f, 0.f);
            }
            mrun[g] = -INFINITY;
            lrun[g] = 0.f;
          }
          mj = -INFINITY;
          lj = 0.f;
        }
        // wait for the item's rows (bounded; after a timeout nothing waits again)
        const uint32_t par = (phase >> s) & 1u;
        phase ^= 1u << s;
        if (!abort_) {
          const bool ok = ptx::mbar_wait_sleep(&ws.full[s], par);
          if (__any_sync(0xFFFFFFFFu, !ok)) {
            abort_ = true;
            if (lane == 0) raise_dev(hdr, DEV_WAIT_TIMEOUT, 0x400u + (unsigned)s);
          }
        }
        const unsigned char* Ks = ws.stage[s][0];
        const unsigned char* Vs = ws.stage[s][1];
        for (int b = 0; b < nr; b += U * RPS) {
          uint4 kr[U], vr[U];
          bool ok[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int r = b + u * RPS + rg;
            ok[u] = r < nr;
            kr[u] = make_uint4(0u, 0u, 0u, 0u);
            vr[u] = kr[u];
            if (ok[u] && act) {
              kr[u] = *reinterpret_cast<const uint4*>(Ks + r * row_bytes + ci * 16);
              vr[u] = *reinterpret_cast<const uint4*>(Vs + r * row_bytes + ci * 16);
            }
          }
          // partial q.k over this lane's slice
          float sc[U][GM];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            float2 f[V2];
            unpack16(kr[u], f);
#pragma unroll
            for (int g = 0; g < GM; ++g) {
              float2 a = make_float2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < V2; ++e) a = ptx::ffma2(qf[g][e], f[e], a);
              sc[u][g] = a.x + a.y;
            }
          }
          float2 p2[U][GM];                      // softmax numerators, duplicated in .x/.y
          if constexpr (kXpose) {
            // [row step][lane slice][query]: lane (rg, ci) writes its GM partials of step u
            float* red = ws.red;
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
              for (int g = 0; g < GM; g += 4)
                *reinterpret_cast<float4*>(red + (u * 2 + rg) * kRedStride + ci * GM + g) =
                    make_float4(sc[u][g], sc[u][g + 1], sc[u][g + 2], sc[u][g + 3]);
            __syncwarp();
            float sj = 0.f, sj2 = 0.f;
#pragma unroll
            for (int t = 0; t < 16; t += 2) {
              sj += red[vrow * kRedStride + t * GM + gj];
              sj2 += red[vrow * kRedStride + (t + 1) * GM + gj];
            }
            sj += sj2;
            if (b + vrow >= nr) sj = -INFINITY;  // row step vrow = u * 2 + rg is row b + vrow
            // maximum of each query over the iteration's rows, then in every lane
            float mx = sj;
#pragma unroll
            for (int off = GM; off < 32; off <<= 1)
              mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
#pragma unroll
            for (int g = 0; g < GM; ++g) {
              const float mt = __shfl_sync(0xFFFFFFFFu, mx, g);
              if (mt > mrun[g]) {                // warp-uniform
                const float a = ptx::ex2(mrun[g] - mt);
                mrun[g] = mt;
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
            ws.pbuf[lane] = make_float2(pj, pj);
            __syncwarp();
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
              for (int g = 0; g < GM; g += 2) {
                const float4 t =
                    *reinterpret_cast<const float4*>(ws.pbuf + (u * 2 + rg) * GM + g);
                p2[u][g] = make_float2(t.x, t.y);
                p2[u][g + 1] = make_float2(t.z, t.w);
              }
          } else {
            for (int off = 1; off < LPR; off <<= 1) {
#pragma unroll
              for (int u = 0; u < U; ++u)
#pragma unroll
                for (int g = 0; g < GM; ++g)
                  sc[u][g] += __shfl_xor_sync(0xFFFFFFFFu, sc[u][g], off);
            }
#pragma unroll
            for (int g = 0; g < GM; ++g) {
              float mt = -INFINITY;
#pragma unroll
              for (int u = 0; u < U; ++u) {
                if (!ok[u]) sc[u][g] = -INFINITY;
                mt = fmaxf(mt, sc[u][g]);
              }
              for (int off = LPR; off < 32; off <<= 1)
                mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, off));
              const float mn = fmaxf(mrun[g], mt);
              const float mu = mn == -INFINITY ? 0.f : mn;
              const float a = ptx::ex2(mrun[g] - mu);
              mrun[g] = mn;
              lrun[g] *= a;
#pragma unroll
              for (int e = 0; e < V2; ++e) o[g][e] = ptx::fmul2(o[g][e], make_float2(a, a));
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const float pv = ptx::ex2(sc[u][g] - mu);
                lrun[g] += pv;
                p2[u][g] = make_float2(pv, pv);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            float2 f[V2];
            unpack16(vr[u], f);
#pragma unroll
            for (int g = 0; g < GM; ++g)
#pragma unroll
              for (int e = 0; e < V2; ++e) o[g][e] = ptx::ffma2(p2[u][g], f[e], o[g][e]);
          }
        }
        __syncwarp();                            // every lane is done with stage s
        issue_next();

        if (last) {
          const bool sgl = (smask >> cl) & 1u;
          float* P = part + shfl64(slot, cl) * pstride;
          if (chi > clo) {
            // fold the sums of the row groups (and, transposed, of the lanes of a query)
            if constexpr (kXpose) {
#pragma unroll
              for (int off = GM; off < 32; off <<= 1)
                lj += __shfl_xor_sync(0xFFFFFFFFu, lj, off);
#pragma unroll
              for (int g = 0; g < GM; ++g) lrun[g] = __shfl_sync(0xFFFFFFFFu, lj, g);
            }
            for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
              for (int g = 0; g < GM; ++g) {
                if constexpr (!kXpose) lrun[g] += __shfl_xor_sync(0xFFFFFFFFu, lrun[g], off);
#pragma unroll
                for (int e = 0; e < V2; ++e) {
                  o[g][e].x += __shfl_xor_sync(0xFFFFFFFFu, o[g][e].x, off);
                  o[g][e].y += __shfl_xor_sync(0xFFFFFFFFu, o[g][e].y, off);
                }
              }
            }
            if (rg == 0 && act) {
#pragma unroll
              for (int g = 0; g < GM; ++g) {
                if (g < G) {
                  if (sgl) {
                    const float inv = lrun[g] > 0.f ? 1.f / lrun[g] : 0.f;
                    *reinterpret_cast<uint4*>(out + ch * GD + g * d + ci * VE) =
                        pack16(o[g], inv, T());
                  } else {
                    float4* dst = reinterpret_cast<float4*>(P + kPartHead + g * d + ci * VE);
#pragma unroll
                    for (int e = 0; e < V2; e += 2)
                      dst[e / 2] =
                          make_float4(o[g][e].x, o[g][e].y, o[g][e + 1].x, o[g][e + 1].y);
                  }
                }
              }
            }
            if (!sgl && lane < G) {
              float mv = mrun[0], lv = lrun[0];
#pragma unroll
              for (int g = 1; g < GM; ++g)
                if (lane == g) {
                  mv = mrun[g];
                  lv = lrun[g];
                }
              P[lane] = mv;
              P[8 + lane] = lv;
            }
          } else if (sgl) {
            // no row of this head at all
            for (int idx = lane * VE; idx < GD; idx += 32 * VE)
              *reinterpret_cast<uint4*>(out + ch * GD + idx) = make_uint4(0u, 0u, 0u, 0u);
          } else if (lane < G) {
            P[lane] = -INFINITY;                 // no row of this head in this chunk
          }
          crem &= crem - 1u;
          cl = crem ? __ffs(crem) - 1 : 32;
          cx = shfl64(lo, cl & 31);
        } else {
          cx += nr;
        }
      }
      if (abort_) {
        // a wait gave up: let the copies that may still be in flight land before leaving
        if (lane == 0)
          for (int s = 0; s < 2; ++s)
            (void)ptx::mbar_wait(&ws.full[s], (phase >> s) & 1u, 20000000ull);
        __syncwarp();
        return;
      }
      if (!more) break;
      hstart += 32;
    }
    c = (int64_t)__shfl_sync(0xFFFFFFFFu, claim, 0) + nworkers;
  }
}

// Merge of the per-chunk partials of every head that spans more than one chunk: one CTA
// per head, each thread four outputs of one query row.  A thread reads (max, sum, o) of
// kCombBatch chunks at once and folds them into a running (max, sum, o), so a head costs
// one round of loads per kCombBatch chunks.  A chunk with no rows of the head has max
// -inf and is skipped (its sum and o were never written).
constexpr int kCombThreads = 128;
constexpr int kCombBatch = 8;
template <typename T>
__global__ void __launch_bounds__(kCombThreads)
decode_combine(const int64_t* __restrict__ cu, const float* __restrict__ part,
               T* __restrict__ out, int Hkv, int G, int d, int64_t cap, int64_t C) {
  ptx::griddep_wait();
  const int64_t h = blockIdx.x;
  const int64_t seg = h / Hkv;
  const int g0 = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g0], end = cu[seg * (Hkv + 1) + g0 + 1];
  const int64_t e = end < cap ? end : cap;
  if (e <= base || base < 0) return;
  const int64_t c0 = base / C, c1 = (e - 1) / C;
  if (c0 == c1) return;                         // finished by the warp that read it
  const int GD = G * d;
  const int64_t stride = kPartHead + (int64_t)GD;
  const float* P0 = part + (c0 + h) * stride;
  const int nsl = (int)(c1 - c0 + 1);
  for (int q4 = threadIdx.x; q4 < GD / 4; q4 += kCombThreads) {
    const int idx = 4 * q4, g = idx / d;
    float M = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < nsl; i0 += kCombBatch) {
      float m[kCombBatch], l[kCombBatch];
      float4 o[kCombBatch];
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u) {
        m[u] = -INFINITY;
        l[u] = 0.f;
        o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i0 + u < nsl) {
          const float* Q = P0 + (i0 + u) * stride;
          m[u] = Q[g];
          l[u] = Q[8 + g];
          o[u] = *reinterpret_cast<const float4*>(Q + kPartHead + idx);
        }
      }
      float Mn = M;
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u) Mn = fmaxf(Mn, m[u]);
      if (Mn == -INFINITY) continue;
      const float a = ptx::ex2(M - Mn);         // 0 while M is still -inf
      L *= a;
      O.x *= a;
      O.y *= a;
      O.z *= a;
      O.w *= a;
#pragma unroll
      for (int u = 0; u < kCombBatch; ++u) {
        if (m[u] > -INFINITY) {
          const float w = ptx::ex2(m[u] - Mn);
          L = fmaf(l[u], w, L);
          O.x = fmaf(o[u].x, w, O.x);
          O.y = fmaf(o[u].y, w, O.y);
          O.z = fmaf(o[u].z, w, O.z);
          O.w = fmaf(o[u].w, w, O.w);
        }
      }
      M = Mn;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    T* dst = out + h * GD + idx;
    dst[0] = from_f<T>(O.x * inv);
    dst[1] = from_f<T>(O.y * inv);
    dst[2] = from_f<T>(O.z * inv);
    dst[3] = from_f<T>(O.w * inv);
  }
}

DecodePlan decode_plan(const Shape& s) {
  DecodePlan p{};
  const int64_t units = s.units();
  // chunk count the launch aims at (the chunk size follows from the flat capacity): a few
  // chunks per worker warp so that the queue evens out uneven heads
  int64_t target = (int64_t)num_sms() * 32;
  if (target < 4 * units) target = 4 * units;
  p.max_chunks = target;
  p.part_slots = target + units;
  size_t off = kWsHeader;
  p.off_part = off;
  off += align_up((size_t)p.part_slots * (kPartHead + s.G() * s.d) * sizeof(float), 256);
  p.off_map = off;
  off += align_up((size_t)target * sizeof(uint32_t), 256);
  p.off_work = off;
  off += 256;
  // tickets of decode_split (zero between launches): CTAs past the scan, then one per head
  p.off_tick = off;
  off += align_up((size_t)(1 + units) * sizeof(uint32_t), 256);
  p.off_end = off;
  return p;
}

static cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a{};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

template <typename T, int GM, int LPRT>
static cudaError_t launch_attn(const Shape& s, const T* q, const void* kf, const void* vf,
                               const int64_t* cu, const int32_t* lens, const uint32_t* map,
                               uint32_t* work, float* part, T* out,
                               int64_t cap, int64_t C, int64_t nchunks, float c2, WsHeader* hdr,
                               cudaStream_t st) {
  const size_t smem = sizeof(DecSmem);
  auto kern = decode_attn<T, GM, LPRT>;
  // the shared-memory opt-in and the resident CTAs per SM, once per instantiation and device
  // (host work on every call would delay the launches behind it)
  static std::atomic<int> slot[kMaxDevices];
  const int per_sm = per_device(slot, [&]() {
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess)
      return 0;
    return n;
  });
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
  int64_t grid = (int64_t)per_sm * num_sms();
  const int64_t need = cdiv(nchunks, kWarps);
  if (grid > need) grid = need;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, (const T*)kf, (const T*)vf, cu, lens, map, work,
                            part, out, s.units(), s.Hkv, s.G(), s.d, cap, C, nchunks, c2, hdr);
}

template <typename T, int LPRT>
static cudaError_t launch_attn_l(const Shape& s, const T* q, const void* kf, const void* vf,
                                 const int64_t* cu, const int32_t* lens, const uint32_t* map,
                                 uint32_t* work, float* part, T* out,
                                 int64_t cap, int64_t C, int64_t nchunks, float c2,
                                 WsHeader* hdr, cudaStream_t st) {
  // group sizes are rounded up to 1, 2, 4 or 8 query heads per KV head
  const int G = s.G();
  switch (G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8) {
    case 1:
      return launch_attn<T, 1, LPRT>(s, q, kf, vf, cu, lens, map, work, part, out, cap, C,
                                     nchunks, c2, hdr, st);
    case 2:
      return launch_attn<T, 2, LPRT>(s, q, kf, vf, cu, lens, map, work, part, out, cap, C,
                                     nchunks, c2, hdr, st);
    case 4:
      return launch_attn<T, 4, LPRT>(s, q, kf, vf, cu, lens, map, work, part, out, cap, C,
                                     nchunks, c2, hdr, st);
    default:
      return launch_attn<T, 8, LPRT>(s, q, kf, vf, cu, lens, map, work, part, out, cap, C,
                                     nchunks, c2, hdr, st);
  }
}

template <typename T>
static cudaError_t launch_attn_g(const Shape& s, const T* q, const void* kf, const void* vf,
                                 const int64_t* cu, const int32_t* lens, const uint32_t* map,
                                 uint32_t* work, float* part, T* out,
                                 int64_t cap, int64_t C, int64_t nchunks, float c2,
                                 WsHeader* hdr, cudaStream_t st) {
  // 256-byte rows (bf16 d = 128, fp32 d = 64): 16 lanes per row, fixed at compile time
  cudaError_t e;
  if (s.d * (int)sizeof(T) == 256)
    e = launch_attn_l<T, 16>(s, q, kf, vf, cu, lens, map, work, part, out, cap, C, nchunks, c2,
                             hdr, st);
  else
    e = launch_attn_l<T, 0>(s, q, kf, vf, cu, lens, map, work, part, out, cap, C, nchunks, c2,
                            hdr, st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)s.units());
  cfg.blockDim = dim3(kCombThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine<T>, cu, (const float*)part, out, s.Hkv, s.G(),
                            s.d, cap, C);
}

// KVEVICT_DECODE_PATH=rows forces the row-balanced split of this file for every shape,
// =heads the one-CTA-per-head kernel, =split the one-launch split and =parts the short heads
// in parts wherever their row size, group and head count allow, whatever the head lengths
// (tests compare the decode paths).
static int decode_path_forced() {
  const char* e = std::getenv("KVEVICT_DECODE_PATH");
  if (e == nullptr) return 0;
  if (std::strcmp(e, "rows") == 0) return 1;
  if (std::strcmp(e, "heads") == 0) return 2;
  if (std::strcmp(e, "split") == 0) return 3;
  if (std::strcmp(e, "parts") == 0) return 4;
  return 0;
}

cudaError_t launch_decode(const Shape& s, const void* q, const void* kn, const void* vn,
                          void* kf, void* vf, const int64_t* cu, int32_t* lens, int64_t cap,
                          float scale, void* out, char* ws, const DecodePlan& p,
                          cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t H = s.units();
  const int forced = decode_path_forced();
  // Measured on GB300 (log-normal head lengths, the cache cold in L2): while the heads fit
  // one wave and are short (every kernel is latency-bound there), the heads in parts (one
  // CTA per head, the rows of the longest spread over the CTAs left) match one CTA per head
  // on even heads and stay flat on skewed ones, where one CTA per head waits on its longest
  // head; the parts kernel also takes calls of a few heads (one layer at a time), whose
  // lengths the capacity does not bound.  The one-launch split wins from there to about
  // 1.5K rows per head, and to about 8K when the heads are few; heads longer still stream
  // best through the row-balanced split.
  const int64_t rows_per_head = cap / H;
  const bool few_heads = H <= 2 * (int64_t)num_sms();
  const bool one_layer = H <= (int64_t)num_sms() / 4;
  if (forced == 0) {
    if (((few_heads && rows_per_head <= kDecodeHeadShortRows) || one_layer) &&
        decode_parts_supported(s, cap, p.part_slots))
      return launch_decode_parts(s, q, kn, vn, kf, vf, cu, lens, cap, scale, out,
                                 reinterpret_cast<float*>(ws + p.off_part), p.part_slots,
                                 reinterpret_cast<uint32_t*>(ws + p.off_tick), hdr, st);
    if (few_heads && rows_per_head <= kDecodeHeadShortRows && decode_head_supported(s, cap))
      return launch_decode_head(s, q, kn, vn, kf, vf, cu, lens, cap, scale, out, hdr, st);
    if ((rows_per_head <= kDecodeSplitRowsMax ||
         (few_heads && rows_per_head <= kDecodeSplitFewRowsMax) || one_layer) &&
        decode_split_supported(s, cap))
      return launch_decode_split(s, q, kn, vn, kf, vf, cu, lens, cap, scale, out,
                                 reinterpret_cast<float*>(ws + p.off_part), p.part_slots,
                                 reinterpret_cast<uint32_t*>(ws + p.off_tick), hdr, st);
  } else if (forced == 4 && decode_parts_supported(s, cap, p.part_slots)) {
    return launch_decode_parts(s, q, kn, vn, kf, vf, cu, lens, cap, scale, out,
                               reinterpret_cast<float*>(ws + p.off_part), p.part_slots,
                               reinterpret_cast<uint32_t*>(ws + p.off_tick), hdr, st);
  } else if (forced == 3 && decode_split_supported(s, cap)) {
    return launch_decode_split(s, q, kn, vn, kf, vf, cu, lens, cap, scale, out,
                               reinterpret_cast<float*>(ws + p.off_part), p.part_slots,
                               reinterpret_cast<uint32_t*>(ws + p.off_tick), hdr, st);
  }
  if (forced != 1 && decode_head_supported(s, forced >= 2 ? 0 : cap))
    return launch_decode_head(s, q, kn, vn, kf, vf, cu, lens, cap, scale, out, hdr, st);
  const int row_bytes = s.d * s.esize();
  const int Ct = kStageBytes / row_bytes;
  int64_t C = cdiv(cap, p.max_chunks);
  if (C < (int64_t)kItemsPerChunkMin * Ct) C = (int64_t)kItemsPerChunkMin * Ct;
  C = cdiv(C, Ct) * Ct;
  const int64_t nchunks = cap > 0 ? cdiv(cap, C) : 0;
  uint32_t* map = reinterpret_cast<uint32_t*>(ws + p.off_map);
  uint32_t* work = reinterpret_cast<uint32_t*>(ws + p.off_work);
  float* part = reinterpret_cast<float*>(ws + p.off_part);
  decode_prep<<<(unsigned)cdiv(H, kPrepWarps), kPrepWarps * 32, 0, st>>>(
      (const char*)kn, (const char*)vn, (char*)kf, (char*)vf, cu, lens, map, work,
      (char*)out, H, s.Hkv, row_bytes, s.G() * s.d * s.esize(), cap, C, nchunks, hdr);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || nchunks == 0) return e;
  const float c2 = scale * 1.4426950408889634f;
  if (s.dtype == KV_BF16)
    e = launch_attn_g<__nv_bfloat16>(s, (const __nv_bfloat16*)q, kf, vf, cu, lens, map, work,
                                     part, (__nv_bfloat16*)out, cap, C, nchunks, c2, hdr, st);
  else
    e = launch_attn_g<float>(s, (const float*)q, kf, vf, cu, lens, map, work, part,
                             (float*)out, cap, C, nchunks, c2, hdr, st);
  if (e == cudaSuccess) count_launches(2);
  return e;
}

}  // namespace kv
