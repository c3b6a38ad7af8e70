// Observation-window scoring on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Ada-KV Algorithm 2 (scoring steps) with the LAVa Definition 1 factor and GQA group
// reduction, for bf16, d = 128 and G*w = 128 window rows per KV head (w in {16, 32, 64}).
//
// Work decomposition.  A (sequence, layer, KV head) "unit" has n keys in T_u tiles of 128.
// The grid (one CTA per SM, cooperative launch so all CTAs are resident) is split into NG
// groups of P_g CTAs; group g handles units g, g+NG, ...; inside a group CTA r owns the
// same contiguous tile range [t0, t1) of every unit.  For each unit a CTA runs
//   P1: S = Q_win K^T on the tensor core (M = 128 window rows, N = 128 keys), online row
//       max / sum of exp2 over its keys -> one (max, sum) partial per row; the CTA that
//       completes the unit's last partial combines them into the row log-sum-exp and
//       publishes it (release flag);
//   P2: S^T = K Q_win^T (M = 128 keys, N = 128 window rows): each epilogue thread owns one
//       key and forms a[q, j] = (1/w) sum_t exp2(z2 - lse2[q,t]); then max-pool, group
//       mean/max and the LAVa V-bar factor.
// Items are ordered P1(u0), P1(u1), P2(u0), P1(u2), P2(u1), ... so a CTA's P2 of unit u
// re-reads its K tiles from L2 after one unit of other traffic, and rarely waits for the
// flag.  Keys whose pooling window crosses a CTA's range boundary are finished by
// score_tc_fixup (score_fixup.cu) from per-range halo copies of the window means.
//
// LAVa: during P2 items (K then comes from L2) the producer also puts the V tiles of the
// range into the ring; a warpgroup of its own folds each one into max ||V[k]||_1 of the
// unit (one row per thread).  P2 writes unscaled scores and the fix-up kernel applies the
// factor after the kernel, so nothing here waits for V.
//
// Roles (768 threads): warp 0 = TMA producer, warp 1 = MMA issuer, warp 2 = TMEM
// allocator, warp 3 = LSE agent, warps 4..19 = epilogue (TMEM lane quadrant = warp % 4,
// column quarter = (warp - 4) / 4), warps 20..23 = LAVa V rows.  Every wait is bounded; on a
// timeout the CTA records DEV_WAIT_TIMEOUT, unwinds, waits (bounded) for its copies and MMAs
// in flight and frees its TMEM.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kv_internal.cuh"
#include "tc_ptx.cuh"

namespace kv {
namespace {

using namespace ptx;

constexpr int kStages = 4;
constexpr int kEpiWarps = 16;                      // 4 TMEM lane quadrants x 4 column quarters
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kVWarps = 4;                         // LAVa V-row reducers (one warpgroup)
constexpr int kThreads = 32 * (4 + kEpiWarps + kVWarps);
constexpr uint32_t kBoxBytes = 128 * 128;          // 128 rows x 64 bf16 (one 128-byte row each)
constexpr uint32_t kTileBytes = 2 * kBoxBytes;     // 128 rows x 128 bf16
constexpr int kAFloats = 6144;                     // window sums of one range, all slots
constexpr int kTBuf = 4;                           // TMEM accumulators of 128 fp32 columns
constexpr uint32_t kTmemCols = 128 * kTBuf;
constexpr int kMaxR = 15;                          // pool / 2
#ifndef KV_TC_LAG
#define KV_TC_LAG 1
#endif

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 2 * kTileBytes;
constexpr uint32_t kOffA = kOffK + kStages * kTileBytes;
constexpr uint32_t kOffLse = kOffA + kAFloats * 4;
constexpr uint32_t kOffPart = kOffLse + 128 * 4;
constexpr uint32_t kOffTail = kOffPart + 4 * 128 * 8;

struct __align__(8) Tail {
  // A ring stage holds either a K tile (consumed by the MMA warp) or, in LAVa P2 items, a
  // V tile (consumed by warp 2).  Each kind completes its own barrier so that no consumer
  // ever has to skip a phase of the barrier it waits on (skipped phases alias in parity).
  uint64_t full[kStages], fullv[kStages], empty[kStages];
  uint64_t qfull[2], qempty[2];
  uint64_t tfull[kTBuf], tempty[kTBuf];
  uint64_t drain;
  uint64_t afull, aempty;   // window sums ready for pooling / pooled (A free again)
  uint32_t vcnt[kStages];  // epilogue warps done with the V entry in each stage
  int64_t pf_unit;      // unit whose -lse already sits in the nlse buffer (-1: none)
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
};
constexpr uint32_t kSmemBytes = kOffTail + sizeof(Tail) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

struct TcParams {
  int n, w, C, G, r, group_max;
  // terms != 0: every query head's term instead of the KV head's score, into
  // scores[units][G][C]: 1 = pooled window mean, 2 = sqrt(sum_t P^2) (r = 0, esc = 2: pass 2
  // then exponentiates twice the log-probability, i.e. forms P^2, and inv_w is 1)
  int terms;
  float esc;
  int64_t units;
  int Pg, PgS, NG, Tu, Tc;
  int ncomb;            // CTAs that combine one unit's partials (power of two <= 16)
  float c2, inv_w;
  float* vbar;        // LAVa: per-unit max ||V[k]||_1 (float bits, atomicMax), else null
  float2* partial;   // [units][128][PgS], PgS = Pg rounded up to even (padding unread)
  float* lse;        // [units][128] (log2 domain)
  uint32_t* done1;   // [units] P1 partials written
  uint32_t* ready;   // [units] LSE row slices published (complete at ncomb)
  float* halo;       // [units][Pg][G][4r]
  float* scores;     // [units][C]
  WsHeader* hdr;
};

// L1 norm of row `row` of a V tile in the ring (128 rows x 128 bf16, two 128-byte swizzled
// boxes).  A row's sum does not depend on the order of its 16-byte pieces, so thread t reads
// physical piece (j + t) % 8 of each box at step j: the 8 threads of a shared-memory phase
// (8 consecutive rows) then hit 8 different bank groups.
__device__ __forceinline__ float vrow_l1_row(const uint8_t* base, int row) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int bx = 0; bx < 2; ++bx) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int pc = (j + row) & 7;
      const uint4 x =
          *reinterpret_cast<const uint4*>(base + bx * kBoxBytes + row * 128 + pc * 16);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        a0 += fabsf(f.x);
        a1 += fabsf(f.y);
      }
    }
  }
  return a0 + a1;
}

// Max-pool over the window means of one range, group reduction, scores of the keys whose
// pooling window lies inside the range, and the halo copies for the fix-up of the others.
// A holds the window sums of keys [sK, eK) (see the epilogue); tid / nthr are this thread's
// index and the number of threads (a multiple of 32) that share the work.
template <int LW>
__device__ __forceinline__ void pool_range(const float* A, int RK, int sK, int eK, int C, int G,
                                           int r, int group_max, float inv_w, int terms,
                                           float* S, float* H, int tid, int nthr) {
  // window mean of query head q at key j (slots hold per-quarter sums for w = 64)
  auto aval = [&](int q, int j) -> float {
    if (LW <= 5) return A[q * RK + (j - sK)];
    return (A[(2 * q) * RK + (j - sK)] + A[(2 * q + 1) * RK + (j - sK)]) * inv_w;
  };
  if (r == 3) {
    // pool 7: one thread per (run of 8 keys, query head); the window maximum is
    // max(max of 4, max of 2, 1) over values loaded once (-inf outside the range);
    // the G query heads of a run sit in adjacent lanes and are combined by shuffles.
    constexpr int RUN = 8;
    const int qh = tid & (G - 1), run = tid / G;
    const int nruns = (eK - sK + RUN - 1) / RUN;
    const int stride = nthr / G;
    for (int rr = run; rr < nruns + (stride - nruns % stride) % stride; rr += stride) {
      const bool live = rr < nruns;
      const int j0 = sK + rr * RUN;
      float v[RUN + 6];
#pragma unroll
      for (int i = 0; i < RUN + 6; ++i) {
        const int jj = j0 - 3 + i;
        v[i] = (live && jj >= sK && jj < eK) ? aval(qh, jj) : -INFINITY;
      }
      float m2[RUN + 5], out[RUN];
#pragma unroll
      for (int i = 0; i < RUN + 5; ++i) m2[i] = fmaxf(v[i], v[i + 1]);
#pragma unroll
      for (int i = 0; i < RUN; ++i)
        out[i] = fmaxf(fmaxf(fmaxf(m2[i], m2[i + 2]), m2[i + 4]), v[i + 6]);
      if (terms) {   // every query head's pooled mean, no group reduction
        if (live) {
#pragma unroll
          for (int i = 0; i < RUN; ++i) {
            const int j = j0 + i;
            if (j >= eK) break;
            const int lo = max(0, j - 3), hi = min(C - 1, j + 3);
            if (lo >= sK && hi < eK) S[(int64_t)qh * C + j] = out[i];
          }
        }
        continue;
      }
#pragma unroll
      for (int i = 0; i < RUN; ++i) {
        float gv = out[i];
        for (int o = 1; o < G; o <<= 1) {
          const float x = __shfl_xor_sync(0xffffffffu, gv, o);
          gv = group_max ? fmaxf(gv, x) : gv + x;
        }
        out[i] = group_max ? gv : gv / (float)G;
      }
      if (live && qh == 0) {
#pragma unroll
        for (int i = 0; i < RUN; ++i) {
          const int j = j0 + i;
          if (j >= eK) break;
          const int lo = max(0, j - 3), hi = min(C - 1, j + 3);
          if (lo >= sK && hi < eK) S[j] = out[i];
        }
      }
    }
  } else if (terms) {
    for (int idx = tid; idx < G * (eK - sK); idx += nthr) {
      const int q = idx / (eK - sK), j = sK + (idx - q * (eK - sK));
      const int lo = max(0, j - r), hi = min(C - 1, j + r);
      if (lo >= sK && hi < eK) {
        float pm = -INFINITY;
        for (int jj = lo; jj <= hi; ++jj) pm = fmaxf(pm, aval(q, jj));
        S[(int64_t)q * C + j] = terms == 2 ? sqrtf(pm) : pm;
      }
    }
  } else {
    for (int j = sK + tid; j < eK; j += nthr) {
      const int lo = max(0, j - r), hi = min(C - 1, j + r);
      if (lo >= sK && hi < eK) {
        float gv = group_max ? -INFINITY : 0.f;
        for (int q = 0; q < G; ++q) {
          float pm = -INFINITY;
          for (int jj = lo; jj <= hi; ++jj) pm = fmaxf(pm, aval(q, jj));
          gv = group_max ? fmaxf(gv, pm) : gv + pm;
        }
        if (!group_max) gv = gv / (float)G;
        S[j] = gv;
      }
    }
  }
  if (r > 0) {   // halo copies for the fix-up of keys near the range's ends
    for (int idx = tid; idx < G * 4 * r; idx += nthr) {
      const int q = idx / (4 * r), sl = idx % (4 * r);
      const int j = sl < 2 * r ? sK + sl : eK - 2 * r + (sl - 2 * r);
      if (j >= sK && j < eK) H[q * 4 * r + sl] = aval(q, j);
    }
  }
}

// P2 of the k-th unit follows P1 of the (k + kLag)-th: P1(0..a-1), then P1(k), P2(k-a) pairs,
// then the last P2s, with a = min(kLag, m).  kind 1 = P1, 2 = P2.
constexpr int kLag = KV_TC_LAG;
__device__ __forceinline__ void item_of(int64_t i, int64_t m, int& kind, int64_t& k) {
  const int64_t a = m < kLag ? m : kLag;
  if (i < a) { kind = 1; k = i; return; }
  const int64_t j = i - a;
  if (j < 2 * (m - a)) {
    if ((j & 1) == 0) { kind = 1; k = a + (j >> 1); } else { kind = 2; k = j >> 1; }
    return;
  }
  kind = 2;
  k = m - a + (j - 2 * (m - a));
}

template <int LW>
__global__ void __launch_bounds__(kThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                const __grid_constant__ CUtensorMap vmap, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Tail* tl = reinterpret_cast<Tail*>(smem + kOffTail);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = blockIdx.x / p.Pg, rank = blockIdx.x % p.Pg;
  const int t0 = (int)(((int64_t)rank * p.Tu) / p.Pg);
  const int t1 = (int)(((int64_t)(rank + 1) * p.Tu) / p.Pg);
  const int t1c = t1 < p.Tc ? t1 : p.Tc;
  const int64_t m = group < p.units ? (p.units - 1 - group) / p.NG + 1 : 0;
  const int64_t n_items = 2 * m;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tl->full[s], 1);
      mbar_init(&tl->fullv[s], 1);
      mbar_init(&tl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tl->qfull[b], 1);
      mbar_init(&tl->qempty[b], 1);
    }
    for (int b = 0; b < kTBuf; ++b) {
      mbar_init(&tl->tfull[b], 1);
      mbar_init(&tl->tempty[b], kEpiWarps);
    }
    mbar_init(&tl->drain, 1);
    mbar_init(&tl->afull, 1);
    mbar_init(&tl->aempty, kVWarps);
    for (int st = 0; st < kStages; ++st) tl->vcnt[st] = 0;
    tl->abort_flag = 0;
    tl->last_flag = 0;
    tl->pf_unit = -1;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&tl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&qmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort_flag = &tl->abort_flag;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      uint32_t g = 0, qi = 0;
      uint32_t kfill[kStages] = {}, vfill[kStages] = {};  // copies per stage and kind
      bool lastv[kStages] = {};                           // kind of each stage's last copy
      uint32_t qissued[2] = {};                           // 1 + use index of the last Q copy
      // P1 keeps its K tiles in L2 for the P2 re-read one unit later; P2 lets them go.
      const uint64_t keep = make_policy_evict_last(), drop = make_policy_evict_first();
      bool ok = true;
      for (int64_t i = 0; i < n_items && ok; ++i) {
        int kind;
        int64_t k;
        item_of(i, m, kind, k);
        const int64_t u = group + k * p.NG;
        const int te = kind == 1 ? t1 : t1c;
        if (t0 >= te) continue;
        const int qb = qi & 1;
        if (!mbar_wait(&tl->qempty[qb], ((qi >> 1) & 1) ^ 1) || *abort_flag) { ok = false; break; }
        qissued[qb] = (qi >> 1) + 1;
        mbar_arrive_expect_tx(&tl->qfull[qb], kTileBytes);
        tma_load_3d_hint(smem + kOffQ + qb * kTileBytes, &qmap, &tl->qfull[qb], 0, 0, (int)u,
                         kind == 1 ? keep : drop);
        tma_load_3d_hint(smem + kOffQ + qb * kTileBytes + kBoxBytes, &qmap, &tl->qfull[qb], 64, 0,
                         (int)u, kind == 1 ? keep : drop);
        const uint64_t pol = kind == 1 ? keep : drop;
        for (int t = t0; t < te; ++t, ++g) {
          const int s = g % kStages;
          if (!mbar_wait(&tl->empty[s], ((g / kStages) & 1) ^ 1) || *abort_flag) { ok = false; break; }
          ++kfill[s];
          lastv[s] = false;
          mbar_arrive_expect_tx(&tl->full[s], kTileBytes);
          tma_load_3d_hint(smem + kOffK + s * kTileBytes, &kmap, &tl->full[s], 0, t * 128, (int)u,
                           pol);
          tma_load_3d_hint(smem + kOffK + s * kTileBytes + kBoxBytes, &kmap, &tl->full[s], 64,
                           t * 128, (int)u, pol);
          // LAVa: the V rows of this tile (and, after the last candidate tile, of the
          // window-only tiles of the range) follow as ring entries that warp 2 consumes
          const int vt_end = (kind == 2 && p.vbar != nullptr) ? (t + 1 < te ? t + 1 : t1) : t;
          for (int vt = t; vt < vt_end && ok; ++vt) {
            ++g;
            const int sv = g % kStages;
            if (!mbar_wait(&tl->empty[sv], ((g / kStages) & 1) ^ 1) || *abort_flag) {
              ok = false;
              break;
            }
            ++vfill[sv];
            lastv[sv] = true;
            mbar_arrive_expect_tx(&tl->fullv[sv], kTileBytes);
            tma_load_3d_hint(smem + kOffK + sv * kTileBytes, &vmap, &tl->fullv[sv], 0, vt * 128,
                             (int)u, drop);
            tma_load_3d_hint(smem + kOffK + sv * kTileBytes + kBoxBytes, &vmap, &tl->fullv[sv], 64,
                             vt * 128, (int)u, drop);
          }
          if (!ok) break;
        }
        ++qi;
      }
      if (!ok) {
        raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 1);
        *abort_flag = 1;
        // let the copies already issued land before the CTA exits: the last copy of each
        // stage is the only phase of its barrier that can still be pending
        for (int s = 0; s < kStages; ++s) {
          if (lastv[s]) mbar_wait(&tl->fullv[s], (vfill[s] - 1) & 1, 20000000ull);
          else if (kfill[s]) mbar_wait(&tl->full[s], (kfill[s] - 1) & 1, 20000000ull);
        }
        for (int b = 0; b < 2; ++b)
          if (qissued[b]) mbar_wait(&tl->qfull[b], (qissued[b] - 1) & 1, 20000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      uint32_t g = 0, gt = 0, qi = 0;   // ring entries (K and V), TMEM accumulators (K)
      uint32_t kuse[kStages] = {};      // K tiles consumed per stage (phases of full[s])
      bool ok = true;
      for (int64_t i = 0; i < n_items && ok; ++i) {
        int kind;
        int64_t k;
        item_of(i, m, kind, k);
        const int te = kind == 1 ? t1 : t1c;
        if (t0 >= te) continue;
        const int qb = qi & 1;
        if (!mbar_wait(&tl->qfull[qb], (qi >> 1) & 1) || *abort_flag) { ok = false; break; }
        const uint32_t qaddr = smem_u32(smem + kOffQ + qb * kTileBytes);
        for (int t = t0; t < te; ++t, ++g, ++gt) {
          const int s = g % kStages, tb = gt % kTBuf;
          if (!mbar_wait(&tl->full[s], kuse[s]++ & 1) ||
              !mbar_wait(&tl->tempty[tb], ((gt / kTBuf) & 1) ^ 1) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kaddr = smem_u32(smem + kOffK + s * kTileBytes);
          const uint32_t d = tmem + tb * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            const uint64_t qd = sdesc_sw128(qaddr + off), kd = sdesc_sw128(kaddr + off);
            if (kind == 1) mma_bf16(d, qd, kd, idesc, kk > 0 ? 1u : 0u);
            else mma_bf16(d, kd, qd, idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&tl->empty[s]);
          mma_commit(&tl->tfull[tb]);
          if (kind == 2 && p.vbar != nullptr) g += (t + 1 < te ? 1 : t1 - t);   // V entries
        }
        if (!ok) break;
        mma_commit(&tl->qempty[qb]);
        ++qi;
      }
      if (!ok) {
        raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 2);
        *abort_flag = 1;
      }
      // every MMA issued has completed before TMEM is freed
      mma_commit(&tl->drain);
      mbar_wait(&tl->drain, 0, 20000000ull);
    }
  } else if (warp == 3) {
    // ------------------------------ LSE agent ---------------------------------
    // For the units it is assigned to (ncomb CTAs per unit, rotating), this warp waits
    // until all P_g partials of the unit are written, merges the partials of its slice of
    // rows into the log-sum-exp and publishes the slice.  It never delays the epilogue.
    const int rpc = 128 / p.ncomb;
    const int nf4 = p.PgS >> 1;                  // float4 (two partials) per row
    for (int64_t k = 0; k < m; ++k) {
      const int ci = (int)(((int64_t)rank - k * p.ncomb) % p.Pg + p.Pg) % p.Pg;
      if (ci >= p.ncomb) continue;
      const int64_t u = group + k * p.NG;
      bool ok = true;
      if (lane == 0) {
        const uint64_t tw = globaltimer();
        while (ld_acquire_u32(&p.done1[u]) < (uint32_t)p.Pg) {
          if (*abort_flag || globaltimer() - tw > 2000000000ull) { ok = false; break; }
          __nanosleep(64);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        if (lane == 0) {
          raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 5);
          *abort_flag = 1;
        }
        break;
      }
      __threadfence();
      for (int rr = 0; rr < rpc; ++rr) {
        const int row = ci * rpc + rr;
        const float4* P4 = reinterpret_cast<const float4*>(p.partial + (u * 128 + row) * p.PgS);
        float M = -INFINITY, S = 0.f;
        constexpr int kV = 4;
        for (int b0 = lane; b0 < nf4; b0 += 32 * kV) {
          float4 v[kV];
#pragma unroll
          for (int j = 0; j < kV; ++j)
            v[j] = b0 + 32 * j < nf4 ? __ldcg(P4 + b0 + 32 * j)
                                    : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
#pragma unroll
          for (int j = 0; j < kV; ++j) {
            const float ms[2] = {v[j].x, v[j].z}, ls[2] = {v[j].y, v[j].w};
            const int q0 = 2 * (b0 + 32 * j);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (q0 + h >= p.Pg || ms[h] == -INFINITY) continue;   // padding / empty
              const float Mn = fmaxf(M, ms[h]);
              S = S * ex2(M - Mn) + ls[h] * ex2(ms[h] - Mn);
              M = Mn;
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
          const float So = __shfl_xor_sync(0xffffffffu, S, o);
          const float Mn = fmaxf(M, Mo);
          float Sn = 0.f;
          if (M != -INFINITY) Sn += S * ex2(M - Mn);
          if (Mo != -INFINITY) Sn += So * ex2(Mo - Mn);
          M = Mn;
          S = Sn;
        }
        if (lane == 0) p.lse[u * 128 + row] = M + log2f(S);
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        atomicAdd(&p.ready[u], 1u);
      }
    }
  } else if (warp >= 4 + kEpiWarps) {
    // ------------------------------ LAVa V rows --------------------------------
    // The V entries the producer puts in the ring during P2 items (K then comes from L2,
    // so the two passes share DRAM evenly): thread t of this warpgroup sums |V| over row t
    // of each V tile, keeps the maximum over the unit's rows in its range, and the last of
    // the four warps done with an entry frees its stage.  The fix-up kernel applies
    // max_k ||V[k]||_1 after this kernel, so nothing here holds the epilogue up.
    {
      const int vt_ = threadIdx.x - 32 * (4 + kEpiWarps);   // V row / pooling thread
      float* A = reinterpret_cast<float*>(smem + kOffA);
      const int RK = (t1 - t0) * 128;
      const bool lava = p.vbar != nullptr;
      uint32_t g = 0, np2 = 0;
      uint32_t vuse[kStages] = {};      // V tiles consumed per stage (phases of fullv[s])
      bool ok = true;
      for (int64_t i = 0; i < n_items && ok; ++i) {
        int kind;
        int64_t k;
        item_of(i, m, kind, k);
        const int te = kind == 1 ? t1 : t1c;
        if (t0 >= te) continue;
        if (kind == 1) { g += te - t0; continue; }
        const int64_t u = group + k * p.NG;
        float vmax = 0.f;
        for (int t = t0; t < te && ok && lava; ++t) {
          ++g;   // the K entry of tile t
          const int nv = t + 1 < te ? 1 : t1 - t;
          for (int j = 0; j < nv; ++j, ++g) {
            const int sv = g % kStages;
            const bool landed = mbar_wait(&tl->fullv[sv], vuse[sv]++ & 1) && !*abort_flag;
            if (landed) vmax = fmaxf(vmax, vrow_l1_row(smem + kOffK + sv * kTileBytes, vt_));
            // the whole warp leaves when any lane's wait gave up; otherwise every lane's
            // reads of the stage are ordered before lane 0 frees it
            if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }
            __syncwarp();
            if (lane == 0 && atomicAdd(&tl->vcnt[sv], 1u) == (uint32_t)(kVWarps - 1)) {
              tl->vcnt[sv] = 0;
              mbar_arrive(&tl->empty[sv]);
            }
          }
        }
        if (!ok) break;
        if (lava) {
          const float wm = warp_max(vmax);
          if (lane == 0 && wm > 0.f)
            atomicMax(reinterpret_cast<unsigned int*>(p.vbar) + u, __float_as_uint(wm));
        }
        // pool the item's window sums once the epilogue has written all of them
        const bool filled = mbar_wait(&tl->afull, np2 & 1) && !*abort_flag;
        if (__any_sync(0xffffffffu, !filled)) { ok = false; break; }   // the whole warp
        ++np2;
        const int sK = t0 * 128, eK = min(te * 128, p.C);
        pool_range<LW>(A, RK, sK, eK, p.C, p.G, p.r, p.group_max, p.inv_w, p.terms,
                       p.scores + u * (int64_t)p.C * (p.terms ? p.G : 1),
                       p.halo + (u * p.Pg + rank) * (int64_t)p.G * 4 * p.r, vt_, 32 * kVWarps);
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->aempty);
      }
      if (!ok && lane == 0) {
        raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 6);
        *abort_flag = 1;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------ epilogue ----------------------------------
    // Warp (4 + 4*qc + quad) reads TMEM lanes [32*quad, 32*quad + 32) and columns
    // [32*qc, 32*qc + 32) of each accumulator.
    constexpr int W = 1 << LW;
    constexpr int SL = LW <= 5 ? (32 >> LW) : 1;   // window-sum slots per column quarter
    constexpr int NSLOT = 4 * SL;                   // slots of all quarters (G or 2G)
    const int quad = warp & 3, qc = (warp - 4) >> 2, et = threadIdx.x - 128;
    const int row = quad * 32 + lane;              // P1: window row; P2: key within the tile
    float* A = reinterpret_cast<float*>(smem + kOffA);
    float* nlse = reinterpret_cast<float*>(smem + kOffLse);
    float2* part_s = reinterpret_cast<float2*>(smem + kOffPart);
    const int RK = (t1 - t0) * 128;                // keys of this CTA's range (A stride)
    const float c2 = p.c2;
    uint32_t g = 0;     // TMEM accumulator counter (K tiles)
    uint32_t np2 = 0;   // P2 items finished (phases of afull / aempty)
    // ok turns false on a wait that gave up or an abort by another role.  The thread then
    // raises the CTA's abort flag, stops waiting and skips the rest of each item's tiles,
    // but keeps to the same sequence of items and named barriers as the other epilogue
    // threads (leaving the item loop early would strand them at a barrier).
    bool ok = true;
    for (int64_t i = 0; i < n_items; ++i) {
      int kind;
      int64_t k;
      item_of(i, m, kind, k);
      const int64_t u = group + k * p.NG;
      const int te = kind == 1 ? t1 : t1c;
      if (t0 >= te) continue;
      if (kind == 2) {
        // the window sums of the previous P2 item have been pooled
        if (*abort_flag || !mbar_wait(&tl->aempty, (np2 & 1) ^ 1)) {
          ok = false;
          *abort_flag = 1;
        }
        if (tl->pf_unit != u) {     // not prefetched during the previous P1 item: wait now
          if (et == 0 && !*abort_flag) {
            const uint64_t tw = globaltimer();
            while (ld_acquire_u32(&p.ready[u]) < (uint32_t)p.ncomb) {
              if (*abort_flag || globaltimer() - tw > 2000000000ull) {
                raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 3);
                *abort_flag = 1;
                break;
              }
              __nanosleep(64);
            }
          }
          named_bar(1, kEpiThreads);
          if (et < 128) nlse[et] = -__ldcg(&p.lse[u * 128 + et]) * p.esc;
        }
        named_bar(1, kEpiThreads);
      }
      // During a P1 item, warp 4 watches for the LSE of the P2 item that comes next and
      // stages it in nlse, so that item rarely has to wait.
      int64_t pf_u = -1;
      if (kind == 1 && warp == 4 && i + 1 < n_items) {
        int k2kind;
        int64_t k2;
        item_of(i + 1, m, k2kind, k2);
        if (k2kind == 2 && t0 < t1c) pf_u = group + k2 * p.NG;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = t0; t < te; ++t, ++g) {
        const int tb = g % kTBuf;
        uint32_t pf_flag = 0;
        if (pf_u >= 0 && lane == 0) pf_flag = ld_relaxed_u32(&p.ready[pf_u]);   // used below
        if (*abort_flag || !mbar_wait(&tl->tfull[tb], (g / kTBuf) & 1)) {
          ok = false;
          *abort_flag = 1;
          break;   // the item's remaining tiles only: its named barriers still follow
        }
        tc_fence_after();
        uint32_t ra[32];
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + tb * 128 + qc * 32, ra);
        tmem_ld_wait(ra);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->tempty[tb]);
        if (kind == 1) {
          const int key0 = t * 128 + qc * 32;
          float v[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(ra[c]);
          if (key0 + 31 > p.n - W) {
            const int limit = p.n - W + (row & (W - 1));   // last key window row t sees
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (key0 + c > limit) v[c] = -INFINITY;
          }
          float mx[11];
#pragma unroll
          for (int j = 0; j < 10; ++j) mx[j] = max3f(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
          mx[10] = fmaxf(v[30], v[31]);
          const float tmax = fmaxf(max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), max3f(mx[6], mx[7], mx[8])), fmaxf(mx[9], mx[10])) * c2;
          const float mn = fmaxf(m_run, tmax);
          if (mn != -INFINITY) {
            const float2 sc = make_float2(c2, c2), sh = make_float2(-mn, -mn);
            float2 sa0 = make_float2(0.f, 0.f), sa1 = sa0;
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const float2 x0 = ffma2(make_float2(v[c], v[c + 1]), sc, sh);
              const float2 x1 = ffma2(make_float2(v[c + 2], v[c + 3]), sc, sh);
              sa0 = fadd2(sa0, make_float2(ex2(x0.x), ex2(x0.y)));
              sa1 = fadd2(sa1, make_float2(ex2(x1.x), ex2(x1.y)));
            }
            const float2 st = fadd2(sa0, sa1);
            l_run = l_run * ex2(m_run - mn) + (st.x + st.y);
            m_run = mn;
          }
        } else {
          constexpr int CPS = 32 / SL;              // columns per slot
          float acc[SL];
#pragma unroll
          for (int j = 0; j < SL; ++j) acc[j] = 0.f;
          const float2* nl2 = reinterpret_cast<const float2*>(nlse + qc * 32);
          const float2 sc = make_float2(c2 * p.esc, c2 * p.esc);
#pragma unroll
          for (int j = 0; j < SL; ++j) {
            float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll
            for (int c = j * CPS; c < (j + 1) * CPS; c += 4) {
              const float2 x0 = ffma2(make_float2(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), sc, nl2[c / 2]);
              const float2 x1 = ffma2(make_float2(__uint_as_float(ra[c + 2]), __uint_as_float(ra[c + 3])), sc, nl2[c / 2 + 1]);
              s0 = fadd2(s0, make_float2(ex2(x0.x), ex2(x0.y)));
              s1 = fadd2(s1, make_float2(ex2(x1.x), ex2(x1.y)));
            }
            const float2 st = fadd2(s0, s1);
            acc[j] += st.x + st.y;
          }
          const int kl = (t - t0) * 128 + row;
#pragma unroll
          for (int j = 0; j < SL; ++j)
            A[(qc * SL + j) * RK + kl] = LW <= 5 ? acc[j] * p.inv_w : acc[j];
        }
        if (pf_u >= 0) {
          if (__shfl_sync(0xffffffffu, pf_flag, 0) >= (uint32_t)p.ncomb) {
            __threadfence();
            const float4 l4 = __ldcg(reinterpret_cast<const float4*>(p.lse + pf_u * 128) + lane);
            const float e = p.esc;
            reinterpret_cast<float4*>(nlse)[lane] =
                make_float4(-l4.x * e, -l4.y * e, -l4.z * e, -l4.w * e);
            __syncwarp();
            if (lane == 0) tl->pf_unit = pf_u;
            pf_u = -1;
          }
        }
      }
      if (kind == 1) {
        part_s[qc * 128 + row] = make_float2(m_run, l_run);
        named_bar(1, kEpiThreads);
        if (et < 128) {
          float M = -INFINITY;
#pragma unroll
          for (int j = 0; j < 4; ++j) M = fmaxf(M, part_s[j * 128 + et].x);
          float L = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 a = part_s[j * 128 + et];
            if (a.x != -INFINITY) L += a.y * ex2(a.x - M);
          }
          p.partial[(u * 128 + et) * p.PgS + rank] = make_float2(M, L);
        }
        named_bar(1, kEpiThreads);
        if (et == 0) {
          __threadfence();   // cumulative: the partials written above become visible first
          atomicAdd(&p.done1[u], 1u);
        }
        named_bar(1, kEpiThreads);     // part_s is free for the next item
      } else {
        // every epilogue warp has written its window sums: the V warpgroup pools them while
        // the epilogue goes on with the next item
        named_bar(1, kEpiThreads);
        if (et == 0) {
          tl->pf_unit = -1;
          mbar_arrive(&tl->afull);
        }
        ++np2;
        named_bar(1, kEpiThreads);
      }
      (void)NSLOT;
    }
    if (!ok) {
      raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 4);
      *abort_flag = 1;
    }
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------- host side ----------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t units,
              uint32_t box_rows = 128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {128, rows, units};
  const cuuint64_t strides[2] = {128 * 2, rows * 128 * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int path_override() {
  const char* e = std::getenv("KVEVICT_SCORE_PATH");
  if (e == nullptr) return 0;
  if (std::strcmp(e, "simt") == 0) return 1;
  if (std::strcmp(e, "tc") == 0) return 2;
  return 0;
}

struct TcPlan {
  int NG, Pg, Tu, Tc, grid;
  size_t off_partial, off_lse, off_flags, off_halo, off_vbar, off_end;
};

bool tc_plan(const Shape& s, TcPlan* out) {
  if (s.dtype != KV_BF16 || s.d != 128 || s.R() != 128) return false;
  if (!(s.w == 16 || s.w == 32 || s.w == 64)) return false;
  if (s.C() < 1 || s.pool / 2 > kMaxR) return false;
  TcPlan p{};
  const int P = num_sms();
  p.Tu = (int)cdiv(s.n, 128);
  p.Tc = (int)cdiv(s.C(), 128);
  const int64_t units = s.units();
  const int slots = s.w <= 32 ? 4 * (32 / s.w) : 4;   // window-sum slots per key
  const int max_tiles = kAFloats / (slots * 128);
  // groups: each keeps about two units of K in L2 (about 64 MiB per group in total)
  const double unit_bytes = (double)s.n * 128 * 2;
  int NG = (int)(64.0 * 1024 * 1024 / (2.0 * unit_bytes));
  if (NG < 1) NG = 1;
  if (NG > P) NG = P;
  if (NG > units) NG = (int)units;
  int Pg = P / NG;
  // every range holds at least one candidate tile (so its P2 item streams all its V rows)
  if (Pg > p.Tc) Pg = p.Tc;
  if (cdiv(p.Tu, Pg) > max_tiles) {
    // ranges too long for the window-mean buffer: use more CTAs per unit
    Pg = (int)cdiv(p.Tu, max_tiles);
    if (Pg > P) return false;
    NG = P / Pg;
    if (NG > units) NG = (int)units;
  }
  p.NG = NG;
  p.Pg = Pg;
  p.grid = NG * Pg;
  const int r = s.pool / 2;
  size_t off = kWsHeader;
  p.off_partial = off;
  off += align_up((size_t)units * ((Pg + 1) & ~1) * 128 * sizeof(float2), 256);
  p.off_lse = off;
  off += align_up((size_t)units * 128 * sizeof(float), 256);
  p.off_flags = off;
  off += align_up((size_t)units * 3 * sizeof(uint32_t), 256);
  p.off_halo = off;
  off += align_up((size_t)units * Pg * s.G() * 4 * r * sizeof(float) + 4, 256);
  p.off_vbar = off;
  off += align_up((size_t)units * sizeof(float), 256);
  p.off_end = off;
  *out = p;
  return true;
}

template <int LW>
cudaError_t launch_main(const CUtensorMap& km, const CUtensorMap& qm, const CUtensorMap& vm,
                        const TcParams& prm, int grid, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<LW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, score_tc_kernel<LW>, km, qm, vm, prm);
}

}  // namespace

bool score_tc_supported(const Shape& s) {
  const int ov = path_override();
  if (ov == 1) return false;
  TcPlan p;
  if (!tc_plan(s, &p)) return false;
  return encode_fn() != nullptr;
}

size_t score_tc_ws(const Shape& s, int) {
  TcPlan p;
  if (!tc_plan(s, &p)) return 0;
  return p.off_end;
}

cudaError_t launch_score_tc(const Shape& s, int mode, int group, const void* q_win,
                            const void* k, const void* v, float* scores, char* ws,
                            cudaStream_t st, int terms) {
  TcPlan tp;
  if (!tc_plan(s, &tp)) return cudaErrorNotSupported;
  const int64_t units = s.units();
  CUtensorMap km, qm, vm;
  if (!make_map(&km, k, (uint64_t)s.n, (uint64_t)units) ||
      !make_map(&qm, q_win, 128, (uint64_t)units))
    return cudaErrorInvalidValue;
  // V is only read for LAVa; otherwise the map is a copy of K's and never used.
  if (mode == KV_SCORE_LAVA) {
    if (!make_map(&vm, v, (uint64_t)s.n, (uint64_t)units)) return cudaErrorInvalidValue;
  } else {
    vm = km;
  }
  TcParams prm{};
  prm.n = s.n;
  prm.w = s.w;
  prm.C = s.C();
  prm.G = s.G();
  prm.r = terms == 2 ? 0 : s.pool / 2;
  prm.group_max = group == KV_GROUP_MAX;
  prm.terms = terms;
  prm.esc = terms == 2 ? 2.0f : 1.0f;
  prm.units = units;
  prm.Pg = tp.Pg;
  prm.PgS = (tp.Pg + 1) & ~1;
  prm.ncomb = 1;
  while (prm.ncomb * 2 <= 16 && prm.ncomb * 2 <= tp.Pg) prm.ncomb *= 2;
  prm.NG = tp.NG;
  prm.Tu = tp.Tu;
  prm.Tc = tp.Tc;
  prm.c2 = (1.0f / sqrtf((float)s.d)) * 1.4426950408889634f;
  prm.inv_w = terms == 2 ? 1.0f : 1.0f / (float)s.w;
  prm.partial = reinterpret_cast<float2*>(ws + tp.off_partial);
  prm.lse = reinterpret_cast<float*>(ws + tp.off_lse);
  prm.done1 = reinterpret_cast<uint32_t*>(ws + tp.off_flags);
  prm.ready = prm.done1 + units;
  prm.halo = reinterpret_cast<float*>(ws + tp.off_halo);
  prm.scores = scores;
  prm.hdr = reinterpret_cast<WsHeader*>(ws);
  cudaError_t e = cudaMemsetAsync(prm.done1, 0, (size_t)units * 3 * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;

  if (mode == KV_SCORE_LAVA) {
    float* vbar = reinterpret_cast<float*>(ws + tp.off_vbar);
    e = cudaMemsetAsync(vbar, 0, (size_t)units * sizeof(float), st);
    if (e != cudaSuccess) return e;
    prm.vbar = vbar;
  }
  switch (s.w) {
    case 16: e = launch_main<4>(km, qm, vm, prm, tp.grid, st); break;
    case 32: e = launch_main<5>(km, qm, vm, prm, tp.grid, st); break;
    default: e = launch_main<6>(km, qm, vm, prm, tp.grid, st); break;
  }
  if (e != cudaSuccess) return e;
  count_launches(1);
  if (prm.vbar != nullptr || (prm.r > 0 && tp.Pg > 1)) {
    e = launch_score_fixup(prm.halo, prm.vbar, units, tp.Pg, tp.Tu, prm.C, prm.G, prm.r,
                           prm.group_max, terms, scores, st);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace kv
