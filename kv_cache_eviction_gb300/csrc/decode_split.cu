// One decode step of attention over the flat cache with every CTA given the same number of
// rows, whatever the heads' lengths.
//
// Ada-KV formal model: the new token's k, v are appended to its head's cache, then
// A = softmax(q K^T / sqrt(d)) and o = A V per query head, over the uneven per-head lengths
// of the flat layout.
//
// After head-adaptive allocation a few heads hold most of the rows, so one CTA per head
// waits on its longest head, and a row-balanced split built from several dependent
// launches spends more time in launch latency than in reading a cache of a few tens of MB.
// Here one launch does the whole step:
//   1. every CTA reads all heads' lengths and forms the exclusive prefix P of their used
//      rows (flat rows plus the appended one), in shared memory: the used rows of all heads
//      are one range [0, T);
//   2. CTA c (one per SM) takes rows [T c / N, T (c + 1) / N) of that range, and its 8 warps
//      an eighth each.  A warp streams the flat rows of each head piece in its eighth
//      through its own ring of bulk copies, in tiles of 2U rows, and reads the new row from
//      k_new / v_new (appending it to the flat buffer);
//   (a call with few rows uses only as many CTAs as give each kSplitMinRows rows);
//   the q rows and the new row of a warp's heads are loaded one head ahead, so neither is a
//   dependent load behind a head's stream;
//   3. a head held by one warp is written out by it; the pieces of a head split between
//      warps are merged in shared memory; a head that crosses CTA boundaries leaves one
//      partial per CTA in global memory, and the last CTA to finish it (a per-head ticket)
//      merges them.
// CTA boundaries inside short heads move to the nearer head end, so only heads longer than
// kSplitSnapRows ever cross CTAs.  The lengths are bumped by the last CTA to count itself
// past step 1 (every CTA has read them by then), as it leaves.  The counters and tickets
// return to zero at the end of every launch, so the workspace only has to start zeroed.
// No CTA waits for another: the grid needs no co-residency.  The launch is a programmatic
// dependent of the call before it on the stream (nothing is touched before that one ends).
#include "decode_rows16.cuh"

namespace kv {

namespace {
using namespace r16;
constexpr int kSWarps = 8;
constexpr int kSThreads = kSWarps * 32;
constexpr int kSPer = (int)(kDecodeSplitHeadsMax / kSThreads);   // heads per thread, step 1
static_assert(kSPer * kSThreads == kDecodeSplitHeadsMax, "scan covers every head");
constexpr int kSCand = kSWarps + 1;   // heads a CTA may have to merge
// Used rows per CTA at least: a small call, such as one layer's heads, runs on as few CTAs
// as that allows.  Measured on GB300 (L2 flushed): 64 rather than 384 spreads a 128K
// context's 34K used rows over every SM (27 vs 32 us) and one layer's 1K rows over 17 CTAs
// instead of 3 (15 vs 20 us), and changes nothing on caches of 1M rows.
constexpr int64_t kSplitMinRows = 64;
// A CTA boundary that falls inside a head of at most this many used rows moves to the
// nearer end of that head: short heads are never split between CTAs (no partials in global
// memory, no ticket), and a CTA's range grows or shrinks by at most half such a head.
// (256 measured slightly ahead of 512 on the 128K cache, equal elsewhere.)
constexpr int64_t kSplitSnapRows = 256;

struct SplitSmem {
  WarpRing ring[kSWarps];   // after the stream: the warps' partials, slots 2k and 2k + 1
  int64_t P[kDecodeSplitHeadsMax + 1];   // used rows of the heads before h
  int32_t base[kDecodeSplitHeadsMax];    // flat row of the head's first row
  uint8_t app[kDecodeSplitHeadsMax];     // the new row is appended to the head
  int64_t wsum[kSWarps];
  int32_t wfirst[kSWarps], wlast[kSWarps];   // heads of each warp's first and last rows
  int32_t cand[kSCand];                      // heads to merge, their warp slots (4 bits
  uint32_t cslots[kSCand];                   // each) and counts, and whether they cross
  int32_t cn[kSCand], ccross[kSCand];        // the CTA's ends
  int32_t ncand, win[2];
  int64_t bnd[2];                            // the CTA's first and end used rows
};
static_assert(sizeof(SplitSmem) <= 227 * 1024, "one CTA per SM");

// Largest h in [0, n) with P[h] <= x, for 0 <= x < P[n]: the head that holds used row x.
__device__ __forceinline__ int head_of(const int64_t* P, int n, int64_t x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (P[mid] <= x) lo = mid;
    else hi = mid;
  }
  return lo;
}
// First used row of CTA c, and the CTA that holds row x (0 <= x < T).
__device__ __forceinline__ int64_t cta_first(int64_t c, int64_t T, int N) { return T * c / N; }
__device__ __forceinline__ int64_t cta_of(int64_t x, int64_t T, int N) {
  return ((x + 1) * N + T - 1) / T - 1;
}

template <bool GL>
__device__ __forceinline__ float ldp(const float* p) {
  if constexpr (GL) return __ldcg(p);
  else return *p;
}
template <bool GL>
__device__ __forceinline__ float4 ldp4(const float* p) {
  if constexpr (GL) return __ldcg(reinterpret_cast<const float4*>(p));
  else return *reinterpret_cast<const float4*>(p);
}

// Merge of n partials (max[8], sum[8], o[G][d]) for the VE floats of o at `off` of query
// row g: slot(i) is the i-th partial, or nullptr for none.  GL: the partials are in global
// memory, written by other CTAs of this launch (read through L2).  kB partials per round of
// loads, folded into a running (M, L, acc).
template <bool GL, int kB, int VE, typename Slot>
__device__ __forceinline__ void merge_slice(int n, Slot slot, int g, int off, float& M,
                                            float& L, float (&acc)[VE]) {
  M = -INFINITY;
  L = 0.f;
#pragma unroll
  for (int x = 0; x < VE; ++x) acc[x] = 0.f;
  for (int i0 = 0; i0 < n; i0 += kB) {
    float m[kB], l[kB];
    float4 o[kB][VE / 4];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      m[u] = -INFINITY;
      l[u] = 0.f;
#pragma unroll
      for (int j = 0; j < VE / 4; ++j) o[u][j] = make_float4(0.f, 0.f, 0.f, 0.f);
      const float* Pp = i0 + u < n ? slot(i0 + u) : nullptr;
      if (Pp != nullptr) {
        m[u] = ldp<GL>(Pp + g);
        l[u] = ldp<GL>(Pp + 8 + g);
#pragma unroll
        for (int j = 0; j < VE / 4; ++j) o[u][j] = ldp4<GL>(Pp + off + 4 * j);
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < kB; ++u) Mn = fmaxf(Mn, m[u]);
    if (Mn == -INFINITY) continue;
    const float a = ptx::ex2(M - Mn);   // 0 while M is still -inf
    L *= a;
#pragma unroll
    for (int x = 0; x < VE; ++x) acc[x] *= a;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      if (m[u] > -INFINITY) {
        const float w = ptx::ex2(m[u] - Mn);
        L = fmaf(l[u], w, L);
#pragma unroll
        for (int j = 0; j < VE / 4; ++j) {
          acc[4 * j] = fmaf(o[u][j].x, w, acc[4 * j]);
          acc[4 * j + 1] = fmaf(o[u][j].y, w, acc[4 * j + 1]);
          acc[4 * j + 2] = fmaf(o[u][j].z, w, acc[4 * j + 2]);
          acc[4 * j + 3] = fmaf(o[u][j].w, w, acc[4 * j + 3]);
        }
      }
    }
    M = Mn;
  }
}

template <typename T, int VE>
__device__ __forceinline__ void store_out(T* dst, float (&acc)[VE], float L) {
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int x = 0; x < VE; ++x) acc[x] *= inv;
  *reinterpret_cast<uint4*>(dst) = pack_row16(acc, T());
}
template <int VE>
__device__ __forceinline__ void store_part(float* P, int g, int off, bool head, float M, float L,
                                           const float (&acc)[VE]) {
  if (head) {
    P[g] = M;
    P[8 + g] = L;
  }
#pragma unroll
  for (int j = 0; j < VE / 4; ++j)
    *reinterpret_cast<float4*>(P + off + 4 * j) =
        make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
}
}  // namespace

// GM: the group size rounded up to 2 or 4 (register arrays); G <= GM is the real one.
template <typename T, int GM>
__global__ void __launch_bounds__(kSThreads, 1)
decode_split(const T* __restrict__ q, const T* __restrict__ kn, const T* __restrict__ vn,
             T* __restrict__ kf, T* __restrict__ vf, const int64_t* __restrict__ cu,
             int32_t* __restrict__ lens, int64_t cap, T* __restrict__ out, int H, int Hkv,
             int G, float c2, float* __restrict__ part, uint32_t* __restrict__ tick,
             int64_t min_rows, int64_t snap_rows, WsHeader* hdr) {
  using Att = RowTileAttn<T, GM>;
  constexpr int VE = Att::VE, V2 = Att::V2, D = Att::D, U = Att::U;
  constexpr int NSL = D / VE;   // 16-byte slices per row
  extern __shared__ __align__(128) unsigned char dsm_raw[];
  SplitSmem& S = *reinterpret_cast<SplitSmem*>(dsm_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int half = lane >> 4, ci = lane & 15;
  const int N = (int)gridDim.x, c = (int)blockIdx.x;
  const int GD = G * D;
  const int pstride = kPartHead + GD;   // floats per partial
  const int nsl = G * NSL;              // output slices per head
  WarpRing& ws = S.ring[warp];

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&ws.full[s], 1);
    ptx::fence_mbar_init();
  }
  // a programmatic dependent launch: the next call on the stream may start launching, and
  // nothing of the previous one is read or written before it is done
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  // ---- 1. used rows of every head and their prefix (all loads first: nothing below may
  // be ordered before them)
  int64_t hb[kSPer], he[kSPer];
  int hl[kSPer];
#pragma unroll
  for (int i = 0; i < kSPer; ++i) {
    const int h = tid * kSPer + i;
    hb[i] = 0;
    he[i] = 0;
    hl[i] = 0;
    if (h < H) {
      const int seg = h / Hkv, g0 = h - seg * Hkv;
      const int64_t* cp = cu + (int64_t)seg * (Hkv + 1) + g0;
      hb[i] = cp[0];
      he[i] = cp[1];
      hl[i] = lens[h];
    }
  }
  int64_t rr[kSPer];
  int64_t rsum = 0;
#pragma unroll
  for (int i = 0; i < kSPer; ++i) {
    const int h = tid * kSPer + i;
    rr[i] = 0;
    if (h < H) {
      const int64_t base = hb[i], end = he[i];
      const int len = hl[i];
      const int64_t e = end < cap ? end : cap;
      int64_t nflat = 0;
      bool app = false;
      if (e > base && base >= 0) {
        nflat = len > 0 ? (int64_t)len : 0;
        if (nflat > e - base) nflat = e - base;
        app = kn != nullptr && len >= 0 && base + len < end && base + len < cap;
      }
      rr[i] = nflat + (app ? 1 : 0);
      // a head with used rows starts below cap, which the launch keeps within int32
      S.base[h] = rr[i] > 0 ? (int32_t)base : 0;
      S.app[h] = app ? 1 : 0;
      if (c == 0) {
        if (end > cap) raise_dev(hdr, DEV_FLAT_CAPACITY, (unsigned)h);
        if (kn != nullptr && !app) raise_dev(hdr, DEV_NO_RESERVE, (unsigned)h);
        if (rr[i] == 0)   // no row of this head can be read: its output is zero
          for (int x = 0; x < nsl; ++x)
            *reinterpret_cast<uint4*>(out + (int64_t)h * GD + x * VE) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    rsum += rr[i];
  }
  int64_t incl = rsum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t t = (int64_t)__shfl_up_sync(0xFFFFFFFFu, (long long)incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) S.wsum[warp] = incl;
  __syncthreads();
  int64_t run = incl - rsum;
  for (int w = 0; w < warp; ++w) run += S.wsum[w];
#pragma unroll
  for (int i = 0; i < kSPer; ++i) {
    const int h = tid * kSPer + i;
    if (h < H) S.P[h] = run;
    run += rr[i];
  }
  if (tid == kSThreads - 1) S.P[H] = run;
  __syncthreads();
  // the last CTA past this point writes the new lengths: every CTA has read lens by then
  // Every CTA has read lens once it is past this point; the last CTA to count itself here
  // writes the new lengths when it leaves (warp 0 waits for the count only then, so the
  // atomic's round trip overlaps the stream).
  uint32_t scanned = 0;
  if (tid == 0) scanned = atomicAdd(&tick[0], 1u);
  auto leave = [&]() {
    if (warp != 0) return;
    const uint32_t old = __shfl_sync(0xFFFFFFFFu, scanned, 0);
    if (old != (uint32_t)(N - 1)) return;
    for (int h = lane; h < H; h += 32)
      if (S.app[h]) lens[h] = (int32_t)(S.P[h + 1] - S.P[h]);
    if (lane == 0) atomicExch(&tick[0], 0u);
  };

  // ---- 2. this CTA's rows, an eighth per warp
  const int64_t Tu = S.P[H];   // used rows of all heads
  const int64_t ne = (Tu + min_rows - 1) / min_rows;
  const int Ne = (int)(ne < 1 ? 1 : ne > N ? N : ne);   // CTAs that take rows
  if (c >= Ne) {
    leave();
    return;
  }
  // CTA k's first row: T k / Ne, moved to the nearer end of a short head it falls in.  Rows
  // of a head longer than kSplitSnapRows are split at the unmoved boundaries, so cta_of and
  // cta_first locate the pieces of such a head exactly.
  auto bound = [&](int64_t k) -> int64_t {
    const int64_t x = cta_first(k, Tu, Ne);
    if (x <= 0 || x >= Tu) return x;
    const int h = head_of(S.P, H, x);
    const int64_t lo = S.P[h], hi = S.P[h + 1];
    if (hi - lo > snap_rows) return x;
    return x - lo <= hi - x ? lo : hi;
  };
  // the CTA's two ends, each found by one thread, shared through shared memory
  if (tid == 0) S.bnd[0] = bound(c);
  if (tid == 32) S.bnd[1] = bound(c + 1);
  __syncthreads();
  const int64_t b0 = S.bnd[0], b1 = S.bnd[1];
  const int64_t span = b1 - b0;
  const int64_t xs = b0 + span * warp / kSWarps, xe = b0 + span * (warp + 1) / kSWarps;

  Att att;
  float am[GM], al[GM];   // the warp's first piece, when its head began in an earlier warp
  float2 ao[GM][V2];
  bool hasA = false, hasB = false;
  int issued = 0, consumed = 0, abort_at = -1;
  if (xs < xe) {
    const int hf = head_of(S.P, H, xs);
    // producer: the flat rows of each piece in turn, kStageRows at a time (lane 0 issues,
    // every lane keeps the cursor)
    int ph = hf;
    int64_t px = xs;
    auto flat_end = [&](int hh) {   // end of head hh's flat rows within this warp's range
      const int64_t fe = S.P[hh + 1] - S.app[hh];
      return fe < xe ? fe : xe;
    };
    auto issue_next = [&]() {
      while (px < xe && px >= flat_end(ph)) {
        ++ph;
        if (S.P[ph] > px) px = S.P[ph];
      }
      if (px >= xe) return;
      const int64_t fe = flat_end(ph);
      const int nr = (int)(fe - px < kStageRows ? fe - px : kStageRows);
      if (abort_at < 0) {
        if (lane == 0) {
          const int s = issued % kStages;
          const int64_t row = (int64_t)S.base[ph] + (px - S.P[ph]);
          const uint32_t bytes = (uint32_t)nr * kRowBytes;
          ptx::mbar_arrive_expect_tx(&ws.full[s], 2u * bytes);
          ptx::bulk_load(ws.st[s][0], reinterpret_cast<const char*>(kf) + row * kRowBytes, bytes,
                         &ws.full[s]);
          ptx::bulk_load(ws.st[s][1], reinterpret_cast<const char*>(vf) + row * kRowBytes, bytes,
                         &ws.full[s]);
        }
        ++issued;
      }
      px += nr;
    };
    __syncwarp();   // the barriers are initialised
    for (int i = 0; i < kStages; ++i) issue_next();

    // q and the new row (k_new / v_new, half 0 of the warp) of a head are loaded when its
    // turn is one head away, so neither is a dependent load behind the head's stream
    uint4 qr[GM];
    uint4 nkr = make_uint4(0u, 0u, 0u, 0u), nvr = nkr;
    auto load_new = [&](int hh) {
      if (half == 0 && S.app[hh]) {
        nkr = *reinterpret_cast<const uint4*>(kn + (int64_t)hh * D + ci * VE);
        nvr = *reinterpret_cast<const uint4*>(vn + (int64_t)hh * D + ci * VE);
      }
    };
    load_q<T, GM>(q, hf, G, ci, qr);
    load_new(hf);
    int qh = hf, hlast = hf;
    for (int h = hf; h < H; ++h) {
      const int64_t Ph = S.P[h], Ph1 = S.P[h + 1];
      const int64_t lo = Ph > xs ? Ph : xs, hi = Ph1 < xe ? Ph1 : xe;
      if (lo >= xe) break;
      if (hi <= lo) continue;   // a head with no used rows
      hlast = h;
      const bool app = S.app[h] != 0;
      const int64_t fend = Ph1 - (app ? 1 : 0);
      const int64_t fe = fend < hi ? fend : hi;
      if (qh != h) {
        load_q<T, GM>(q, h, G, ci, qr);
        load_new(h);
      }
      att.begin(qr, c2);
      const uint4 ckr = nkr, cvr = nvr;   // this head's new row
      // the next head's q and new row, while this one streams
      if (h + 1 < H && Ph1 < xe) {
        load_q<T, GM>(q, h + 1, G, ci, qr);
        load_new(h + 1);
        qh = h + 1;
      }
      for (int64_t x = lo; x < fe;) {
        const int nr = (int)(fe - x < kStageRows ? fe - x : kStageRows);
        const int s = consumed % kStages;
        if (abort_at < 0) {
          const bool landed = ptx::mbar_wait(&ws.full[s], (uint32_t)((consumed / kStages) & 1));
          if (__any_sync(0xFFFFFFFFu, !landed)) {
            abort_at = consumed;
            if (lane == 0) raise_dev(hdr, DEV_WAIT_TIMEOUT, 0x700u + (unsigned)s);
          }
        }
        for (int b = 0; b < nr; b += Att::kRows) {
          uint4 kr[U], vr[U];
          load_tile<Att>(ws.st[s][0], ws.st[s][1], b, nr, kr, vr);
          att.tile(kr, vr, nr - b, ws.red, ws.pbuf);
        }
        __syncwarp();   // every lane is done with stage s
        if (abort_at < 0) ++consumed;
        issue_next();
        x += nr;
      }
      if (app && hi == Ph1) {
        // the new row: attended to from k_new / v_new, and appended at base + len
        uint4 kr[U], vr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          kr[u] = make_uint4(0u, 0u, 0u, 0u);
          vr[u] = kr[u];
        }
        if (half == 0) {
          kr[0] = ckr;
          vr[0] = cvr;
          const int64_t row = (int64_t)S.base[h] + (fend - Ph);
          reinterpret_cast<uint4*>(kf + row * D)[ci] = kr[0];
          reinterpret_cast<uint4*>(vf + row * D)[ci] = vr[0];
        }
        att.tile(kr, vr, 1, ws.red, ws.pbuf);
      }
      att.finish();
      if (lo == Ph && hi == Ph1) {
        // the whole head is in this warp: its output
        if (half == 0) {
#pragma unroll
          for (int g = 0; g < GM; ++g) {
            if (g < G) {
              float acc[VE];
#pragma unroll
              for (int e2 = 0; e2 < V2; ++e2) {
                acc[2 * e2] = att.o[g][e2].x;
                acc[2 * e2 + 1] = att.o[g][e2].y;
              }
              store_out<T, VE>(out + ((int64_t)h * G + g) * D + ci * VE, acc, att.l[g]);
            }
          }
        }
      } else if (Ph < xs) {
        // began in an earlier warp: the warp's first piece, kept until the stream is done
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          am[g] = att.m[g];
          al[g] = att.l[g];
#pragma unroll
          for (int e2 = 0; e2 < V2; ++e2) ao[g][e2] = att.o[g][e2];
        }
        hasA = true;
      } else {
        hasB = true;   // goes on past this warp: the warp's last piece, still in att
      }
    }
    if (lane == 0) {
      S.wfirst[warp] = hf;
      S.wlast[warp] = hlast;
    }
  }
  if (abort_at >= 0 && lane == 0) {
    // a wait gave up: let the copies issued and not yet read land before the memory is reused
    for (int it = abort_at; it < issued; ++it)
      (void)ptx::mbar_wait(&ws.full[it % kStages], (uint32_t)((it / kStages) & 1), 20000000ull);
  }
  __syncthreads();   // every ring is idle: its memory holds the warps' partials now

  // ---- 3. merges
  float* wp = reinterpret_cast<float*>(dsm_raw);   // slot 2k: warp k's first piece, 2k + 1: last
  auto put = [&](float* Pp, const float (&m)[GM], const float (&l)[GM],
                 const float2 (&o)[GM][V2]) {
    if (half != 0) return;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        if (ci == 0) {
          Pp[g] = m[g];
          Pp[8 + g] = l[g];
        }
#pragma unroll
        for (int e2 = 0; e2 < V2; e2 += 2)
          *reinterpret_cast<float4*>(Pp + kPartHead + g * D + ci * VE + 2 * e2) =
              make_float4(o[g][e2].x, o[g][e2].y, o[g][e2 + 1].x, o[g][e2 + 1].y);
      }
    }
  };
  if (hasA) put(wp + (2 * warp) * pstride, am, al, ao);
  if (hasB) put(wp + (2 * warp + 1) * pstride, att.m, att.l, att.o);
  if (span <= 0) {   // no rows here (uniform in the CTA)
    leave();
    return;
  }
  auto warp_first = [&](int k) { return b0 + span * k / kSWarps; };
  if (tid == 0) {
    // heads split between warps, or crossing the CTA's ends: each holds the first row of a
    // non-empty warp or the CTA's last row
    auto warp_of = [&](int64_t x) {
      int k = kSWarps - 1;
      while (k > 0 && warp_first(k) > x) --k;
      return k;
    };
    int nc = 0, prev = -1, klast = 0;
    for (int k = 0; k <= kSWarps; ++k) {
      int h;
      if (k < kSWarps) {
        if (warp_first(k) >= warp_first(k + 1)) continue;   // an empty eighth
        h = S.wfirst[k];
        klast = k;
      } else {
        h = S.wlast[klast];
      }
      if (h == prev) continue;
      prev = h;
      const int64_t Ph = S.P[h], Ph1 = S.P[h + 1];
      const bool cross = Ph < b0 || Ph1 > b1;
      const int ka = warp_of(Ph > b0 ? Ph : b0), kb = warp_of((Ph1 < b1 ? Ph1 : b1) - 1);
      if (!cross && ka == kb) continue;   // written by its warp
      uint32_t slots = 0;
      int n = 0;
      for (int kk = ka; kk <= kb; ++kk)
        if (warp_first(kk) < warp_first(kk + 1)) {
          slots |= (uint32_t)(Ph < warp_first(kk) ? 2 * kk : 2 * kk + 1) << (4 * n);
          ++n;
        }
      S.cand[nc] = h;
      S.cslots[nc] = slots;
      S.cn[nc] = n;
      S.ccross[nc] = cross ? 1 : 0;
      ++nc;
    }
    S.ncand = nc;
  }
  __syncthreads();   // partials and candidates in place
  const int ncand = S.ncand;
  for (int idx = tid; idx < ncand * nsl; idx += kSThreads) {
    const int ic = idx / nsl, sl0 = idx - ic * nsl;
    const int g = sl0 / NSL, sl = sl0 - g * NSL;
    const int off = kPartHead + g * D + sl * VE;
    const int h = S.cand[ic];
    const uint32_t slots = S.cslots[ic];
    float M, L, acc[VE];
    merge_slice<false, 4, VE>(
        S.cn[ic], [&](int i) -> const float* { return wp + ((slots >> (4 * i)) & 15u) * pstride; },
        g, off, M, L, acc);
    if (!S.ccross[ic]) {
      store_out<T, VE>(out + ((int64_t)h * G + g) * D + sl * VE, acc, L);
    } else {
      float* Pg = part + (int64_t)(S.P[h] < b0 ? 2 * c : 2 * c + 1) * pstride;
      store_part<VE>(Pg, g, off, sl == 0, M, L, acc);
    }
  }
  // heads crossing the CTA's ends (its first and last candidates): this CTA's partials are
  // out, and the last of each head's CTAs merges them
  const int nx = ncand == 0 ? 0 : (S.ccross[0] + (ncand > 1 ? S.ccross[ncand - 1] : 0));
  if (nx == 0) {   // uniform in the CTA
    leave();
    return;
  }
  __threadfence();
  __syncthreads();
  if (tid < 2) {
    int ic = -1;
    if (tid == 0 && S.ccross[0]) ic = 0;
    if (tid == 1 && ncand > 1 && S.ccross[ncand - 1]) ic = ncand - 1;
    int won = 0;
    if (ic >= 0) {
      const int h = S.cand[ic];
      const int64_t ca = cta_of(S.P[h], Tu, Ne), cb = cta_of(S.P[h + 1] - 1, Tu, Ne);
      uint32_t npc = (uint32_t)(cb - ca + 1);   // the head's CTAs with rows
      if (Tu < Ne) {
        npc = 0;
        for (int64_t cc = ca; cc <= cb; ++cc)
          npc += cta_first(cc, Tu, Ne) < cta_first(cc + 1, Tu, Ne);
      }
      const uint32_t old = atomicAdd(&tick[1 + h], 1u);
      if (old + 1u == npc) {
        atomicExch(&tick[1 + h], 0u);
        won = 1;
      }
    }
    S.win[tid] = won ? ic : -1;
  }
  __syncthreads();
  if (S.win[0] < 0 && S.win[1] < 0) {
    leave();
    return;
  }
  __threadfence();
  for (int idx = tid; idx < 2 * nsl; idx += kSThreads) {
    const int wi = idx / nsl, sl0 = idx - wi * nsl;
    const int ic = S.win[wi];
    if (ic < 0) continue;
    const int g = sl0 / NSL, sl = sl0 - g * NSL;
    const int off = kPartHead + g * D + sl * VE;
    const int h = S.cand[ic];
    const int64_t ca = cta_of(S.P[h], Tu, Ne), cb = cta_of(S.P[h + 1] - 1, Tu, Ne);
    float M, L, acc[VE];
    merge_slice<true, 8, VE>(
        (int)(cb - ca + 1),
        [&](int i) -> const float* {
          const int64_t cc = ca + i;
          if (!(cta_first(cc, Tu, Ne) < cta_first(cc + 1, Tu, Ne))) return nullptr;
          return part + (cc == ca ? 2 * cc + 1 : 2 * cc) * pstride;
        },
        g, off, M, L, acc);
    store_out<T, VE>(out + ((int64_t)h * G + g) * D + sl * VE, acc, L);
  }
  leave();
}

bool decode_split_supported(const Shape& s, int64_t cap) {
  const int64_t H = s.units();
  return s.d * s.esize() == kRowBytes && s.G() <= 4 && H > 0 && H <= kDecodeSplitHeadsMax &&
         cap <= (int64_t)INT32_MAX;
}

// One instantiation: its shared-memory opt-in and resident CTAs per SM once per device
// (each kernel needs its own), then the launch of one wave.
template <typename T, int GM>
static cudaError_t launch_split_t(const Shape& s, const void* q, const void* kn, const void* vn,
                                  void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                  int64_t cap, float c2, void* out, float* part,
                                  int64_t part_slots, uint32_t* tick, WsHeader* hdr,
                                  cudaStream_t st) {
  const size_t smem = sizeof(SplitSmem);
  static std::atomic<int> slot[kMaxDevices];
  const int per_sm = per_device(slot, [&]() {
    int n = 0;
    if (cudaFuncSetAttribute(decode_split<T, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split<T, GM>, kSThreads,
                                                      smem) != cudaSuccess)
      return 0;
    return n;
  });
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
  int64_t grid = (int64_t)per_sm * num_sms();
  if (2 * grid > part_slots) grid = part_slots / 2;   // two partial slots per CTA
  if (grid < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_split<T, GM>, (const T*)q, (const T*)kn,
                                           (const T*)vn, (T*)kf, (T*)vf, cu, lens, cap, (T*)out,
                                           (int)s.units(), s.Hkv, s.G(), c2, part, tick,
                                           kSplitMinRows, kSplitSnapRows, hdr);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

cudaError_t launch_decode_split(const Shape& s, const void* q, const void* kn, const void* vn,
                                void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                int64_t cap, float scale, void* out, float* part,
                                int64_t part_slots, uint32_t* tick, WsHeader* hdr,
                                cudaStream_t st) {
  const float c2 = scale * 1.4426950408889634f;
  const int G = s.G();
  const int GM = G <= 2 ? 2 : 4;   // tiles of 32 scores: GM >= 2
#define KV_SPLIT_CASE(T, M)                                                                  \
  return launch_split_t<T, M>(s, q, kn, vn, kf, vf, cu, lens, cap, c2, out, part, part_slots, \
                              tick, hdr, st)
  if (s.dtype == KV_BF16) {
    switch (GM) {
      case 2: KV_SPLIT_CASE(__nv_bfloat16, 2);
      default: KV_SPLIT_CASE(__nv_bfloat16, 4);
    }
  }
  switch (GM) {
    case 2: KV_SPLIT_CASE(float, 2);
    default: KV_SPLIT_CASE(float, 4);
  }
#undef KV_SPLIT_CASE
}

}  // namespace kv
