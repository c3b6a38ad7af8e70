// One decode step of attention over the flat cache of a few hundred short heads, with the
// rows of the long heads dealt out to more CTAs.
//
// Ada-KV formal model: the new token's k, v are appended to its head's cache, then
// A = softmax(q K^T / sqrt(d)) and o = A V per query head, over the uneven per-head lengths
// of the flat layout.
//
// With one CTA per head (decode_head.cu) a step waits on its longest head.  Here a head's
// flat rows are cut into part 0 (its first P0 - 128 to P0 + 63 rows, and at least one fill)
// and extra parts of kQPart = 192 rows (4 warps x 3 ring stages of 16 rows: one fill of every
// warp's ring) from its end, the one next to part 0 shorter where part 0 keeps a whole first
// fill.  The head's own CTA takes part 0 and the new row; the extra parts go
// round-robin to the CTAs past the heads' own (a launch of two CTAs per SM has more CTAs than
// heads), then to the heads' CTAs.  P0 is a multiple of kQPart chosen by every CTA from the
// head lengths: the smallest candidate whose extra parts all find an idle CTA (else the
// largest), so a cache of even heads runs one CTA per head and a skewed one spreads its long
// heads.  A head of one part is written out by its CTA; the parts of a longer head leave
// partials in global memory and the last of them to finish (a per-head ticket) merges them.
//
//   1. the head's own CTA loads its q, new row, offsets and length and requests the first
//      fill of part 0; every CTA then reads all heads' lengths, picks P0 and forms, in
//      shared memory, the prefix of the heads' extra parts;
//   2. it takes its parts one at a time.  Stage s (16 rows) of a part belongs to warp s % 4,
//      which streams its stages through its ring of bulk copies (a stage is refilled as soon
//      as it is read) and the tile loop of decode_rows16.cuh.  The warps' partials are merged
//      in shared memory (each warp's transpose buffer);
//   3. the lengths of the heads that took the new row are bumped once no CTA reads them any
//      more: by the last CTA to have read every length it needs (right after its scan, when
//      no CTA has more than kQXMax extra parts), else by the last CTA to finish; that CTA
//      returns the counter to zero.
// Rows of 256 bytes (bf16 d = 128, fp32 d = 64), G <= 4.  Tickets and the counter are zero
// between launches; the launch is a programmatic dependent of the call before it.
#include "decode_heads.cuh"
#include "decode_rows16.cuh"

namespace kv {

namespace {
using namespace r16;
constexpr int kQWarps = 4;
constexpr int kQThreads = kQWarps * 32;
constexpr int kQSlice = kStages * kStageRows;     // rows of one warp's ring fill
constexpr int kQPart = kQWarps * kQSlice;         // rows of one part
constexpr int kQPer = (int)((kDecodePartsHeadsMax + kQThreads - 1) / kQThreads);
static_assert(kQPer * kQThreads >= kDecodePartsHeadsMax, "scan covers every head");
// candidate sizes of part 0, in parts of kQPart: 1, 2, 3, 4, 6, 8, 12, 16 (arithmetic, not a
// table: a constant-bank miss would wait behind the step's bulk copies in DRAM)
constexpr int kNP0 = 8;
// extra parts per CTA up to which every CTA reads its extra parts' lengths right after the
// scan, so the lengths can be bumped early (step 3)
constexpr int kQXMax = 8;
__host__ __device__ constexpr int p0_mult(int k) {
  return k < 4 ? k + 1 : (k & 1 ? 8 : 6) << ((k - 4) >> 1);
}
static_assert(p0_mult(0) == 1 && p0_mult(1) == 2 && p0_mult(3) == 4 && p0_mult(4) == 6 &&
                  p0_mult(5) == 8 && p0_mult(6) == 12 && p0_mult(7) == 16, "candidate sizes");

struct PartsSmem {
  WarpRing ring[kQWarps];   // a warp's partial goes to its transpose buffer (red)
  int32_t xpre[kDecodePartsHeadsMax + 1];   // extra parts of the heads before h
  int32_t wsum[kQWarps];
  int32_t ksum[kQWarps][kNP0];   // per warp: extra parts for each candidate P0
  int32_t xlen[kQXMax];          // lengths of the heads of this CTA's extra parts
  int32_t win;
};
static_assert(kPartHead + 4 * 128 <= kRedFloats, "a warp's partial fits its buffer (G <= 4)");

// Extra parts of a head of `flat` rows past part 0's p0: whole parts of kQPart rows taken
// from the head's end, part 0 keeping the rest (p0 - 128 to p0 + 63 rows, and never less
// than the first fill: with p0 = one fill, the extra part next to part 0 leaves it the rows
// that fill already holds).  A remainder of fewer than kQSliver rows stays in part 0 (merging
// its partial would cost more than reading it there), a longer one becomes an extra part (a
// further ring fill of the own CTA would cost more than the merge).
constexpr int kQSliver = 64;
__device__ __forceinline__ int extra_parts(int flat, int p0) {
  return flat > p0 ? (flat - p0 + kQPart - kQSliver) / kQPart : 0;
}
}  // namespace

// GM: the group size rounded up to 2 or 4 (register arrays); G <= GM is the real one.
template <typename T, int GM>
__global__ void __launch_bounds__(kQThreads, 2)
decode_parts(const T* __restrict__ q, const T* __restrict__ kn, const T* __restrict__ vn,
             T* __restrict__ kf, T* __restrict__ vf, const int64_t* __restrict__ cu,
             int32_t* __restrict__ lens, int64_t cap, T* __restrict__ out, int H, int Hkv,
             int G, float c2, float* __restrict__ part, int64_t part_slots,
             uint32_t* __restrict__ tick, WsHeader* hdr) {
  using Att = RowTileAttn<T, GM>;
  constexpr int VE = Att::VE, V2 = Att::V2, D = Att::D, U = Att::U;
  constexpr int NSL = D / VE;   // 16-byte slices per row
  extern __shared__ __align__(128) unsigned char dsm_raw[];
  PartsSmem& S = *reinterpret_cast<PartsSmem*>(dsm_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int half = lane >> 4, ci = lane & 15;
  const int Nc = (int)gridDim.x, c = (int)blockIdx.x;
  const int GD = G * D;
  const int pstride = kPartHead + GD;   // floats per partial
  const int nsl = G * NSL;              // output slices per head
  WarpRing& ws = S.ring[warp];
  const bool has_new = kn != nullptr;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&ws.full[s], 1);
    ptx::fence_mbar_init();
  }
  // a programmatic dependent launch: the next call on the stream may start launching, and
  // nothing of the previous one is read or written before it is done
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();

  // Stage s (rows [16 s, 16 s + 16) of a part) belongs to warp s % 4; `seq` counts this
  // warp's ring uses so far (slot seq % 3, parity (seq / 3) & 1).
  uint32_t seq = 0;
  auto nstages = [](int R) { return (R + kStageRows - 1) / kStageRows; };
  auto my_stages = [&](int R) {
    const int n = nstages(R);
    return n > warp ? (n - warp + kQWarps - 1) / kQWarps : 0;
  };
  // lane 0: this warp's stage ls of a part of R rows starting at flat row row0, into ring
  // use seq + ls
  auto issue = [&](int64_t row0, int R, int ls) {
    const int srow = (warp + kQWarps * ls) * kStageRows;
    const int st = (int)((seq + ls) % kStages);
    const uint32_t bytes = (uint32_t)min(kStageRows, R - srow) * kRowBytes;
    ptx::mbar_arrive_expect_tx(&ws.full[st], 2u * bytes);
    ptx::bulk_load(ws.st[st][0], reinterpret_cast<const char*>(kf) + (row0 + srow) * kRowBytes,
                   bytes, &ws.full[st]);
    ptx::bulk_load(ws.st[st][1], reinterpret_cast<const char*>(vf) + (row0 + srow) * kRowBytes,
                   bytes, &ws.full[st]);
  };
  // lane 0 waits for stage ls of the part, the warp runs its tiles, lane 0 refills the stage
  // with stage ls + 3 when that is below `cnt`.  Every stage read so far was refilled, so at
  // stage ls the copies in flight are stages [ls, min(cnt, ls + 3)); on a wait that gives up
  // those are waited for (bounded) and `ok` turns false.
  Att att;
  bool ok = true;
  auto consume = [&](int64_t row0, int R, int cnt) {
    for (int ls = 0; ls < cnt && ok; ++ls) {
      const uint32_t k = seq + ls;
      const int st = (int)(k % kStages);
      const bool landed = ptx::mbar_wait(&ws.full[st], (k / kStages) & 1u);
      if (__any_sync(0xFFFFFFFFu, !landed)) {
        ok = false;
        if (lane == 0) {
          raise_dev(hdr, DEV_WAIT_TIMEOUT, 0x900u + (unsigned)st);
          for (int l2 = ls; l2 < min(cnt, ls + kStages); ++l2)
            (void)ptx::mbar_wait(&ws.full[(seq + l2) % kStages], ((seq + l2) / kStages) & 1u,
                                 20000000ull);
        }
        break;
      }
      const int rows = min(kStageRows, R - (warp + kQWarps * ls) * kStageRows);
      for (int b = 0; b < rows; b += Att::kRows) {
        uint4 kr[U], vr[U];
        load_tile<Att>(ws.st[st][0], ws.st[st][1], b, rows, kr, vr);
        att.tile(kr, vr, rows - b, ws.red, ws.pbuf);
      }
      __syncwarp();   // every lane is done with stage st: refill it
      if (lane == 0 && ls + kStages < cnt) issue(row0, R, ls + kStages);
    }
  };

  // The end of a part: the new row (in its warp), each warp's (max, sum, o) merged in shared
  // memory, then the output of a one-part head, or the part's partial and its ticket (the
  // last part of the head to finish merges them).  Every thread of the CTA takes part.
  auto finish_part = [&](int h, int pi, int nparts, const HeadRows& hr, bool newrow, uint4 nkr,
                         uint4 nvr) {
    if (newrow) {
      // the new row, attended to from k_new / v_new and appended at base + len
      uint4 kr[U], vr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        kr[u] = make_uint4(0u, 0u, 0u, 0u);
        vr[u] = kr[u];
      }
      if (half == 0) {
        kr[0] = nkr;
        vr[0] = nvr;
        const int64_t row = hr.base + hr.len;
        reinterpret_cast<uint4*>(kf + row * D)[ci] = nkr;
        reinterpret_cast<uint4*>(vf + row * D)[ci] = nvr;
      }
      att.tile(kr, vr, 1, ws.red, ws.pbuf);
    }
    att.finish();
    // this warp's (max, sum, o) into its transpose buffer
    __syncwarp();
    float* wp = ws.red;
    if (half == 0) {
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g < G) {
          if (ci == 0) {
            wp[g] = att.m[g];
            wp[8 + g] = att.l[g];
          }
#pragma unroll
          for (int e2 = 0; e2 < V2; e2 += 2)
            *reinterpret_cast<float4*>(wp + kPartHead + g * D + ci * VE + 2 * e2) =
                make_float4(att.o[g][e2].x, att.o[g][e2].y, att.o[g][e2 + 1].x,
                            att.o[g][e2 + 1].y);
        }
      }
    }
    __syncthreads();   // the four warps' partials are in place
    // merge the warps: thread t takes 16 bytes of one query row
    const int slot = pi == 0 ? h : H + S.xpre[h] + pi - 1;
    for (int idx = tid; idx < nsl; idx += kQThreads) {
      const int g = idx / NSL, sl = idx - g * NSL;
      const int off = kPartHead + g * D + sl * VE;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kQWarps; ++w) M = fmaxf(M, S.ring[w].red[g]);
      float L = 0.f, acc[VE];
#pragma unroll
      for (int x = 0; x < VE; ++x) acc[x] = 0.f;
      if (M > -INFINITY) {
#pragma unroll
        for (int w = 0; w < kQWarps; ++w) {
          const float* P = S.ring[w].red;
          if (P[g] == -INFINITY) continue;
          const float sc = ptx::ex2(P[g] - M);
          L = fmaf(P[8 + g], sc, L);
#pragma unroll
          for (int x = 0; x < VE; ++x) acc[x] = fmaf(P[off + x], sc, acc[x]);
        }
      }
      if (nparts == 1) {
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int x = 0; x < VE; ++x) acc[x] *= inv;
        *reinterpret_cast<uint4*>(out + ((int64_t)h * G + g) * D + sl * VE) =
            pack_row16(acc, T());
      } else if (slot < part_slots) {
        float* Pg = part + (int64_t)slot * pstride;
        if (sl == 0) {
          Pg[g] = M;
          Pg[8 + g] = L;
        }
#pragma unroll
        for (int x = 0; x < VE; x += 4)
          *reinterpret_cast<float4*>(Pg + off + x) =
              make_float4(acc[x], acc[x + 1], acc[x + 2], acc[x + 3]);
      }
    }
    if (nparts > 1) {
      // the last of the head's parts to finish merges them (every slot: 8 per round).  The
      // CTA's partial is written before the barrier; the fence of the thread that takes the
      // ticket orders it (cumulatively) before the ticket, and the winner's fence orders the
      // other parts' partials before its CTA reads them.
      __syncthreads();
      if (tid == 0) {
        // every part takes its ticket (so the count returns to zero); a part without a slot
        // (the host's slot count rules it out) is left out of the merge
        if (slot >= part_slots) raise_dev(hdr, DEV_SELECT, 0x9000u + (unsigned)h);
        int win = 0;
        __threadfence();
        const uint32_t old = atomicAdd(&tick[1 + h], 1u);
        if (old + 1u == (uint32_t)nparts) {
          atomicExch(&tick[1 + h], 0u);
          __threadfence();
          win = 1;
        }
        S.win = win;
      }
      __syncthreads();
      if (S.win) {
        const int xbase = H + S.xpre[h];
        for (int idx = tid; idx < nsl; idx += kQThreads) {
          const int g = idx / NSL, sl = idx - g * NSL;
          const int off = kPartHead + g * D + sl * VE;
          float M = -INFINITY, L = 0.f, acc[VE];
#pragma unroll
          for (int x = 0; x < VE; ++x) acc[x] = 0.f;
          for (int i0 = 0; i0 < nparts; i0 += 8) {
            float m[8], l[8];
            float4 o[8][VE / 4];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              m[u] = -INFINITY;
              l[u] = 0.f;
#pragma unroll
              for (int j = 0; j < VE / 4; ++j) o[u][j] = make_float4(0.f, 0.f, 0.f, 0.f);
              const int i = i0 + u;
              const int64_t sl_i = i == 0 ? h : xbase + i - 1;
              if (i < nparts && sl_i < part_slots) {
                const float* Pp = part + sl_i * pstride;
                m[u] = __ldcg(Pp + g);
                l[u] = __ldcg(Pp + 8 + g);
#pragma unroll
                for (int j = 0; j < VE / 4; ++j)
                  o[u][j] = __ldcg(reinterpret_cast<const float4*>(Pp + off + 4 * j));
              }
            }
            float Mn = M;
#pragma unroll
            for (int u = 0; u < 8; ++u) Mn = fmaxf(Mn, m[u]);
            if (Mn == -INFINITY) continue;
            const float a = ptx::ex2(M - Mn);   // 0 while M is still -inf
            L *= a;
#pragma unroll
            for (int x = 0; x < VE; ++x) acc[x] *= a;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (m[u] > -INFINITY) {
                const float wgt = ptx::ex2(m[u] - Mn);
                L = fmaf(l[u], wgt, L);
#pragma unroll
                for (int j = 0; j < VE / 4; ++j) {
                  acc[4 * j] = fmaf(o[u][j].x, wgt, acc[4 * j]);
                  acc[4 * j + 1] = fmaf(o[u][j].y, wgt, acc[4 * j + 1]);
                  acc[4 * j + 2] = fmaf(o[u][j].z, wgt, acc[4 * j + 2]);
                  acc[4 * j + 3] = fmaf(o[u][j].w, wgt, acc[4 * j + 3]);
                }
              }
            }
            M = Mn;
          }
          const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
          for (int x = 0; x < VE; ++x) acc[x] *= inv;
          *reinterpret_cast<uint4*>(out + ((int64_t)h * G + g) * D + sl * VE) =
              pack_row16(acc, T());
        }
      }
    }
    __syncthreads();   // the transpose buffers and S.win are free for the next part
  };

  // ---- 1. every head's length, the size of part 0 and the prefix of the extra parts.  Every
  // CTA reads all heads' lengths, so the loads are coalesced (thread t takes heads t,
  // t + 128, ...) and issued before the bulk copies, and the offsets are not read here (a few
  // hundred CTAs re-reading the same lines hold up the L2 slices that the copies need too).
  // The parts are laid out on the lengths (clipped to the capacity); a head's own CTA clips
  // its rows to the head's extent when it reads them, and checks its head.  The lengths go to
  // shared memory (the prefix array, written only at the end of the scan), where each thread
  // then reads the kQPer consecutive heads it scans.
  int hl[kQPer];
#pragma unroll
  for (int i = 0; i < kQPer; ++i) {
    const int h = tid + kQThreads * i;
    hl[i] = h < H ? lens[h] : 0;
  }
  // The head's own CTA requests the first fill of part 0 before the scan, which runs while
  // the copies are in flight.  Part 0 holds at least the head's first min(flat, kQPart) rows,
  // so these are its first stages whatever P0 turns out to be.  (q and the new row are loaded first: behind the
  // copies they would wait for the step's traffic too.)
  HeadRows own{0, 0, 0, false};
  int pre = 0;   // stages of the own part 0 this warp has requested before the scan
  uint4 qr0[GM];
  uint4 nkr0 = make_uint4(0u, 0u, 0u, 0u), nvr0 = nkr0;
  if (c < H) {
    load_q<T, GM>(q, c, G, ci, qr0);
    if (has_new && half == 0) {
      nkr0 = *reinterpret_cast<const uint4*>(kn + (int64_t)c * D + ci * VE);
      nvr0 = *reinterpret_cast<const uint4*>(vn + (int64_t)c * D + ci * VE);
    }
    const int seg = c / Hkv, g = c - seg * Hkv;
    const int64_t end = cu[(int64_t)seg * (Hkv + 1) + g + 1];
    own = head_rows_of(cu[(int64_t)seg * (Hkv + 1) + g], end, lens[c], cap, has_new);
    if (tid == 0) {
      if (end > cap) raise_dev(hdr, DEV_FLAT_CAPACITY, (unsigned)c);
      if (has_new && !own.app) raise_dev(hdr, DEV_NO_RESERVE, (unsigned)c);
    }
    const int R1 = min(own.flat, kQPart);
    pre = min(kStages, my_stages(R1));
    if (lane == 0)
      for (int ls = 0; ls < pre; ++ls) issue(own.base, R1, ls);
  }
  int32_t* flat_s = S.xpre;
#pragma unroll
  for (int i = 0; i < kQPer; ++i) {
    const int h = tid + kQThreads * i;
    if (h < H) flat_s[h] = (int)min((int64_t)max(hl[i], 0), cap);
  }
  __syncthreads();
  int fl[kQPer];
#pragma unroll
  for (int i = 0; i < kQPer; ++i) {
    const int h = tid * kQPer + i;
    fl[i] = h < H ? flat_s[h] : 0;
  }
  // extra parts of every head for each candidate P0, summed over the CTA's threads
#pragma unroll
  for (int k = 0; k < kNP0; ++k) {
    int t = 0;
#pragma unroll
    for (int i = 0; i < kQPer; ++i) t += extra_parts(fl[i], p0_mult(k) * kQPart);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
    if (lane == 0) S.ksum[warp][k] = t;
  }
  __syncthreads();
  // the smallest P0 whose extra parts all find an idle CTA, else the largest
  const int idle = Nc > H ? Nc - H : 0;
  int P0 = p0_mult(kNP0 - 1) * kQPart;
  for (int k = 0; k < kNP0; ++k) {
    const int tot = S.ksum[0][k] + S.ksum[1][k] + S.ksum[2][k] + S.ksum[3][k];
    if (tot <= idle) {
      P0 = p0_mult(k) * kQPart;
      break;
    }
  }
  int nx[kQPer];
  int xs = 0;
#pragma unroll
  for (int i = 0; i < kQPer; ++i) {
    nx[i] = extra_parts(fl[i], P0);
    xs += nx[i];
  }
  int incl = xs;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) S.wsum[warp] = incl;
  __syncthreads();
  int run = incl - xs;
  for (int w = 0; w < warp; ++w) run += S.wsum[w];
#pragma unroll
  for (int i = 0; i < kQPer; ++i) {
    const int h = tid * kQPer + i;
    if (h < H) S.xpre[h] = run;
    run += nx[i];
  }
  if (tid == kQThreads - 1) S.xpre[H] = run;
  __syncthreads();
  const int NX = S.xpre[H];
  const int e0 = ((c - H) % Nc + Nc) % Nc;
  auto extra_head = [&](int e) {   // the head holding extra part e: largest h, xpre[h] <= e
    int lo = 0, hi = H;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (S.xpre[mid] <= e) lo = mid;
      else hi = mid;
    }
    return lo;
  };
  // The lengths are bumped (for the heads that take the new row) once no CTA reads them any
  // more.  When every CTA has at most kQXMax extra parts, each one reads its extra parts'
  // lengths now and counts itself done with the lengths; the CTA that counted last bumps
  // them.  Otherwise the last CTA to finish does it.  The early count is a relaxed atomic
  // whose result is looked at only once the CTA's parts are done: every length this CTA
  // read was consumed before the barrier ahead of it, so its reads are complete, and a
  // fence or release here would hold this thread until its own bulk copies in flight had
  // landed (measured: about 2 us on the first stage of every CTA).
  const bool early_bump = (NX + Nc - 1) / Nc <= kQXMax;
  uint32_t done_before = 0;   // tid 0: CTAs counted before this one
  if (early_bump) {
    const int nmine = NX > e0 ? (NX - e0 + Nc - 1) / Nc : 0;
    if (tid < nmine) S.xlen[tid] = lens[extra_head(e0 + tid * Nc)];
    __syncthreads();
    if (tid == 0) done_before = atomicAdd(&tick[0], 1u);
  }

  // ---- 2. this CTA's parts: the rest of part 0 of its own head, then every Nc-th extra part
  const int nown = c < H ? 1 : 0;
  for (int pidx = 0;; ++pidx) {
    int h, pi;
    if (pidx < nown) {
      h = c;
      pi = 0;
    } else {
      const int e = e0 + (pidx - nown) * Nc;
      if (e >= NX) break;
      h = extra_head(e);
      pi = 1 + e - S.xpre[h];
    }
    const int nparts = 1 + S.xpre[h + 1] - S.xpre[h];
    uint4 qr[GM];
    if (pi > 0) load_q<T, GM>(q, h, G, ci, qr);   // before the copies (see above)
    HeadRows hr = own;
    if (pi > 0) {
      const int seg = h / Hkv, g = h - seg * Hkv;
      hr = head_rows_of(cu[(int64_t)seg * (Hkv + 1) + g], cu[(int64_t)seg * (Hkv + 1) + g + 1],
                        early_bump ? S.xlen[pidx - nown] : lens[h], cap, has_new);
    }
    // the part's rows (none where the layout, on the lengths, ran past the head's extent)
    // (part 0 never holds fewer rows than the first fill requested before the scan, even
    // where lengths past a head's extent make the layout disagree with its rows: every stage
    // in flight is read before the CTA moves on)
    const int R0 = hr.flat - kQPart * (nparts - 1);     // rows left to part 0 by the layout
    const int P0e = max(R0, min(hr.flat, kQPart));       // part 0's rows
    const int r0 = pi == 0 ? 0 : max(R0 + (pi - 1) * kQPart, P0e);
    const int R = pi == 0 ? P0e : max(min(R0 + pi * kQPart, hr.flat) - r0, 0);
    const int64_t row0 = hr.base + r0;
    const int cnt = my_stages(R);
    const int fill = min(kStages, cnt);      // stages in flight before the first is read
    const int sent = pi == 0 ? pre : 0;      // of those, requested before the scan
    // the new row: in the warp that would take the stage after part 0's last
    const bool newrow = pi == 0 && hr.app && warp == nstages(R) % kQWarps;
    // the first fill (the own part's was requested before the scan)
    if (lane == 0 && ok)
      for (int ls = sent; ls < fill; ++ls) issue(row0, R, ls);
    att.begin(pi == 0 ? qr0 : qr, c2);
    consume(row0, R, cnt);
    seq += (uint32_t)cnt;
    finish_part(h, pi, nparts, hr, newrow, nkr0, nvr0);   // the new row is the own head's
  }

  // ---- 3. the lengths: bumped by the CTA that counted itself done with them last (early),
  // else by the last CTA to finish (every CTA has read them by then)
  if (tid == 0) {
    if (!early_bump) done_before = atom_add_release_u32(&tick[0], 1u);
    const int win = done_before == (uint32_t)(Nc - 1) ? 1 : 0;
    if (win) fence_acq_rel_gpu();
    S.win = win;
  }
  __syncthreads();
  if (S.win) {
    for (int h = tid; h < H; h += kQThreads) {
      const HeadRows hr = head_rows(cu, lens, h, Hkv, cap, has_new);
      if (hr.app) lens[h] = hr.len + 1;
    }
    if (tid == 0) atomicExch(&tick[0], 0u);
  }
}

bool decode_parts_supported(const Shape& s, int64_t cap, int64_t part_slots) {
  const int64_t H = s.units();
  return s.d * s.esize() == kRowBytes && s.G() <= 4 && H > 0 && H <= kDecodePartsHeadsMax &&
         cap <= (int64_t)INT32_MAX && H + cap / kQPart + 1 <= part_slots;
}

// One instantiation: its shared-memory opt-in once per device (each kernel needs its own),
// then the launch of two CTAs per SM (at least one per head).
template <typename T, int GM>
static cudaError_t launch_parts_t(const Shape& s, const void* q, const void* kn, const void* vn,
                                  void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                  int64_t cap, float c2, void* out, float* part,
                                  int64_t part_slots, uint32_t* tick, WsHeader* hdr,
                                  cudaStream_t st) {
  const size_t smem = sizeof(PartsSmem);
  static std::atomic<int> opted[kMaxDevices];
  if (!per_device(opted, [&]() {
        return cudaFuncSetAttribute(decode_parts<T, GM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem) == cudaSuccess ? 1 : 0;
      }))
    return cudaErrorInvalidConfiguration;
  int64_t grid = 2 * (int64_t)num_sms();
  if (grid < s.units()) grid = s.units();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_parts<T, GM>, (const T*)q, (const T*)kn,
                                           (const T*)vn, (T*)kf, (T*)vf, cu, lens, cap, (T*)out,
                                           (int)s.units(), s.Hkv, s.G(), c2, part, part_slots,
                                           tick, hdr);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

cudaError_t launch_decode_parts(const Shape& s, const void* q, const void* kn, const void* vn,
                                void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                int64_t cap, float scale, void* out, float* part,
                                int64_t part_slots, uint32_t* tick, WsHeader* hdr,
                                cudaStream_t st) {
  const float c2 = scale * 1.4426950408889634f;
  const int GM = s.G() <= 2 ? 2 : 4;   // tiles of 32 scores: GM >= 2
#define KV_PARTS_CASE(T, M)                                                                  \
  return launch_parts_t<T, M>(s, q, kn, vn, kf, vf, cu, lens, cap, c2, out, part, part_slots, \
                              tick, hdr, st)
  if (s.dtype == KV_BF16) {
    switch (GM) {
      case 2: KV_PARTS_CASE(__nv_bfloat16, 2);
      default: KV_PARTS_CASE(__nv_bfloat16, 4);
    }
  }
  switch (GM) {
    case 2: KV_PARTS_CASE(float, 2);
    default: KV_PARTS_CASE(float, 4);
  }
#undef KV_PARTS_CASE
}

}  // namespace kv
