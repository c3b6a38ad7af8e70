// Per-head selection and the flat cache gather.
//
// Ada-KV Algorithm 2: per-head Top-B_g eviction decision, selection of the kept
// K/V rows, concatenation of the observation window; the flat layout that puts
// every head of a layer into one tensor (cu_seqlens-style offsets), filled by a
// cache-update kernel.  CriticalKV: two-stage greedy selection, stage 1 by the
// attention score, stage 2 by (A + eps) * ||(V W^O)_j||_1.
//
// The selection is one CTA per head and two streaming passes over the head's keys, through
// a ring of bulk copies.  Pass A histograms the first digit (top 11 bits) of the largest key
// of every aligned group of 4 positions; the bin g holding the K-th largest group maximum has
// at least K groups at or above it, so at least K keys have a first digit >= g and tau, the
// K-th largest key, has one too.  Pass B, walking the head backwards (its first chunks are
// the ones pass A left in L2), collects every key with a first digit >= g (and every forced
// position) into shared memory in position order.  The exact radix select and the ordered
// emission then work on that short union alone.  A union that outgrows shared memory (large
// budgets) moves to the head's region of the workspace, which has room for every key.
#include <cstdlib>
#include <cstring>

#include "bulk_ring.cuh"
#include "kv_internal.cuh"
#include "radix_select.cuh"

namespace kv {

namespace {
constexpr int kScanThreads = 1024;
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelStages = 4;
constexpr int kSelStage = 16384;   // bytes per ring stage
constexpr int kUnion = 4096;       // candidate (position, key) pairs a CTA can hold
constexpr int kGatherThreads = 256;
constexpr uint32_t kNoBin = 0xFFFFFFFFu;
}

// Offsets of every head in the flat buffer and the initial lengths.
__global__ void __launch_bounds__(kScanThreads)
compact_offsets(const int32_t* __restrict__ head_budget, int64_t H, int Hkv, int w, int n,
                int reserve, int64_t cap, const int64_t* __restrict__ row_base,
                int64_t* __restrict__ cu, int32_t* __restrict__ lens, WsHeader* hdr) {
  __shared__ int64_t scratch[32];
  int64_t carry = row_base != nullptr ? *row_base : 0;   // the first row of the output
  for (int64_t t0 = 0; t0 < H; t0 += kScanThreads) {
    const int64_t h = t0 + threadIdx.x;
    int64_t val = 0;
    if (h < H) {
      int hb = head_budget[h];
      if (hb < w || hb > n) {
        raise_dev(hdr, DEV_HEAD_BUDGET, (unsigned)h);
        hb = hb < w ? w : n;
      }
      lens[h] = hb;
      val = (int64_t)hb + reserve;
    }
    int64_t tot;
    const int64_t incl = block_incl_scan64(val, scratch, &tot);
    if (h < H) {
      const int64_t seg = h / Hkv;
      const int g = (int)(h - seg * Hkv);
      cu[seg * (Hkv + 1) + g] = carry + incl - val;
      if (g == Hkv - 1) cu[seg * (Hkv + 1) + Hkv] = carry + incl;
    }
    carry += tot;
  }
  if (threadIdx.x == 0 && carry > cap) raise_dev(hdr, DEV_FLAT_CAPACITY, 0);
}


// Keys of a head in aligned groups of 4 flat positions: pos0 is the head position of the
// group's first value (negative or >= C outside the head; the caller masks those).
struct ScoreSrc {            // Ada-KV / LAVa scores; CriticalKV stage 1
  static constexpr bool kTwo = false;
  const float* S;            // the head's scores
  __device__ void keys(const float4& x, const float4&, int, uint32_t (&k)[4], bool (&f)[4]) const {
    k[0] = score_key(x.x); k[1] = score_key(x.y); k[2] = score_key(x.z); k[3] = score_key(x.w);
    f[0] = f[1] = f[2] = f[3] = false;
  }
  __device__ uint32_t key_at(int i) const { return score_key(S[i]); }
  __device__ bool forced_at(int) const { return false; }
  __device__ bool forced_key(uint32_t) const { return false; }
  // the largest key of a group whose four values all lie in the head (score_key is
  // monotonic, and fmaxf skips a NaN as score_key maps it to the smallest key)
  __device__ uint32_t full_max(const float4& x, const float4&, int) const {
    return score_key(fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
  }
  // the values of a group whose key has a first digit >= g (1 <= g < 1024): for x > 0 the
  // key is x's bit pattern, so the test is x >= the float whose bit pattern is g << 21
  __device__ uint32_t cand_mask(const float4& x, const float4&, int, uint32_t g) const {
    if (g == 0u) return 0xFu;
    if (g >= 1024u) return 0u;
    const float t = __uint_as_float(g << 21);
    if (!(fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)) >= t)) return 0u;
    return (x.x >= t ? 1u : 0u) | (x.y >= t ? 2u : 0u) | (x.z >= t ? 4u : 0u) |
           (x.w >= t ? 8u : 0u);
  }
};
struct KappaSrc {            // CriticalKV stage 2: stage-1 positions are forced, key 0
  static constexpr bool kTwo = true;
  const float* S;            // the head's scores
  const float* Cn;           // the head's ||(V W^O)_j||_1
  const uint32_t* F;         // the head's stage-1 bits (bits_mode)
  float eps;
  int C;
  bool bits_mode;
  uint32_t tau1;             // otherwise stage 1 kept key > tau1, and key == tau1 at
  int pcut1;                 // positions <= pcut1
  bool given;                // Cn already holds the stage-2 key (kappa itself)
  // stage-1 membership of position p with score s
  __device__ bool in1(int p, float s) const {
    if (p < 0 || p >= C) return false;
    if (bits_mode) return ((__ldcg(F + (p >> 5)) >> (p & 31)) & 1u) != 0u;
    const uint32_t k = score_key(s);
    return k > tau1 || (k == tau1 && p <= pcut1);
  }
  __device__ uint32_t kappa_key(float s, float c) const {
    return score_key(given ? c : __fmul_rn(__fadd_rn(s, eps), c)) + 1u;
  }
  __device__ void keys(const float4& x, const float4& y, int pos0, uint32_t (&k)[4],
                       bool (&f)[4]) const {
    const float xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      f[c] = in1(pos0 + c, xs[c]);
      k[c] = f[c] ? 0u : kappa_key(xs[c], ys[c]);
    }
  }
  __device__ uint32_t key_at(int i) const {
    const float s = S[i];
    return in1(i, s) ? 0u : kappa_key(s, Cn[i]);
  }
  __device__ bool forced_at(int i) const { return in1(i, S[i]); }
  // a listed entry with key k is forced exactly when k is 0 (a kappa key is at least 1)
  __device__ bool forced_key(uint32_t k) const { return k == 0u; }
  __device__ uint32_t full_max(const float4& x, const float4& y, int pos0) const {
    uint32_t k[4];
    bool f[4];
    keys(x, y, pos0, k, f);
    return max(max(k[0], k[1]), max(k[2], k[3]));
  }
  __device__ uint32_t cand_mask(const float4& x, const float4& y, int pos0, uint32_t g) const {
    uint32_t k[4];
    bool f[4];
    keys(x, y, pos0, k, f);
    uint32_t cm = 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) cm |= (f[c] || (k[c] >> 21) >= g) ? 1u << c : 0u;
    return cm;
  }
};

struct HeadSelSmem {
  uint32_t hist[2048];
  uint32_t scr[2 * 32 + 8];
  uint32_t res[2];
  int32_t upos[kUnion];       // the union, in position order, fills [fill, kUnion)
  uint32_t ukey[kUnion];
  uint64_t full[kSelStages];
};
using SelRing = BulkRing<kSelStages, kSelStage>;

// What select_head produces: the kept positions as rows, or as bits (the whole-head
// select only), or only tau and the position of the last kept tau-equal key (the
// streaming select only; CriticalKV stage 1).
enum { kOutRows = 0, kOutBits = 1, kOutTau = 2 };

// Ordered selection of one head's positions [0, C), keys and forced positions from `src`
// (staged values from stream base pointers s0 / s1 = flat index 0 of the arrays).  keep(j)
// = forced(j) || key(j) > tau || (key(j) == tau && j is among the keq lowest tau-equal
// positions), tau the K-th largest key.  kOutRows: kept positions in ascending order to
// kept[base + r] (rows >= cap skipped); kOutBits: bits of bits[] (the head's words);
// kOutTau: *tau_out = tau and *pcut_out = the position of the keq-th tau-equal key (-1 when
// keq is 0), so keep(j) = key(j) > tau || (key(j) == tau && j <= pcut).  Returns the number
// kept; ok turns false (the same in every thread) if a wait gave up.
template <int OUT, class Src>
__device__ uint32_t select_head(SelRing& R, HeadSelSmem& sm, unsigned char* ring_mem,
                                const Src& src, const float* s0, const float* s1, int64_t flat0,
                                int C, int64_t K, int32_t* kept, int64_t base, int64_t cap,
                                uint32_t* bits, int32_t* gpos, uint32_t* gkey, bool streaming,
                                bool& ok, uint32_t* tau_out = nullptr, int* pcut_out = nullptr) {
  constexpr bool BITS = OUT == kOutBits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t below = (1u << lane) - 1u;
  const bool any = K > 0;
  if (!any && !Src::kTwo) {   // nothing to select and nothing forced
    if (BITS)
      for (int wd = threadIdx.x; wd < (C + 31) / 32; wd += kSelThreads) bits[wd] = 0u;
    if (OUT == kOutTau && threadIdx.x == 0) {
      *tau_out = 0xFFFFFFFFu;
      *pcut_out = -1;
    }
    __syncthreads();
    return 0;
  }
  if (streaming) {
    // the aligned window [a0, a1) of flat indices goes through the ring; the < 4 keys of
    // the head past a1 (the tail) are read directly
    const int64_t a0 = flat0 & ~(int64_t)3;
    const int64_t a1 = max(a0, (flat0 + C) & ~(int64_t)3);
    const int64_t tail0 = max(a1, flat0), tailn = flat0 + C - tail0;
    const int64_t nbytes = (a1 - a0) * 4;
    const unsigned char* w0 = reinterpret_cast<const unsigned char*>(s0 + a0);
    const unsigned char* w1 = Src::kTwo ? reinterpret_cast<const unsigned char*>(s1 + a0) : nullptr;
    constexpr int kGroups = kSelStage / 16 / (Src::kTwo ? 2 : 1);   // per chunk
    // group j of a chunk at byte offset off: its keys, and which of them lie in the head
    auto group = [&](const unsigned char* st0, const unsigned char* st1, int64_t off, int j,
                     bool in, uint32_t (&k)[4], bool (&f)[4]) -> uint32_t {
      const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 x = in ? reinterpret_cast<const float4*>(st0)[j] : zero;
      const float4 y = (Src::kTwo && in) ? reinterpret_cast<const float4*>(st1)[j] : zero;
      const int pos0 = (int)(a0 + off / 4 + 4 * j - flat0);
      src.keys(x, y, pos0, k, f);
      uint32_t vm = 0u;
#pragma unroll
      for (int c = 0; c < 4; ++c) vm |= (in && (unsigned)(pos0 + c) < (unsigned)C) ? 1u << c : 0u;
      return vm;
    };

    // ---- pass A: first digit of every group's largest key
    uint32_t g = 2048u;   // with K == 0 only forced positions are candidates
    if (any) {
      for (int i = threadIdx.x; i < 2048; i += kSelThreads) sm.hist[i] = 0u;
      __syncthreads();
      ok = ring_pass(R, w0, w1, nbytes, false,
                     [&](const unsigned char* st0, const unsigned char* st1, int64_t off,
                         uint32_t bytes) {
        const int ng = (int)(bytes / 16);
        for (int jb = 0; jb < kGroups; jb += kSelThreads) {
          const int j = jb + (int)threadIdx.x;
          const int pos0 = (int)(a0 + off / 4 + 4 * j - flat0);
          uint32_t bin = kNoBin;
          if (j < ng) {
            const float4 x = reinterpret_cast<const float4*>(st0)[j];
            const float4 y = Src::kTwo ? reinterpret_cast<const float4*>(st1)[j] : x;
            if (pos0 >= 0 && pos0 + 3 < C) {
              bin = src.full_max(x, y, pos0) >> 21;
            } else {   // the head's first or last group
              uint32_t k[4];
              bool f[4];
              src.keys(x, y, pos0, k, f);
              uint32_t m = 0u;
              bool have = false;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                if ((unsigned)(pos0 + c) < (unsigned)C) {
                  m = max(m, k[c]);
                  have = true;
                }
              bin = have ? m >> 21 : kNoBin;
            }
          }
          hist_add_runs(sm.hist, bin);
        }
      });
      if (!ok) return 0;
      if (warp == 0) {   // the tail's keys form one more group
        uint32_t m = 0u;
        for (int64_t i = tail0; i < tail0 + tailn; ++i) m = max(m, src.key_at((int)(i - flat0)));
        hist_add_runs(sm.hist, (lane == 0 && tailn > 0) ? m >> 21 : kNoBin);
      }
      __syncthreads();
      block_pick<kSelThreads>(sm.hist, 2048, (uint32_t)K, sm.scr, sm.res);
      __syncthreads();
      g = sm.res[0];
      __syncthreads();
    }

    // ---- pass B: the union of keys with first digit >= g and forced positions, filled from
    // the end of the buffer backwards (chunks come last to first), so it ends up ascending
    uint32_t fill = kUnion;
    bool spilled = false;   // the union moved to the head's global region (C entries)
    if (threadIdx.x == 0) {
      uint32_t fl = kUnion;
      for (int64_t i = tail0 + tailn - 1; i >= tail0; --i) {
        const int p = (int)(i - flat0);
        const uint32_t k = src.key_at(p);
        if (src.forced_at(p) || (k >> 21) >= g) {
          --fl;
          sm.upos[fl] = p;
          sm.ukey[fl] = k;
        }
      }
      sm.res[0] = fl;
    }
    __syncthreads();
    fill = sm.res[0];
    __syncthreads();
    constexpr int kPerWarp = kGroups / kSelWarps;   // groups of a chunk per warp, in order
    ok = ring_pass(R, w0, w1, nbytes, true,
                   [&](const unsigned char* st0, const unsigned char* st1, int64_t off,
                       uint32_t bytes) {
      const int ng = (int)(bytes / 16);
      auto cand = [&](int j) -> uint32_t {
        if (j >= ng) return 0u;
        const float4 x = reinterpret_cast<const float4*>(st0)[j];
        const float4 y = Src::kTwo ? reinterpret_cast<const float4*>(st1)[j] : x;
        const int pos0 = (int)(a0 + off / 4 + 4 * j - flat0);
        uint32_t cm = src.cand_mask(x, y, pos0, g);
        if (pos0 < 0 || pos0 + 3 >= C) {   // the head's first or last group
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if ((unsigned)(pos0 + c) >= (unsigned)C) cm &= ~(1u << c);
        }
        return cm;
      };
      uint32_t cmu[kPerWarp / 32];   // candidate masks of this lane's groups
      uint32_t wc = 0;                // this warp's candidates in the chunk
#pragma unroll
      for (int u = 0; u < kPerWarp / 32; ++u) {
        cmu[u] = cand(warp * kPerWarp + u * 32 + lane);
        wc += __popc(cmu[u]);
      }
      wc = warp_sum_u(wc);
      if (lane == 0) sm.scr[warp] = wc;
      __syncthreads();
      // the warps' counts, scanned across the lanes of every warp
      uint32_t c = lane < kSelWarps ? sm.scr[lane] : 0u, ci = c;
#pragma unroll
      for (int d = 1; d < kSelWarps; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, ci, d);
        if (lane >= d) ci += y;
      }
      const uint32_t T = __shfl_sync(0xFFFFFFFFu, ci, kSelWarps - 1);
      const uint32_t before = __shfl_sync(0xFFFFFFFFu, ci - c, warp);
      if (T == 0u) return;   // the same in every thread
      if (!spilled && T > fill) {
        // the shared-memory union is full: move it to the end of the head's global region
        // (room for every key of the head) and go on there
        const uint32_t n = kUnion - fill;
        for (uint32_t t = threadIdx.x; t < n; t += kSelThreads) {
          gpos[C - n + t] = sm.upos[fill + t];
          gkey[C - n + t] = sm.ukey[fill + t];
        }
        fill = (uint32_t)C - n;
        spilled = true;      // the same in every thread
      }
      int32_t* UP = spilled ? gpos : sm.upos;
      uint32_t* UK = spilled ? gkey : sm.ukey;
      uint32_t o = fill - T + before;
#pragma unroll
      for (int u = 0; u < kPerWarp / 32; ++u) {
        const int j = warp * kPerWarp + u * 32 + lane;
        const uint32_t n = __popc(cmu[u]);
        uint32_t incl = n;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
          if (lane >= d) incl += y;
        }
        if (cmu[u]) {
          uint32_t k[4];
          bool f[4];
          (void)group(st0, st1, off, j, true, k, f);
          uint32_t q = o + incl - n;
          const int pos0 = (int)(a0 + off / 4 + 4 * j - flat0);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if ((cmu[u] >> c) & 1u) {
              UP[q] = pos0 + c;
              UK[q] = k[c];
              ++q;
            }
          }
        }
        o += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      fill -= T;
    });
    if (!ok) return 0;
    {
      const int u0 = (int)fill, nu = (spilled ? C : kUnion) - (int)fill;
      // the union's entries (written by this CTA before the last barrier of the pass)
      auto ukey_at = [&](int t) -> uint32_t { return spilled ? gkey[t] : sm.ukey[t]; };
      auto upos_at = [&](int t) -> int { return spilled ? gpos[t] : sm.upos[t]; };
      // ---- tau and keq over the union (every key above tau, and tau's first digit, is in it)
      uint32_t prefix = 0, mask = 0, krem = any ? (uint32_t)K : 0u;
      if (any) {
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
          const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
          const int nb = pass == 2 ? 1024 : 2048;
          for (int i = threadIdx.x; i < nb; i += kSelThreads) sm.hist[i] = 0u;
          __syncthreads();
          for (int b0 = 0; b0 < nu; b0 += 8 * kSelThreads) {
            uint32_t kk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int t = b0 + u * kSelThreads + (int)threadIdx.x;
              kk[u] = t < nu ? ukey_at(u0 + t) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int t = b0 + u * kSelThreads + (int)threadIdx.x;
              // (forced positions have key 0: counted like every key, as in the full select)
              const bool in =
                  t < nu && (pass == 0 ? (kk[u] >> 21) >= g : (kk[u] & mask) == prefix);
              hist_add_runs(sm.hist, in ? (kk[u] >> sh) & (uint32_t)(nb - 1) : kNoBin);
            }
          }
          __syncthreads();
          block_pick<kSelThreads>(sm.hist, nb, krem, sm.scr, sm.res);
          __syncthreads();
          prefix |= sm.res[0] << sh;
          mask |= (uint32_t)(nb - 1) << sh;
          krem = sm.res[1];
          __syncthreads();
        }
      }
      const uint32_t tau = any ? prefix : 0xFFFFFFFFu;   // no key equals 0xFFFFFFFF
      const uint32_t keq = any ? krem : 0u;
      // ---- ordered emission: warp w takes a contiguous slice of the union
      const int per = (nu + kSelWarps - 1) / kSelWarps;
      const int e0 = u0 + min(nu, warp * per), e1 = u0 + min(nu, warp * per + per);
      uint32_t nkeep = 0, neq = 0;
      for (int t = e0 + lane; t < e1; t += 32) {
        const uint32_t k = ukey_at(t);
        const bool f = src.forced_key(k);
        nkeep += (f || k > tau) ? 1u : 0u;
        neq += (!f && k == tau) ? 1u : 0u;
      }
      nkeep = warp_sum_u(nkeep);
      neq = warp_sum_u(neq);
      if (lane == 0) {
        sm.scr[warp] = nkeep;
        sm.scr[32 + warp] = neq;
      }
      __syncthreads();
      if (OUT == kOutTau) {
        // the keq-th tau-equal entry of the union: the warp whose slice holds it finds it
        uint32_t eqb = 0;
        for (int w = 0; w < warp; ++w) eqb += sm.scr[32 + w];
        const uint32_t mine = sm.scr[32 + warp];
        if (keq > 0u && eqb < keq && keq <= eqb + mine) {
          uint32_t seen = eqb;
          for (int tb = e0; tb < e1; tb += 32) {
            const int t = tb + lane;
            const uint32_t k = t < e1 ? ukey_at(t) : 0u;
            const bool iseq = t < e1 && !src.forced_key(k) && k == tau;
            const uint32_t meq = __ballot_sync(0xFFFFFFFFu, iseq);
            if (iseq && seen + __popc(meq & below) + 1u == keq) sm.res[0] = (uint32_t)upos_at(t);
            seen += __popc(meq);
            if (seen >= keq) break;   // the same in every lane
          }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
          *tau_out = tau;
          *pcut_out = keq > 0u ? (int)sm.res[0] : -1;
        }
        __syncthreads();
        return 0;
      }
      uint32_t eqc = 0, outc = 0, total = 0;
      {
        uint32_t eq = 0;
        for (int w = 0; w < kSelWarps; ++w) {
          const uint32_t e = sm.scr[32 + w];
          const uint32_t take = eq >= keq ? 0u : (keq - eq < e ? keq - eq : e);
          if (w == warp) {
            eqc = eq;
            outc = total;
          }
          total += sm.scr[w] + take;
          eq += e;
        }
      }
      for (int tb = e0; tb < e1; tb += 32) {
        const int t = tb + lane;
        const bool in = t < e1;
        const uint32_t k = in ? ukey_at(t) : 0u;
        const int j = in ? upos_at(t) : 0;
        const bool f = in && src.forced_key(k);
        const bool iseq = in && !f && k == tau;
        bool keep = in && (f || k > tau);
        const uint32_t meq = __ballot_sync(0xFFFFFFFFu, iseq);
        if (iseq && eqc + __popc(meq & below) < keq) keep = true;
        const uint32_t mk = __ballot_sync(0xFFFFFFFFu, keep);
        if (keep) {
          const int64_t row = base + outc + __popc(mk & below);
          if (row < cap) kept[row] = j;
        }
        eqc += __popc(meq);
        outc += __popc(mk);
      }
      __syncthreads();   // the union and scr are reused by the next selection
      return total;
    }
  }
  // ---- the radix select over the whole head, keys read from global memory; the ring's
  // memory (no copy in flight) holds its state
  ClusterSelectSmem& cs = *reinterpret_cast<ClusterSelectSmem*>(ring_mem);
  const uint32_t total = cluster_topk_select<kSelThreads, BITS>(
      0, C, K, [&](int j) { return src.key_at(j); }, [&](int j) { return src.forced_at(j); },
      kept, base, cap, bits, cs);
  __syncthreads();
  return total;
}

// One CTA per head: threshold(s), ordered kept positions, window and reserve rows.
template <bool CRIT>
__global__ void __launch_bounds__(kSelThreads, 2)
head_select(const float* __restrict__ scores, const float* __restrict__ crit, uint32_t can,
            uint32_t cad, float ceps, int kappa_given, const int32_t* __restrict__ lens,
            const int64_t* __restrict__ cu, int Hkv, int C, int w, int reserve,
            int32_t* __restrict__ kept, int64_t cap, uint32_t* __restrict__ flags, int64_t words,
            int32_t* __restrict__ gpos, uint32_t* __restrict__ gkey, int streaming,
            WsHeader* hdr) {
  __shared__ HeadSelSmem sm;
  extern __shared__ __align__(128) unsigned char ring_mem[];
  const int64_t h = blockIdx.x;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g];
  const int64_t Bg = (int64_t)lens[h] - w;   // lens was clamped to [w, n]
  const int64_t flat0 = h * (int64_t)C;
  SelRing R;
  R.init(ring_mem, sm.full);
  __syncthreads();
  bool ok = true;
  uint32_t n = 0;
  if (!CRIT) {
    const ScoreSrc src{scores + flat0};
    n = select_head<kOutRows>(R, sm, ring_mem, src, scores, nullptr, flat0, C, Bg, kept, base,
                              cap, nullptr, gpos + flat0, gkey + flat0, streaming != 0, ok);
  } else {
    uint32_t* F = flags + h * words;
    const int64_t K1 = ((int64_t)can * Bg) / cad;
    const int64_t K2 = Bg - K1;
    const ScoreSrc src1{scores + flat0};
    KappaSrc src2{scores + flat0, crit + flat0, F, ceps, C, false, 0u, -1, kappa_given != 0};
    if (streaming) {
      // stage 1 yields its threshold and tie cut; stage 2 tests membership from the score
      __shared__ uint32_t tau1;
      __shared__ int pcut1;
      (void)select_head<kOutTau>(R, sm, ring_mem, src1, scores, nullptr, flat0, C, K1, nullptr,
                                 0, 0, nullptr, gpos + flat0, gkey + flat0, true, ok, &tau1,
                                 &pcut1);
      __syncthreads();
      src2.tau1 = tau1;
      src2.pcut1 = pcut1;
    } else {
      (void)select_head<kOutBits>(R, sm, ring_mem, src1, scores, nullptr, flat0, C, K1, nullptr,
                                  0, 0, F, gpos + flat0, gkey + flat0, false, ok);
      __syncthreads();   // the stage-1 bits are complete
      src2.bits_mode = true;
    }
    if (ok)
      n = select_head<kOutRows>(R, sm, ring_mem, src2, scores, crit, flat0, C, K2, kept, base,
                                cap, nullptr, gpos + flat0, gkey + flat0, streaming != 0, ok);
  }
  if (threadIdx.x == 0) {
    if (!ok) raise_dev(hdr, DEV_WAIT_TIMEOUT, 0x800u + (unsigned)(h & 0xFF));
    else if (n != (uint32_t)Bg) raise_dev(hdr, DEV_SELECT, (unsigned)h);
  }
  for (int t = threadIdx.x; t < w + reserve; t += kSelThreads) {
    const int64_t row = base + Bg + t;
    if (row < cap) kept[row] = t < w ? C + t : -1;
  }
}

// Copy the kept rows of K and V into the flat buffers, 16 bytes per thread.
__global__ void __launch_bounds__(kGatherThreads)
compact_gather(const char* __restrict__ k, const char* __restrict__ v,
               const int32_t* __restrict__ kept, const int64_t* __restrict__ cu,
               const int32_t* __restrict__ lens, int Hkv, int n, int row_bytes, int64_t cap,
               char* __restrict__ kf, char* __restrict__ vf) {
  const int64_t h = blockIdx.y;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g];
  const int64_t len = lens[h];
  const int vecs = row_bytes >> 4;
  const char* Ks = k + h * (int64_t)n * row_bytes;
  const char* Vs = v + h * (int64_t)n * row_bytes;
  const int64_t total = len * vecs;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / vecs;
    const int c = (int)(idx - r * vecs);
    const int64_t row = base + r;
    if (row >= cap) continue;
    const int64_t src = kept[row];
    if (src < 0 || src >= n) continue;   // never read outside the source head
    const uint4 a = reinterpret_cast<const uint4*>(Ks + src * row_bytes)[c];
    const uint4 b = reinterpret_cast<const uint4*>(Vs + src * row_bytes)[c];
    reinterpret_cast<uint4*>(kf + row * row_bytes)[c] = a;
    reinterpret_cast<uint4*>(vf + row * row_bytes)[c] = b;
  }
}

// KVEVICT_SELECT_PATH=global forces the radix select over the whole head with the keys read
// from global memory (the path a candidate union too long for shared memory takes); tests
// compare the two.
static bool global_select_forced() {
  const char* e = std::getenv("KVEVICT_SELECT_PATH");
  return e != nullptr && std::strcmp(e, "global") == 0;
}

CompactPlan compact_plan(const Shape& s, bool critical) {
  CompactPlan p{};
  size_t off = kWsHeader;
  p.off_flags = off;
  p.flag_words = critical ? cdiv(s.C() > 0 ? s.C() : 1, 32) : 0;
  off += align_up((size_t)s.units() * p.flag_words * sizeof(uint32_t), 256);
  // a head's candidate union, when it outgrows shared memory: room for every key
  p.off_union = off;
  off += align_up((size_t)s.units() * (s.C() > 0 ? s.C() : 0) * sizeof(int32_t), 256);
  off += align_up((size_t)s.units() * (s.C() > 0 ? s.C() : 0) * sizeof(uint32_t), 256);
  p.off_end = off;
  return p;
}

cudaError_t launch_compact(const Shape& s, const void* k, const void* v, const float* scores,
                           const float* crit, uint32_t can, uint32_t cad, float ceps,
                           bool kappa_given, const int32_t* head_budget, int reserve,
                           int32_t* kept, int64_t* cu, int32_t* lens, void* kf, void* vf,
                           int64_t cap, char* ws, const CompactPlan& p, cudaStream_t st,
                           const int64_t* row_base) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t H = s.units();
  compact_offsets<<<1, kScanThreads, 0, st>>>(head_budget, H, s.Hkv, s.w, s.n, reserve, cap,
                                               row_base, cu, lens, hdr);
  if (H > 0) {
    const int C = s.C();
    // the bulk copies need 16-byte aligned score (and norm) arrays
    const bool streaming = C > 0 && !global_select_forced() &&
                           (reinterpret_cast<uintptr_t>(scores) & 15u) == 0 &&
                           (crit == nullptr || (reinterpret_cast<uintptr_t>(crit) & 15u) == 0);
    const size_t ring_bytes = (size_t)kSelStages * kSelStage;
    int32_t* gpos = reinterpret_cast<int32_t*>(ws + p.off_union);
    uint32_t* gkey = reinterpret_cast<uint32_t*>(
        ws + p.off_union + align_up((size_t)H * C * sizeof(int32_t), 256));
    auto kern = crit ? head_select<true> : head_select<false>;
    static std::atomic<int> opted[2][kMaxDevices];   // per kernel, per device
    const int ok = per_device(opted[crit ? 1 : 0], [&]() {
      return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)ring_bytes) == cudaSuccess ? 1 : 0;
    });
    if (!ok) return cudaErrorInvalidConfiguration;
    // a cluster of one CTA: the whole-head fallback's cluster barriers are the block's own
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)H);
    cfg.blockDim = dim3(kSelThreads);
    cfg.dynamicSmemBytes = ring_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(
        &cfg, kern, scores, crit, can, cad, ceps, kappa_given ? 1 : 0, (const int32_t*)lens,
        (const int64_t*)cu, s.Hkv,
        C, s.w, reserve, kept, cap, reinterpret_cast<uint32_t*>(ws + p.off_flags), p.flag_words,
        gpos, gkey, streaming ? 1 : 0, hdr);
    if (e != cudaSuccess) return e;
  }
  const int row_bytes = s.d * s.esize();
  int gx = (int)cdiv((int64_t)num_sms() * 16, H);
  if (gx < 1) gx = 1;
  if (gx > 64) gx = 64;
  compact_gather<<<dim3(gx, (unsigned)H), kGatherThreads, 0, st>>>(
      (const char*)k, (const char*)v, kept, cu, lens, s.Hkv, s.n, row_bytes, cap, (char*)kf,
      (char*)vf);
  count_launches(3);
  return cudaGetLastError();
}

// StreamingLLM preset: head h keeps its first min(sinks, B_g) positions and the most recent
// B_g - that many before the window, then the window C..n-1; reserve rows get -1.
__global__ void __launch_bounds__(kGatherThreads)
streaming_kept(const int64_t* __restrict__ cu, const int32_t* __restrict__ lens, int Hkv, int C,
               int w, int sinks, int reserve, int64_t cap, int32_t* __restrict__ kept) {
  const int64_t h = blockIdx.y;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g];
  const int64_t Bg = (int64_t)lens[h] - w;   // lens was clamped to [w, n]
  const int64_t sk = Bg < sinks ? Bg : sinks;
  const int64_t total = Bg + w + reserve;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = base + i;
    if (row < 0 || row >= cap) continue;
    int64_t pos;
    if (i < sk) pos = i;
    else if (i < Bg) pos = C - (Bg - sk) + (i - sk);
    else if (i < Bg + w) pos = C + (i - Bg);
    else pos = -1;
    kept[row] = (int32_t)pos;
  }
}

cudaError_t launch_compact_streaming(const Shape& s, const void* k, const void* v, int sinks,
                                     const int32_t* head_budget, int reserve, int32_t* kept,
                                     int64_t* cu, int32_t* lens, void* kf, void* vf, int64_t cap,
                                     char* ws, cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t H = s.units();
  compact_offsets<<<1, kScanThreads, 0, st>>>(head_budget, H, s.Hkv, s.w, s.n, reserve, cap,
                                               nullptr, cu, lens, hdr);
  int gx = (int)cdiv((int64_t)num_sms() * 16, H);
  if (gx < 1) gx = 1;
  if (gx > 64) gx = 64;
  streaming_kept<<<dim3(gx, (unsigned)H), kGatherThreads, 0, st>>>(cu, lens, s.Hkv, s.C(), s.w,
                                                                    sinks, reserve, cap, kept);
  const int row_bytes = s.d * s.esize();
  compact_gather<<<dim3(gx, (unsigned)H), kGatherThreads, 0, st>>>(
      (const char*)k, (const char*)v, kept, cu, lens, s.Hkv, s.n, row_bytes, cap, (char*)kf,
      (char*)vf);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace kv
