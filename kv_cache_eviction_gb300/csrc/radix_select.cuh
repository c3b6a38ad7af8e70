// Radix select of the K largest 32-bit keys of one head, and the ordered selection that
// follows it, over the CTAs of one thread-block cluster.
//
// Used for the per-head Top-B_g of Ada-KV Algorithm 2 and for both stages of the
// CriticalKV selection.  No sort: three histogram passes over the keys (11, 11 and 10
// bits, most significant first) narrow down tau, the K-th largest key.  The result is
// (tau, keq): every key > tau is selected, plus the keq lowest-position keys equal to tau,
// which is the (key desc, position asc) total order.
//
// Each CTA of the cluster owns a contiguous slice of the positions.  It builds its own
// histogram in shared memory; the slices' histograms are summed into rank 0's shared memory
// with distributed-shared-memory atomics, rank 0 finds the bin that holds the K-th key,
// and every CTA reads the result back from rank 0.  A kernel launched without a cluster
// is a cluster of one CTA and runs the same code.
//
// Only the first pass has to look at every key.  Once the first digit of tau is known, a
// key whose first digit is smaller can be neither selected nor tau-equal, so each warp lists
// the positions of its slice that remain (first digit at or above tau's, or forced), in
// position order, in shared memory; the later passes and the ordered selection walk the
// lists.  A CTA with a list that overflows walks its whole slice instead (same results).
#pragma once

#include <cooperative_groups.h>

#include "kv_common.cuh"

namespace kv {

namespace cg = cooperative_groups;

constexpr int kMaxCluster = 8;
constexpr int kListCap = 4096;   // candidate positions per CTA, split evenly over its warps

struct ClusterSelectSmem {
  uint32_t hist[2048];              // this CTA's histogram of the current pass
  uint32_t ghist[2048];             // rank 0: the cluster's histogram
  uint32_t scr[128];                // block scans and per-warp counts / offsets
  uint32_t res[2];                  // rank 0: (bin, rank of the K-th key within it)
  uint32_t cnt[kMaxCluster][2];     // rank 0: (keys kept outright, tau-equal keys) per rank
  uint32_t lcount[32];              // candidates listed by each warp
  uint32_t lover;                   // some warp's list overflowed
  uint32_t gath, gtot;              // the union of the lists is gathered; its length
  uint32_t ustart[kMaxCluster * 32 + 1];   // start of (rank, warp)'s list in the union
  int32_t list[kListCap];           // warp w: list[w * kListCap / warps ...]
};

// Union of the cluster's candidate keys gathered into one CTA (the ghist words of a CTA
// other than the pick's rank 0 are free by then, and rank 0's after its last pick).
constexpr int kUnionCap = 2048;

// One CTA: the bin of histogram h (nb bins) holding the krem-th largest key, counted from
// the top, and krem's rank inside it, into res[0..1]; with fewer than krem keys in all, bin
// 0 (a caller's bound then covers every key).  All threads call it; scr holds the scan.
template <int BLOCK>
__device__ void block_pick(const uint32_t* h, int nb, uint32_t krem, uint32_t* scr,
                           uint32_t* res) {
  if (threadIdx.x == 0) {
    res[0] = 0u;
    res[1] = krem;
  }
  // thread t owns reversed bins [t*per, (t+1)*per)
  const int per = nb / BLOCK;
  uint32_t local = 0;
  for (int q = 0; q < per; ++q) local += h[nb - 1 - ((int)threadIdx.x * per + q)];
  uint32_t total;
  const uint32_t incl = block_incl_scan(local, scr, &total);   // ends with a barrier
  const uint32_t excl = incl - local;
  if (excl < krem && krem <= incl) {
    uint32_t acc = excl;
    for (int q = 0; q < per; ++q) {
      const int bin = nb - 1 - ((int)threadIdx.x * per + q);
      const uint32_t c = h[bin];
      if (acc + c >= krem) {
        res[0] = (uint32_t)bin;
        res[1] = krem - acc;
        break;
      }
      acc += c;
    }
  }
}

// Sums this CTA's histogram of the pass (nb bins, complete in sm.hist) into rank 0's, lets
// rank 0 find the bin holding the krem-th largest key (bins counted from the top), and
// returns (bin, krem's rank inside it) to every thread of every CTA.  Rank 0 clears its
// cluster histogram for the next pass.
template <int BLOCK>
__device__ void cluster_pick(ClusterSelectSmem& sm, int nb, uint32_t krem, uint32_t& bin_out,
                             uint32_t& kr_out) {
  cg::cluster_group cl = cg::this_cluster();
  const bool lead = cl.block_rank() == 0;
  uint32_t* lead_g = cl.map_shared_rank(sm.ghist, 0);
  const uint32_t* lead_res = cl.map_shared_rank(sm.res, 0);
  __syncthreads();
  for (int i = threadIdx.x; i < nb; i += BLOCK) {
    const uint32_t c = sm.hist[i];
    if (c) atomicAdd(lead_g + i, c);
  }
  cl.sync();
  if (lead) {
    block_pick<BLOCK>(sm.ghist, nb, krem, sm.scr, sm.res);
    __syncthreads();
    for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.ghist[i] = 0u;   // next pass
  }
  cl.sync();
  // rank 0 writes res again only after the next pass's first cluster barrier, which every
  // CTA reaches after this read
  bin_out = lead_res[0];
  kr_out = lead_res[1];
}

// Given per-warp counts in sm.scr[w] (kept outright) and sm.scr[32 + w] (tau-equal), in
// position order of the warps, exchanges the CTAs' totals through rank 0 (or, with
// have_totals, takes every rank's totals from this CTA's sm.cnt) and leaves in
// sm.scr[64 + w] the tau-equal keys and in sm.scr[96 + w] the kept positions of the whole
// cluster that come before warp w's first position.  Returns the cluster's kept count.
template <int BLOCK>
__device__ uint32_t cluster_order_offsets(ClusterSelectSmem& sm, uint32_t keq,
                                          bool have_totals = false) {
  constexpr int NW = BLOCK / 32;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank(), ncta = (int)cl.num_blocks();
  __syncthreads();
  if (!have_totals) {
    if (threadIdx.x == 0) {
      uint32_t g = 0, e = 0;
      for (int w = 0; w < NW; ++w) {
        g += sm.scr[w];
        e += sm.scr[32 + w];
      }
      uint32_t* lc = cl.map_shared_rank(&sm.cnt[0][0], 0);
      lc[2 * rank] = g;
      lc[2 * rank + 1] = e;
    }
    cl.sync();
  }
  if (threadIdx.x == 0) {
    // every rank's totals: rank 0's copy, or this CTA's own (have_totals)
    const uint32_t* lc = have_totals ? &sm.cnt[0][0] : cl.map_shared_rank(&sm.cnt[0][0], 0);
    // the tau-equal quota goes to the lowest positions: to the ranks in order, then to the
    // warps of this CTA in order
    uint32_t eq = 0, total = 0, out = 0, eqc = 0;
    for (int r = 0; r < ncta; ++r) {
      const uint32_t g = lc[2 * r], e = lc[2 * r + 1];
      const uint32_t take = eq >= keq ? 0u : (keq - eq < e ? keq - eq : e);
      if (r < rank) {
        out += g + take;   // kept positions of the ranks before this one
        eqc += e;          // tau-equal keys of the ranks before this one
      }
      total += g + take;
      eq += e;
    }
    for (int w = 0; w < NW; ++w) {
      const uint32_t e = sm.scr[32 + w];
      const uint32_t take = eqc >= keq ? 0u : (keq - eqc < e ? keq - eqc : e);
      sm.scr[64 + w] = eqc;
      sm.scr[96 + w] = out;
      out += sm.scr[w] + take;
      eqc += e;
    }
    sm.scr[0] = total;
  }
  __syncthreads();
  const uint32_t total = sm.scr[0];
  __syncthreads();   // scr[0] is a per-warp count again in the caller's next use
  return total;
}

// Top-K selection over the cluster's positions: keep(j) = forced(j) || key(j) > tau ||
// (key(j) == tau && rank of j among the tau-equal keys of all CTAs < keq), tau the K-th
// largest key.  Positions [p0, p1) are this CTA's; every CTA of the cluster calls it with
// the same K (K <= the number of non-forced positions of all CTAs).  Kept positions go,
// ascending over the whole cluster, to kept[base + r] (rows >= cap are skipped) or, with
// BITS, as one bit per position to bits[j / 32] (p0 must then be a multiple of 32).  key(j)
// and forced(j) must give the same answer on every call.  Returns the cluster's number of
// kept positions.
template <int BLOCK, bool BITS, typename KeyFn, typename ForcedFn>
__device__ uint32_t cluster_topk_select(int p0, int p1, int64_t K, KeyFn key, ForcedFn forced,
                                        int32_t* kept, int64_t base, int64_t cap,
                                        uint32_t* bits, ClusterSelectSmem& sm) {
  static_assert(BLOCK <= 1024 && (1024 % BLOCK) == 0, "block must divide 1024");
  constexpr int NW = BLOCK / 32;
  constexpr int LW = kListCap / NW;   // list entries per warp
  constexpr int U = 8;                // keys per thread fetched before use
  cg::cluster_group cl = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t below = (1u << lane) - 1u;
  if (threadIdx.x == 0) sm.lover = 0u;
  if (cl.block_rank() == 0)
    for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.ghist[i] = 0u;
  cl.sync();

  // ---- first digit, over every key of the CTA
  const bool any = K > 0;   // the same in every CTA
  uint32_t prefix = 0, mask = 0, krem = any ? (uint32_t)K : 0u;
  uint32_t bin0 = 2048u;    // with K == 0 no key is a candidate: only forced positions
  if (any) {
    for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.hist[i] = 0u;
    __syncthreads();
    for (int b0 = p0; b0 < p1; b0 += U * BLOCK) {
      uint32_t kk[U];
      bool valid[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int i = b0 + k * BLOCK + (int)threadIdx.x;
        valid[k] = i < p1;
        kk[k] = valid[k] ? key(i) : 0u;
      }
#pragma unroll
      for (int k = 0; k < U; ++k) hist_add_runs(sm.hist, valid[k] ? kk[k] >> 21 : 0xFFFFFFFFu);
    }
    uint32_t b, kr;
    cluster_pick<BLOCK>(sm, 2048, krem, b, kr);
    prefix = b << 21;
    mask = 0x7FFu << 21;
    krem = kr;
    bin0 = b;
  }

  // ---- candidate lists: warp w lists, in order, the positions of its slice whose first
  // digit is >= bin0 or that are forced
  const int n = p1 > p0 ? p1 - p0 : 0;
  const int per = (((n + NW - 1) / NW) + 31) & ~31;   // slice length, a multiple of 32
  const int s0 = min(p1, p0 + warp * per), s1 = min(p1, s0 + per);
  int32_t* L = sm.list + warp * LW;
  {
    uint32_t lc = 0;
    bool over = false;
    for (int jb = s0; jb < s1 && !over; jb += 32 * U) {
      uint32_t kk[U];
      bool ff[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = jb + 32 * u + lane;
        kk[u] = j < s1 ? key(j) : 0u;
        ff[u] = j < s1 ? forced(j) : false;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = jb + 32 * u + lane;
        const bool c = j < s1 && (ff[u] || (kk[u] >> 21) >= bin0);
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, c);
        if (lc + __popc(m) > (uint32_t)LW) {
          over = true;   // the same in every lane
        } else if (!over) {
          if (c) L[lc + __popc(m & below)] = j;
          lc += __popc(m);
        }
      }
    }
    if (lane == 0) {
      sm.lcount[warp] = lc;
      if (over) sm.lover = 1u;
    }
  }
  __syncthreads();
  const bool listed = sm.lover == 0u;   // the same in every thread of the CTA
  const int cw = listed ? (int)sm.lcount[warp] : 0;

  // ---- remaining digits
  if (any) {
#pragma unroll 1
    for (int pass = 1; pass < 3; ++pass) {
      const int sh = pass == 1 ? 10 : 0;
      const int nb = pass == 2 ? 1024 : 2048;
      for (int i = threadIdx.x; i < nb; i += BLOCK) sm.hist[i] = 0u;
      __syncthreads();
      auto add = [&](uint32_t k, bool ok) {
        hist_add_runs(sm.hist, (ok && (k & mask) == prefix) ? (k >> sh) & (uint32_t)(nb - 1)
                                                            : 0xFFFFFFFFu);
      };
      if (listed) {
        for (int b = 0; b < cw; b += 32 * U) {
          uint32_t kk[U];
          bool ok[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int idx = b + 32 * u + lane;
            ok[u] = idx < cw;
            kk[u] = ok[u] ? key(L[idx]) : 0u;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) add(kk[u], ok[u]);
        }
      } else {
        for (int b0 = p0; b0 < p1; b0 += U * BLOCK) {
          uint32_t kk[U];
          bool ok[U];
#pragma unroll
          for (int k = 0; k < U; ++k) {
            const int i = b0 + k * BLOCK + (int)threadIdx.x;
            ok[k] = i < p1;
            kk[k] = ok[k] ? key(i) : 0u;
          }
#pragma unroll
          for (int k = 0; k < U; ++k) add(kk[k], ok[k]);
        }
      }
      uint32_t b, kr;
      cluster_pick<BLOCK>(sm, nb, krem, b, kr);
      prefix |= b << sh;
      mask |= (uint32_t)(nb - 1) << sh;
      krem = kr;
    }
  }
  const uint32_t tau = any ? prefix : 0xFFFFFFFFu;   // no key equals 0xFFFFFFFF
  const uint32_t keq = any ? krem : 0u;

  // ---- ordered selection: per-warp counts, cluster offsets, then each warp emits in order
  uint32_t nkeep = 0, neq = 0;
  if (listed) {
    for (int idx = lane; idx < cw; idx += 32) {
      const int j = L[idx];
      const bool f = forced(j);
      const uint32_t k = key(j);
      nkeep += (f || k > tau) ? 1u : 0u;
      neq += (!f && k == tau) ? 1u : 0u;
    }
  } else {
    for (int jb = s0; jb < s1; jb += 32 * U) {
      uint32_t kk[U];
      bool ff[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = jb + 32 * u + lane;
        kk[u] = j < s1 ? key(j) : 0u;
        ff[u] = j < s1 ? forced(j) : false;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool in = jb + 32 * u + lane < s1;
        nkeep += (in && (ff[u] || kk[u] > tau)) ? 1u : 0u;
        neq += (in && !ff[u] && kk[u] == tau) ? 1u : 0u;
      }
    }
  }
  nkeep = warp_sum_u(nkeep);
  neq = warp_sum_u(neq);
  if (lane == 0) {
    sm.scr[warp] = nkeep;
    sm.scr[32 + warp] = neq;
  }
  if (BITS && listed) {
    // the CTA's words start clear; kept bits are then set one by one
    for (int wd = p0 / 32 + (int)threadIdx.x; wd < (p1 + 31) / 32; wd += BLOCK) bits[wd] = 0u;
  }
  const uint32_t total = cluster_order_offsets<BLOCK>(sm, keq);
  uint32_t eqc = sm.scr[64 + warp], outc = sm.scr[96 + warp];
  auto emit = [&](int j, bool in, uint32_t k, bool f) {
    const bool iseq = in && !f && k == tau;
    bool keep = in && (f || k > tau);
    const uint32_t meq = __ballot_sync(0xFFFFFFFFu, iseq);
    if (iseq && eqc + __popc(meq & below) < keq) keep = true;
    const uint32_t mk = __ballot_sync(0xFFFFFFFFu, keep);
    if (BITS) {
      if (listed) {
        if (keep) atomicOr(bits + (j >> 5), 1u << (j & 31));
      } else if (lane == 0) {
        bits[(j - lane) >> 5] = mk;   // j - lane: the word's first position
      }
    } else if (keep) {
      const int64_t row = base + outc + __popc(mk & below);
      if (row < cap) kept[row] = j;
    }
    eqc += __popc(meq);
    outc += __popc(mk);
  };
  if (listed) {
    for (int b = 0; b < cw; b += 32) {
      const int idx = b + lane;
      const bool in = idx < cw;
      const int j = in ? L[idx] : 0;
      emit(j, in, in ? key(j) : 0u, in ? forced(j) : false);
    }
  } else {
    for (int jb = s0; jb < s1; jb += 32 * U) {
      uint32_t kk[U];
      bool ff[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = jb + 32 * u + lane;
        kk[u] = j < s1 ? key(j) : 0u;
        ff[u] = j < s1 ? forced(j) : false;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j0 = jb + 32 * u;
        if (j0 >= s1) break;   // uniform across the warp
        emit(j0 + lane, j0 + lane < s1, kk[u], ff[u]);
      }
    }
  }
  __syncthreads();   // lists and scr are reused by the next call
  return total;
}

// Keys of a staged span: the selection reads 32-bit raw values from shared memory and maps
// them to keys.  Scores: the raw value is the fp32 score, the key its score_key, nothing is
// forced.  Stored keys: the raw value is the key itself and 0 marks a forced position.
struct ScoreKeys {
  static __device__ __forceinline__ uint32_t key(uint32_t raw) {
    return score_key(__uint_as_float(raw));
  }
  static __device__ __forceinline__ bool forced(uint32_t) { return false; }
};
struct StoredKeys {
  static __device__ __forceinline__ uint32_t key(uint32_t raw) { return raw; }
  static __device__ __forceinline__ bool forced(uint32_t raw) { return raw == 0u; }
};

// The largest key of each aligned group of 4 slots, added to sm.hist as its first digit
// (11 bits).  v holds the group's raw values, q its index, valid(slot) tells the span's slots.
// Called the same number of times by every lane of a warp.
template <class P, typename ValidFn>
__device__ __forceinline__ void add_group_max(ClusterSelectSmem& sm, const uint4& v, int q,
                                              bool in, ValidFn valid) {
  uint32_t m = 0u;
  bool have = false;
  const uint32_t r[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (in && valid(4 * q + c)) {
      m = max(m, P::key(r[c]));
      have = true;
    }
  }
  hist_add_runs(sm.hist, have ? m >> 21 : 0xFFFFFFFFu);
}

// cluster_topk_select over a span staged in shared memory: raw[slot] holds position
// slot - shift for slots [s0, s1), raw is 16-byte aligned and readable up to the next multiple
// of 4 slots.  Before any exact pass, a histogram of the first digit of each aligned group
// of 4 slots' largest key gives a bin g whose groups number at least K, so at least K keys
// have a first digit >= g and tau's first digit is >= g.  The candidate lists then hold the
// positions with first digit >= g (or forced), read 16 bytes at a time.  When every CTA's
// list fits and their union is short, each CTA copies the union's keys (in position order:
// rank, warp, entry) into its own shared memory and finds tau and the per-rank counts there,
// with block barriers only; otherwise the three exact passes go through rank 0's histogram
// as in cluster_topk_select, over the lists or, for a CTA whose list overflowed, its span.
// The result is the same as cluster_topk_select's.
//
// hist_ready: the caller has put the group-max histogram of this span into sm.hist, cleared
// rank 0's sm.ghist and synchronised the cluster after the clear.
template <int BLOCK, bool BITS, class P>
__device__ uint32_t cluster_topk_select_staged(const uint32_t* raw, int s0, int s1, int shift,
                                               int64_t K, int32_t* kept, int64_t base,
                                               int64_t cap, uint32_t* bits,
                                               ClusterSelectSmem& sm, bool hist_ready) {
  static_assert(BLOCK <= 1024 && (1024 % BLOCK) == 0, "block must divide 1024");
  constexpr int NW = BLOCK / 32;
  constexpr int LW = kListCap / NW;   // list entries per warp
  constexpr int U = 4;                // 16-byte groups per thread fetched before use
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank(), ncta = (int)cl.num_blocks();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t below = (1u << lane) - 1u;
  const uint4* raw4 = reinterpret_cast<const uint4*>(raw);
  const int nq = (s1 + 3) >> 2;        // groups holding the span (group 0 holds slot s0)
  auto valid = [&](int slot) { return (unsigned)(slot - s0) < (unsigned)(s1 - s0); };
  auto comp = [](const uint4& v, int c) { return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w; };
  if (threadIdx.x == 0) sm.lover = 0u;
  if (!hist_ready) {
    if (rank == 0)
      for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.ghist[i] = 0u;
    cl.sync();
  }

  // ---- lower bound g for tau's first digit, from the groups' largest keys
  const bool any = K > 0;   // the same in every CTA
  uint32_t g = 2048u;       // with K == 0 no key is a candidate: only forced positions
  if (any) {
    if (!hist_ready) {
      for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.hist[i] = 0u;
      __syncthreads();
      for (int qb = 0; qb < nq; qb += U * BLOCK) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int q = qb + u * BLOCK + (int)threadIdx.x;
          v[u] = q < nq ? raw4[q] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int q = qb + u * BLOCK + (int)threadIdx.x;
          add_group_max<P>(sm, v[u], q, q < nq, valid);
        }
      }
    }
    uint32_t b, kr;
    cluster_pick<BLOCK>(sm, 2048, (uint32_t)K, b, kr);
    g = b;
  }

  // ---- candidate lists: warp w lists, in order, the slots of its groups whose key has a
  // first digit >= g or that are forced
  const int per = (nq + NW - 1) / NW;
  const int q0 = min(nq, warp * per), q1 = min(nq, q0 + per);
  int32_t* L = sm.list + warp * LW;
  {
    uint32_t lc = 0;
    bool over = false;
    for (int qb = q0; qb < q1 && !over; qb += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int q = qb + 32 * u + lane;
        v[u] = q < q1 ? raw4[q] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int q = qb + 32 * u + lane;
        // the span's slots of this group: all four but in the first and the last group
        uint32_t vm = 0u;
        if (q < q1) {
          vm = 0xFu;
          if (q == 0 || q == nq - 1) {
            vm = 0u;
#pragma unroll
            for (int c = 0; c < 4; ++c) vm |= valid(4 * q + c) ? 1u << c : 0u;
          }
        }
        uint32_t cm = 0u;   // candidate components of this lane's group
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t r = comp(v[u], c);
          if (P::forced(r) || (P::key(r) >> 21) >= g) cm |= 1u << c;
        }
        cm &= vm;
        if (__ballot_sync(0xFFFFFFFFu, cm != 0u) == 0u) continue;   // the common case
        const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, cm & 1u);
        const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, cm & 2u);
        const uint32_t b2 = __ballot_sync(0xFFFFFFFFu, cm & 4u);
        const uint32_t b3 = __ballot_sync(0xFFFFFFFFu, cm & 8u);
        const uint32_t tot = __popc(b0) + __popc(b1) + __popc(b2) + __popc(b3);
        if (lc + tot > (uint32_t)LW) {
          over = true;   // the same in every lane
        } else if (!over) {
          uint32_t o = lc + __popc(b0 & below) + __popc(b1 & below) + __popc(b2 & below) +
                       __popc(b3 & below);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (cm & (1u << c)) L[o++] = 4 * q + c;
          lc += tot;
        }
      }
    }
    if (lane == 0) {
      sm.lcount[warp] = lc;
      if (over) sm.lover = 1u;
    }
  }
  if (threadIdx.x == 0) sm.gath = 1u;
  __syncthreads();
  // every CTA's lists and counts are complete (rank 0's histogram is clear again)
  cl.sync();
  {
    // thread r*NW + w reads the length of rank r's warp-w list; a scan gives the union's
    // layout (rank-major, in position order)
    const int ne = ncta * NW;   // <= BLOCK
    uint32_t c = 0;
    if ((int)threadIdx.x < ne) {
      const int r = (int)threadIdx.x / NW, w = (int)threadIdx.x - r * NW;
      const ClusterSelectSmem* R = cl.map_shared_rank(&sm, r);
      c = R->lcount[w];
      if (w == 0 && R->lover) sm.gath = 0u;
    }
    uint32_t tot;
    const uint32_t incl = block_incl_scan(c, sm.scr, &tot);   // ends with a barrier
    if ((int)threadIdx.x < ne) sm.ustart[threadIdx.x] = incl - c;
    if (threadIdx.x == 0) {
      sm.ustart[ne] = tot;
      sm.gtot = tot;
      if (tot > (uint32_t)kUnionCap) sm.gath = 0u;
    }
  }
  __syncthreads();
  const bool gather = sm.gath != 0u;   // the same in every CTA of the cluster
  const bool listed = sm.lover == 0u;   // the same in every thread of the CTA
  const int cw = listed ? (int)sm.lcount[warp] : 0;
  auto keyat = [&](int slot) { return P::key(raw[slot]); };

  // ---- exact digits (the first over keys with first digit >= g: tau's is among them)
  uint32_t prefix = 0, mask = 0, krem = any ? (uint32_t)K : 0u;
  if (gather) {
    // the union's raw values, rank-major, into this CTA's ghist words
    const int ut = (int)sm.gtot;
    uint32_t* Uk = sm.ghist;
    for (int t = threadIdx.x; t < ut; t += BLOCK) {
      int lo = 0, hi = ncta * NW;   // (rank, warp) with ustart[e] <= t < ustart[e + 1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm.ustart[mid] <= (uint32_t)t) lo = mid; else hi = mid;
      }
      const int r = lo / NW, w = lo - r * NW;
      const int32_t* Lr = cl.map_shared_rank(sm.list, r) + w * LW;
      const uint32_t* rawr = cl.map_shared_rank(raw, r);
      Uk[t] = rawr[Lr[t - (int)sm.ustart[lo]]];
    }
    if (any && ut <= BLOCK) {
      // one entry per thread: its rank among the union's keys (key desc, position asc; a
      // forced entry's key is 0, below every key that can be selected), tau the key ranked
      // K - 1 and keq = K - (keys above tau); every key above tau is in the union
      uint32_t* Kk = sm.hist;
      const int t = threadIdx.x;
      const uint32_t kt = t < ut ? P::key(Uk[t]) : 0u;
      if (t < ut) Kk[t] = kt;
      if (t == 0) sm.res[0] = 0u;
      __syncthreads();
      if (t < ut) {
        uint32_t rk = 0;
        for (int j = 0; j < ut; ++j) {
          const uint32_t kj = Kk[j];
          rk += (kj > kt || (kj == kt && j < t)) ? 1u : 0u;
        }
        if (rk == (uint32_t)K - 1u) sm.res[0] = kt;
      }
      __syncthreads();
      prefix = sm.res[0];
      uint32_t above = (t < ut && kt > prefix) ? 1u : 0u;
      above = warp_sum_u(above);
      if (t == 0) sm.res[1] = 0u;
      __syncthreads();
      if (lane == 0 && above) atomicAdd(&sm.res[1], above);
      __syncthreads();
      krem = (uint32_t)K - sm.res[1];
      __syncthreads();   // res is read by every thread before anyone writes it again
    } else if (any) {
#pragma unroll 1
      for (int pass = 0; pass < 3; ++pass) {
        const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int i = threadIdx.x; i < nb; i += BLOCK) sm.hist[i] = 0u;
        __syncthreads();   // (pass 0: also the union's keys are in place)
        for (int b0 = 0; b0 < ut; b0 += BLOCK) {
          const int t = b0 + (int)threadIdx.x;
          const uint32_t k = t < ut ? P::key(Uk[t]) : 0u;
          const bool in = t < ut && (pass == 0 ? (k >> 21) >= g : (k & mask) == prefix);
          hist_add_runs(sm.hist, in ? (k >> sh) & (uint32_t)(nb - 1) : 0xFFFFFFFFu);
        }
        __syncthreads();
        block_pick<BLOCK>(sm.hist, nb, krem, sm.scr, sm.res);
        __syncthreads();
        prefix |= sm.res[0] << sh;
        mask |= (uint32_t)(nb - 1) << sh;
        krem = sm.res[1];
        __syncthreads();   // res and scr are written again by the next pass
      }
    }
  } else if (any) {
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int nb = pass == 2 ? 1024 : 2048;
      for (int i = threadIdx.x; i < nb; i += BLOCK) sm.hist[i] = 0u;
      __syncthreads();
      auto add = [&](uint32_t k, bool ok) {
        const bool in = ok && (pass == 0 ? (k >> 21) >= g : (k & mask) == prefix);
        hist_add_runs(sm.hist, in ? (k >> sh) & (uint32_t)(nb - 1) : 0xFFFFFFFFu);
      };
      if (listed) {
        for (int b = 0; b < cw; b += 32 * 8) {
          uint32_t kk[8];
          bool ok[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int idx = b + 32 * u + lane;
            ok[u] = idx < cw;
            kk[u] = ok[u] ? keyat(L[idx]) : 0u;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) add(kk[u], ok[u]);
        }
      } else {
        for (int b0 = s0; b0 < s1; b0 += 8 * BLOCK) {
          uint32_t kk[8];
          bool ok[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = b0 + k * BLOCK + (int)threadIdx.x;
            ok[k] = i < s1;
            kk[k] = ok[k] ? keyat(i) : 0u;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) add(kk[k], ok[k]);
        }
      }
      uint32_t b, kr;
      cluster_pick<BLOCK>(sm, nb, krem, b, kr);
      prefix |= b << sh;
      mask |= (uint32_t)(nb - 1) << sh;
      krem = kr;
    }
  }
  const uint32_t tau = any ? prefix : 0xFFFFFFFFu;   // no key equals 0xFFFFFFFF
  const uint32_t keq = any ? krem : 0u;

  // ---- ordered selection: per-warp counts, cluster offsets, then each warp emits in order.
  // Unlisted CTAs walk their slots in warp slices of whole 32-position words.
  if (gather) {
    // every rank's (kept outright, tau-equal) counts from the union
    if (threadIdx.x < 2 * kMaxCluster) (&sm.cnt[0][0])[threadIdx.x] = 0u;
    __syncthreads();
    const int ut = (int)sm.gtot;
    for (int t = threadIdx.x; t < ut; t += BLOCK) {
      int r = 0;
      while (r + 1 < ncta && sm.ustart[(r + 1) * NW] <= (uint32_t)t) ++r;
      const uint32_t v = sm.ghist[t];
      const bool f = P::forced(v);
      const uint32_t k = P::key(v);
      if (f || k > tau) atomicAdd(&sm.cnt[r][0], 1u);
      else if (k == tau) atomicAdd(&sm.cnt[r][1], 1u);
    }
  }
  const int n = s1 - s0;
  const int wper = (((n + NW - 1) / NW) + 31) & ~31;
  const int w0 = min(s1, s0 + warp * wper), w1 = min(s1, w0 + wper);
  uint32_t nkeep = 0, neq = 0;
  auto tally = [&](int slot) {
    const uint32_t r = raw[slot];
    const bool f = P::forced(r);
    const uint32_t k = P::key(r);
    nkeep += (f || k > tau) ? 1u : 0u;
    neq += (!f && k == tau) ? 1u : 0u;
  };
  if (listed) {
    for (int idx = lane; idx < cw; idx += 32) tally(L[idx]);
  } else {
    for (int i = w0 + lane; i < w1; i += 32) tally(i);
  }
  nkeep = warp_sum_u(nkeep);
  neq = warp_sum_u(neq);
  if (lane == 0) {
    sm.scr[warp] = nkeep;
    sm.scr[32 + warp] = neq;
  }
  if (BITS && listed) {
    // the CTA's words start clear; kept bits are then set one by one
    const int p0 = s0 - shift, p1 = s1 - shift;
    for (int wd = p0 / 32 + (int)threadIdx.x; wd < (p1 + 31) / 32; wd += BLOCK) bits[wd] = 0u;
  }
  const uint32_t total = cluster_order_offsets<BLOCK>(sm, keq, gather);
  uint32_t eqc = sm.scr[64 + warp], outc = sm.scr[96 + warp];
  auto emit = [&](int slot, bool in) {
    const uint32_t r = in ? raw[slot] : 0u;
    const bool f = in && P::forced(r);
    const uint32_t k = P::key(r);
    const int j = slot - shift;
    const bool iseq = in && !f && k == tau;
    bool keep = in && (f || k > tau);
    const uint32_t meq = __ballot_sync(0xFFFFFFFFu, iseq);
    if (iseq && eqc + __popc(meq & below) < keq) keep = true;
    const uint32_t mk = __ballot_sync(0xFFFFFFFFu, keep);
    if (BITS) {
      if (listed) {
        if (keep) atomicOr(bits + (j >> 5), 1u << (j & 31));
      } else if (lane == 0) {
        bits[j >> 5] = mk;   // lane 0 holds the word's first position
      }
    } else if (keep) {
      const int64_t row = base + outc + __popc(mk & below);
      if (row < cap) kept[row] = j;
    }
    eqc += __popc(meq);
    outc += __popc(mk);
  };
  if (listed) {
    for (int b = 0; b < cw; b += 32) {
      const int idx = b + lane;
      emit(idx < cw ? L[idx] : 0, idx < cw);
    }
  } else {
    for (int ib = w0; ib < w1; ib += 32) emit(ib + lane, ib + lane < w1);
  }
  __syncthreads();   // lists and scr are reused by the next call
  // other CTAs read this one's lists and staged keys: none changes them before all are done
  if (gather) cl.sync();
  return total;
}

}  // namespace kv
