// Radix select of the K largest 32-bit keys, and the ordered selection that follows it, over
// the CTAs of one thread-block cluster; and block_pick, the bin search over one histogram
// that the allocation and the streaming per-head selection use too.
//
// The per-head Top-B_g of Ada-KV Algorithm 2 and both stages of the CriticalKV selection
// fall back to cluster_topk_select, keys read from global memory, when a head's candidate
// union does not fit in shared memory.  No sort: three histogram passes over the keys (11,
// 11 and 10 bits, most significant first) narrow down tau, the K-th largest key.  The result
// is (tau, keq): every key > tau is selected, plus the keq lowest-position keys equal to
// tau, which is the (key desc, position asc) total order.
//
// Each CTA of the cluster owns a contiguous slice of the positions.  It builds its own
// histogram in shared memory; the slices' histograms are summed into rank 0's shared memory
// with distributed-shared-memory atomics, rank 0 finds the bin that holds the K-th key,
// and every CTA reads the result back from rank 0.  A cluster of one CTA runs the same code.
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
  int32_t list[kListCap];           // warp w: list[w * kListCap / warps ...]
};

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
// position order of the warps, exchanges the CTAs' totals through rank 0 and leaves in
// sm.scr[64 + w] the tau-equal keys and in sm.scr[96 + w] the kept positions of the whole
// cluster that come before warp w's first position.  Returns the cluster's kept count.
template <int BLOCK>
__device__ uint32_t cluster_order_offsets(ClusterSelectSmem& sm, uint32_t keq) {
  constexpr int NW = BLOCK / 32;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank(), ncta = (int)cl.num_blocks();
  __syncthreads();
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
  if (threadIdx.x == 0) {
    const uint32_t* lc = cl.map_shared_rank(&sm.cnt[0][0], 0);
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

}  // namespace kv
