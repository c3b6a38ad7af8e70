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
#pragma once

#include <cooperative_groups.h>

#include "kv_common.cuh"

namespace kv {

namespace cg = cooperative_groups;

constexpr int kMaxCluster = 8;

struct ClusterSelectSmem {
  uint32_t hist[2048];              // this CTA's histogram of the current pass
  uint32_t ghist[2048];             // rank 0: the cluster's histogram
  uint32_t scr[128];                // block scans
  uint32_t res[2];                  // rank 0: (bin, rank of the K-th key within it)
  uint32_t cnt[kMaxCluster][2];     // rank 0: (keys kept outright, tau-equal keys) per rank
};

// Positions [p0, p1) are this CTA's.  Every CTA of the cluster must call it with the same
// K (0 <= K <= the number of positions of all CTAs); key_of(i) must return the same key on
// every call for the same i.
template <int BLOCK, typename KeyFn>
__device__ void cluster_topk_threshold(int p0, int p1, int64_t K, KeyFn key_of,
                                       ClusterSelectSmem& sm, uint32_t& tau_out,
                                       uint32_t& keq_out) {
  static_assert(BLOCK <= 1024 && (1024 % BLOCK) == 0, "block must divide 1024");
  if (K <= 0) {
    tau_out = 0xFFFFFFFFu;
    keq_out = 0;
    return;
  }
  cg::cluster_group cl = cg::this_cluster();
  const bool lead = cl.block_rank() == 0;
  uint32_t* lead_g = cl.map_shared_rank(sm.ghist, 0);
  const uint32_t* lead_res = cl.map_shared_rank(sm.res, 0);
  if (lead)
    for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.ghist[i] = 0u;
  cl.sync();
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)K;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = threadIdx.x; i < nb; i += BLOCK) sm.hist[i] = 0u;
    __syncthreads();
    // 8 keys per thread per step, all fetched before use (latency hiding); the step count
    // is the same for every thread so the warp votes of hist_add_runs stay convergent
    constexpr int U = 8;
    for (int b0 = p0; b0 < p1; b0 += U * BLOCK) {
      uint32_t key[U];
      bool valid[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int i = b0 + k * BLOCK + (int)threadIdx.x;
        valid[k] = i < p1;
        key[k] = valid[k] ? key_of(i) : 0u;
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const uint32_t bin = (valid[k] && (key[k] & mask) == prefix)
                                 ? (key[k] >> sh) & (uint32_t)(nb - 1) : 0xFFFFFFFFu;
        hist_add_runs(sm.hist, bin);
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nb; i += BLOCK) {
      const uint32_t c = sm.hist[i];
      if (c) atomicAdd(lead_g + i, c);
    }
    cl.sync();
    if (lead) {
      // counts from the top bin downwards: thread t owns reversed bins [t*per, (t+1)*per)
      const int per = nb / BLOCK;
      uint32_t local = 0;
      for (int q = 0; q < per; ++q) local += sm.ghist[nb - 1 - ((int)threadIdx.x * per + q)];
      uint32_t total;
      const uint32_t incl = block_incl_scan(local, sm.scr, &total);
      const uint32_t excl = incl - local;
      if (excl < krem && krem <= incl) {
        uint32_t acc = excl;
        for (int q = 0; q < per; ++q) {
          const int bin = nb - 1 - ((int)threadIdx.x * per + q);
          const uint32_t c = sm.ghist[bin];
          if (acc + c >= krem) {
            sm.res[0] = (uint32_t)bin;
            sm.res[1] = krem - acc;
            break;
          }
          acc += c;
        }
      }
      __syncthreads();
      for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.ghist[i] = 0u;   // next pass
    }
    cl.sync();
    // rank 0 writes res again only after the next pass's first cluster barrier, which every
    // CTA reaches after this read
    const uint32_t bin = lead_res[0], kr = lead_res[1];
    prefix |= bin << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    krem = kr;
  }
  tau_out = prefix;
  keq_out = krem;
}

// Ordered selection of the cluster's positions: keep(j) = forced(j) || key(j) > tau ||
// (key(j) == tau && rank of j among the tau-equal keys of all CTAs < keq).  Kept positions
// go, ascending over the whole cluster, to kept[base + r] (rows >= cap are skipped) or, with
// BITS, as one bit per position to bits[j / 32] (p0 must then be a multiple of 32).  Two
// sweeps over [p0, p1): counts per warp slice and per CTA (exchanged through rank 0), then
// each warp emits its slice with ballots.  Returns the cluster's number of kept positions.
template <int BLOCK, bool BITS, typename KeyFn, typename ForcedFn>
__device__ uint32_t cluster_select_ordered(int p0, int p1, KeyFn key, ForcedFn forced,
                                           uint32_t tau, uint32_t keq, int32_t* kept,
                                           int64_t base, int64_t cap, uint32_t* bits,
                                           ClusterSelectSmem& sm) {
  constexpr int NW = BLOCK / 32;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank(), ncta = (int)cl.num_blocks();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p1 > p0 ? p1 - p0 : 0;
  const int per = (((n + NW - 1) / NW) + 31) & ~31;   // slice length, a multiple of 32
  const int s0 = min(p1, p0 + warp * per), s1 = min(p1, s0 + per);
  constexpr int U = 8;   // 32-key steps fetched per batch (latency hiding)
  uint32_t nkeep = 0, neq = 0;
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
  nkeep = warp_sum_u(nkeep);
  neq = warp_sum_u(neq);
  if (lane == 0) {
    sm.scr[warp] = nkeep;
    sm.scr[32 + warp] = neq;
  }
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
    // warp slices of this CTA in order
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
      sm.scr[64 + w] = eqc;    // tau-equal keys before this warp's slice
      sm.scr[96 + w] = out;    // kept positions before this warp's slice
      out += sm.scr[w] + take;
      eqc += e;
    }
    sm.scr[0] = total;
  }
  __syncthreads();
  uint32_t eqc = sm.scr[64 + warp], outc = sm.scr[96 + warp];
  const uint32_t total = sm.scr[0];
  const uint32_t below = (1u << lane) - 1u;
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
      const int j = j0 + lane;
      const bool in = j < s1;
      const bool iseq = in && !ff[u] && kk[u] == tau;
      bool keep = in && (ff[u] || kk[u] > tau);
      const uint32_t meq = __ballot_sync(0xFFFFFFFFu, iseq);
      if (iseq && eqc + __popc(meq & below) < keq) keep = true;
      const uint32_t mk = __ballot_sync(0xFFFFFFFFu, keep);
      if (BITS) {
        if (lane == 0) bits[j0 >> 5] = mk;
      } else if (keep) {
        const int64_t row = base + outc + __popc(mk & below);
        if (row < cap) kept[row] = j;
      }
      eqc += __popc(meq);
      outc += __popc(mk);
    }
  }
  __syncthreads();   // scr is reused by the caller
  return total;
}

}  // namespace kv
