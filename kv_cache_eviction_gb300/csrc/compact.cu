// Per-head selection and the flat cache gather.
//
// Ada-KV Algorithm 2: per-head Top-B_g eviction decision, selection of the kept
// K/V rows, concatenation of the observation window; the flat layout that puts
// every head of a layer into one tensor (cu_seqlens-style offsets), filled by a
// cache-update kernel.  CriticalKV: two-stage greedy selection, stage 1 by the
// attention score, stage 2 by (A + eps) * ||(V W^O)_j||_1.
#include "kv_internal.cuh"
#include "radix_select.cuh"

namespace kv {

namespace {
constexpr int kScanThreads = 1024;
constexpr int kSelThreads = 1024;
constexpr int kGatherThreads = 256;
}

// 64-bit inclusive block scan (one value per thread).
__device__ __forceinline__ int64_t block_incl_scan64(int64_t v, int64_t* scratch, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t s = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) scratch[lane] = s;
  }
  __syncthreads();
  const int64_t base = warp > 0 ? scratch[warp - 1] : 0;
  *total = scratch[nw - 1];
  __syncthreads();
  return base + x;
}

// Offsets of every head in the flat buffer and the initial lengths.
__global__ void __launch_bounds__(kScanThreads)
compact_offsets(const int32_t* __restrict__ head_budget, int64_t H, int Hkv, int w, int n,
                int reserve, int64_t cap, int64_t* __restrict__ cu, int32_t* __restrict__ lens,
                WsHeader* hdr) {
  __shared__ int64_t scratch[32];
  int64_t carry = 0;
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


// Ordered selection of positions j in [0, C): keep(j) = forced(j) || key(j) > tau ||
// (key(j) == tau && rank of j among the tau-equal keys < keq), i.e. the (key desc,
// position asc) order.  Kept positions go, ascending, to kept[base + r] (rows >= cap are
// skipped) or, with BITS, as one bit per position to bits[j / 32].  Two sweeps: per-warp
// counts over contiguous slices, one scan of the warp totals, then each warp emits its
// slice with ballots.  Returns the number of kept positions.  All threads must call it.
template <int BLOCK, bool BITS, typename KeyFn, typename ForcedFn>
__device__ uint32_t select_ordered(int C, KeyFn key, ForcedFn forced, uint32_t tau, uint32_t keq,
                                   int32_t* kept, int64_t base, int64_t cap, uint32_t* bits,
                                   uint32_t* scr /* 4 * 32 */) {
  constexpr int NW = BLOCK / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (((C + NW - 1) / NW) + 31) & ~31;   // slice length, a multiple of 32
  const int s0 = min(C, warp * per), s1 = min(C, s0 + per);
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
  if (lane == 0) { scr[warp] = nkeep; scr[32 + warp] = neq; }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t eq = 0, out = 0;
    for (int w = 0; w < NW; ++w) {
      const uint32_t e = scr[32 + w];
      const uint32_t take = eq >= keq ? 0u : (keq - eq < e ? keq - eq : e);
      scr[64 + w] = eq;    // tau-equal keys before this warp's slice
      scr[96 + w] = out;   // kept positions before this warp's slice
      out += scr[w] + take;
      eq += e;
    }
    scr[0] = out;          // total (the per-warp counts are no longer needed)
  }
  __syncthreads();
  uint32_t eqc = scr[64 + warp], outc = scr[96 + warp];
  const uint32_t total = scr[0];
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

// One CTA per head: threshold(s), ordered kept positions, window and reserve rows.
__global__ void __launch_bounds__(kSelThreads)
compact_select(const float* __restrict__ scores, const float* __restrict__ crit, uint32_t can,
               uint32_t cad, float ceps, const int32_t* __restrict__ lens,
               const int64_t* __restrict__ cu, int Hkv, int C, int w, int reserve,
               int32_t* __restrict__ kept, int64_t cap, uint32_t* __restrict__ flags,
               int64_t words, WsHeader* hdr) {
  __shared__ RadixSmem rs;
  const int64_t h = blockIdx.x;
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g];
  const int64_t Bg = (int64_t)lens[h] - w;   // lens was clamped to [w, n]
  const float* S = scores + h * (int64_t)C;
  __shared__ uint32_t scr[128];
  auto no = [](int) { return false; };
  if (crit == nullptr) {
    uint32_t tau, keq;
    auto key = [&](int64_t i) { return score_key(S[i]); };
    block_topk_threshold<kSelThreads>(C, Bg, key, rs, tau, keq);
    const uint32_t n = select_ordered<kSelThreads, false>(
        C, [&](int j) { return key(j); }, no, tau, keq, kept, base, cap, nullptr, scr);
    if (threadIdx.x == 0 && n != (uint32_t)Bg) raise_dev(hdr, DEV_SELECT, (unsigned)h);
  } else {
    const float* Cn = crit + h * (int64_t)C;
    uint32_t* F = flags + h * words;
    const int64_t K1 = ((int64_t)can * Bg) / cad;
    const int64_t K2 = Bg - K1;
    uint32_t tau1, keq1;
    auto key1 = [&](int64_t i) { return score_key(S[i]); };
    block_topk_threshold<kSelThreads>(C, K1, key1, rs, tau1, keq1);
    // stage-1 membership bits
    select_ordered<kSelThreads, true>(C, [&](int j) { return key1(j); }, no, tau1, keq1,
                                      nullptr, 0, 0, F, scr);
    auto in1 = [&](int64_t i) { return ((F[i >> 5] >> (i & 31)) & 1u) != 0u; };
    auto key2 = [&](int64_t i) -> uint32_t {
      if (in1(i)) return 0u;
      const float kap = __fmul_rn(__fadd_rn(S[i], ceps), Cn[i]);
      return score_key(kap) + 1u;
    };
    uint32_t tau2, keq2;
    block_topk_threshold<kSelThreads>(C, K2, key2, rs, tau2, keq2);
    const uint32_t n = select_ordered<kSelThreads, false>(
        C, [&](int j) { return key2(j); }, [&](int j) { return in1(j); }, tau2, keq2, kept,
        base, cap, nullptr, scr);
    if (threadIdx.x == 0 && n != (uint32_t)Bg) raise_dev(hdr, DEV_SELECT, (unsigned)h);
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

CompactPlan compact_plan(const Shape& s, bool critical) {
  CompactPlan p{};
  size_t off = kWsHeader;
  p.off_flags = off;
  p.flag_words = critical ? cdiv(s.C() > 0 ? s.C() : 1, 32) : 0;
  off += align_up((size_t)s.units() * p.flag_words * sizeof(uint32_t), 256);
  p.off_end = off;
  return p;
}

cudaError_t launch_compact(const Shape& s, const void* k, const void* v, const float* scores,
                           const float* crit, uint32_t can, uint32_t cad, float ceps,
                           const int32_t* head_budget, int reserve, int32_t* kept,
                           int64_t* cu, int32_t* lens, void* kf, void* vf, int64_t cap,
                           char* ws, const CompactPlan& p, cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int64_t H = s.units();
  compact_offsets<<<1, kScanThreads, 0, st>>>(head_budget, H, s.Hkv, s.w, s.n, reserve, cap, cu,
                                               lens, hdr);
  compact_select<<<(unsigned)H, kSelThreads, 0, st>>>(
      scores, crit, can, cad, ceps, lens, cu, s.Hkv, s.C(), s.w, reserve, kept, cap,
      reinterpret_cast<uint32_t*>(ws + p.off_flags), p.flag_words, hdr);
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

}  // namespace kv
