// Re-compaction of a flat cache: a smaller per-head Top-B_g chosen among the rows a head
// still holds, gathered into a second flat buffer.
//
// LAVa: after layer l is prefilled, the layers below it are compressed again with the same
// LAVa scores and budgets that shrink as more layers share the memory (online prefill and
// layer budget adjustment).  A layer compressed earlier no longer has its full K/V, only its
// flat cache; since top-B sets of one total order are nested, choosing the top B'_g among
// the rows a head holds gives what choosing among all its candidates would.  With the
// uncompacted K/V as the source (every position held), the same call compacts a freshly
// prefilled layer, at a row base that another call's offsets decide on the device.
//
// Three launches:
//   recompact_offsets (one CTA): new lengths (head_budget, at most the rows held) and the
//     offsets, from *row_base;
//   recompact_select (one CTA per head, a cluster of one): the rows whose position is a
//     candidate (0 <= pos < C) compete by (score desc, position asc); every other row (the
//     window, and rows with no position such as decode appends) is kept; the exact radix
//     select of radix_select.cuh lists the kept source rows, ascending, in the workspace at
//     the head's own source offset;
//   recompact_gather: positions and K/V rows of the listed source rows to the new buffer.
#include "kv_internal.cuh"
#include "radix_select.cuh"

namespace kv {

namespace {
constexpr int kOffThreads = 1024;
constexpr int kRSelThreads = 512;
constexpr int kRGatherThreads = 256;
}  // namespace

size_t recompact_ws_bytes(int64_t src_rows) {
  // the row lists, or, for the uncompacted source, the candidate regions of kv_compact's
  // selection (two 4-byte values per candidate)
  const size_t r = (size_t)(src_rows > 0 ? src_rows : 0);
  return kWsHeader + 2 * align_up(r * sizeof(int32_t), 256);
}

// Source extent of head h: its first source row and the rows it holds.
struct SrcHead {
  int64_t base, m;
};
__device__ __forceinline__ SrcHead src_head(int64_t h, int Hkv, int n,
                                            const int64_t* __restrict__ src_cu,
                                            const int32_t* __restrict__ src_lens,
                                            int64_t src_rows) {
  if (src_cu == nullptr) return {h * (int64_t)n, (int64_t)n};
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t b = src_cu[seg * (Hkv + 1) + g], e = src_cu[seg * (Hkv + 1) + g + 1];
  int64_t m = src_lens[h];
  const int64_t room = (e < src_rows ? e : src_rows) - b;
  if (b < 0 || room < 0) return {0, 0};
  if (m < 0) m = 0;
  if (m > room) m = room;
  return {b, m};
}

__global__ void __launch_bounds__(kOffThreads)
recompact_offsets(const int32_t* __restrict__ head_budget, const int64_t* __restrict__ src_cu,
                  const int32_t* __restrict__ src_lens, int64_t src_rows, int64_t H, int Hkv,
                  int n, int reserve, const int64_t* __restrict__ row_base, int64_t cap,
                  int64_t* __restrict__ cu, int32_t* __restrict__ lens, WsHeader* hdr) {
  __shared__ int64_t scratch[32];
  int64_t carry = row_base != nullptr ? *row_base : 0;
  for (int64_t h0 = 0; h0 < H; h0 += kOffThreads) {
    const int64_t h = h0 + threadIdx.x;
    int64_t ext = 0;
    int32_t len = 0;
    if (h < H) {
      const SrcHead sh = src_head(h, Hkv, n, src_cu, src_lens, src_rows);
      int64_t want = head_budget[h];
      if (want < 0 || want > sh.m) {
        raise_dev(hdr, DEV_HEAD_BUDGET, (unsigned)h);
        want = want < 0 ? 0 : sh.m;
      }
      len = (int32_t)want;
      ext = want + reserve;
    }
    int64_t total;
    const int64_t incl = block_incl_scan64(ext, scratch, &total);
    if (h < H) {
      const int64_t start = carry + incl - ext;
      const int64_t seg = h / Hkv;
      const int g = (int)(h - seg * Hkv);
      cu[seg * (Hkv + 1) + g] = start;
      if (g == Hkv - 1) cu[seg * (Hkv + 1) + Hkv] = start + ext;
      lens[h] = len;
      if (start + ext > cap) raise_dev(hdr, DEV_FLAT_CAPACITY, (unsigned)h);
    }
    carry += total;
  }
}

__global__ void __launch_bounds__(kRSelThreads)
recompact_select(const float* __restrict__ scores, const int32_t* __restrict__ src_kept,
                 const int64_t* __restrict__ src_cu, const int32_t* __restrict__ src_lens,
                 int64_t src_rows, int Hkv, int n, int C, const int32_t* __restrict__ lens,
                 int32_t* __restrict__ list, WsHeader* hdr) {
  __shared__ ClusterSelectSmem sm;
  __shared__ uint32_t red[kRSelThreads / 32];
  const int64_t h = blockIdx.x;
  const SrcHead sh = src_head(h, Hkv, n, src_cu, src_lens, src_rows);
  const int m = (int)sh.m;
  const float* sc = scores + h * (int64_t)C;
  auto pos = [&](int r) -> int64_t {
    return src_kept == nullptr ? (int64_t)r : (int64_t)src_kept[sh.base + r];
  };
  auto forced = [&](int r) {
    const int64_t p = pos(r);
    return !(p >= 0 && p < C);
  };
  auto key = [&](int r) -> uint32_t {
    const int64_t p = pos(r);
    return (p >= 0 && p < C) ? score_key(sc[p]) : 0u;
  };
  // rows that are kept whatever the scores
  uint32_t nf = 0;
  for (int r = threadIdx.x; r < m; r += kRSelThreads) nf += forced(r) ? 1u : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) nf += __shfl_xor_sync(0xFFFFFFFFu, nf, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = nf;
  __syncthreads();
  uint32_t F = 0;
  for (int i = 0; i < kRSelThreads / 32; ++i) F += red[i];
  const int64_t keep = lens[h];   // at most m (recompact_offsets)
  int64_t K = keep - (int64_t)F;
  if (K < 0) {
    if (threadIdx.x == 0) raise_dev(hdr, DEV_HEAD_BUDGET, (unsigned)h);
    K = 0;
  }
  // the kept source rows, ascending; rows past `keep` (too many forced ones) are skipped
  const uint32_t got = cluster_topk_select<kRSelThreads, false>(
      0, m, K, key, forced, list, sh.base, sh.base + keep, nullptr, sm);
  if (threadIdx.x == 0 && (int64_t)got != K + (int64_t)F) raise_dev(hdr, DEV_SELECT, (unsigned)h);
}

__global__ void __launch_bounds__(kRGatherThreads)
recompact_gather(const int32_t* __restrict__ src_kept, const int64_t* __restrict__ src_cu,
                 const int32_t* __restrict__ src_lens, int64_t src_rows, int Hkv, int n,
                 const char* __restrict__ sk, const char* __restrict__ sv, int row_bytes,
                 const int32_t* __restrict__ list, const int64_t* __restrict__ cu,
                 const int32_t* __restrict__ lens, int reserve, int64_t cap,
                 int32_t* __restrict__ kept, char* __restrict__ kf, char* __restrict__ vf) {
  const int64_t h = blockIdx.y;
  const SrcHead sh = src_head(h, Hkv, n, src_cu, src_lens, src_rows);
  const int64_t seg = h / Hkv;
  const int g = (int)(h - seg * Hkv);
  const int64_t base = cu[seg * (Hkv + 1) + g];
  const int64_t len = lens[h];
  const int vecs = row_bytes >> 4;
  const int64_t total = len * vecs;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx / vecs;
    const int c = (int)(idx - i * vecs);
    const int64_t row = base + i;
    if (row < 0 || row >= cap) continue;
    const int64_t r = list[sh.base + i];
    if (r < 0 || r >= sh.m) continue;   // never read outside the head's source rows
    const int64_t srow = sh.base + r;
    if (c == 0) kept[row] = src_kept == nullptr ? (int32_t)r : src_kept[srow];
    reinterpret_cast<uint4*>(kf + row * row_bytes)[c] =
        reinterpret_cast<const uint4*>(sk + srow * row_bytes)[c];
    reinterpret_cast<uint4*>(vf + row * row_bytes)[c] =
        reinterpret_cast<const uint4*>(sv + srow * row_bytes)[c];
  }
  if (blockIdx.x == 0)
    for (int t = threadIdx.x; t < reserve; t += blockDim.x) {
      const int64_t row = base + len + t;
      if (row >= 0 && row < cap) kept[row] = -1;
    }
}

cudaError_t launch_recompact(const Shape& s, const float* scores, const int32_t* head_budget,
                             const int32_t* src_kept, const int64_t* src_cu,
                             const int32_t* src_lens, const void* src_k, const void* src_v,
                             int64_t src_rows, int reserve, const int64_t* row_base,
                             int32_t* kept, int64_t* cu, int32_t* lens, void* kf, void* vf,
                             int64_t cap, char* ws, cudaStream_t st) {
  if (src_kept == nullptr) {
    // every position held: kv_compact's selection (streamed per-head Top-B_g over the
    // scores, the window kept) and gather, from the row base
    return launch_compact(s, src_k, src_v, scores, nullptr, 1, 2, 0.0f, false, head_budget,
                          reserve, kept, cu, lens, kf, vf, cap, ws, compact_plan(s, false), st,
                          row_base);
  }
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  int32_t* list = reinterpret_cast<int32_t*>(ws + kWsHeader);
  const int64_t H = s.units();
  recompact_offsets<<<1, kOffThreads, 0, st>>>(head_budget, src_cu, src_lens, src_rows, H, s.Hkv,
                                                s.n, reserve, row_base, cap, cu, lens, hdr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // a cluster of one CTA: the select's cluster barriers are the block's own
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)H);
  cfg.blockDim = dim3(kRSelThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, recompact_select, scores, src_kept, src_cu, src_lens, src_rows,
                         s.Hkv, s.n, s.C(), (const int32_t*)lens, list, hdr);
  if (e != cudaSuccess) return e;
  const int row_bytes = s.d * s.esize();
  int gx = (int)cdiv((int64_t)num_sms() * 16, H);
  if (gx < 1) gx = 1;
  if (gx > 64) gx = 64;
  recompact_gather<<<dim3(gx, (unsigned)H), kRGatherThreads, 0, st>>>(
      src_kept, src_cu, src_lens, src_rows, s.Hkv, s.n, (const char*)src_k, (const char*)src_v,
      row_bytes, list, cu, lens, reserve, cap, kept, (char*)kf, (char*)vf);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace kv
