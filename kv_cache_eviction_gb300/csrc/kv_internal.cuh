// Internal launch interface between the C ABI (kvevict_api.cu) and the kernels.
#pragma once

#include <atomic>

#include "kv_common.cuh"

namespace kv {

// ------------------------- per-device launch state ---------------------------
// Launch settings (shared-memory opt-ins, resident CTAs per SM, SM counts) belong to a
// device, so they are cached per device: a process may drive several GPUs.
constexpr int kMaxDevices = 64;
// The device current on the calling thread, or -1 if it cannot be read.
int current_device();
// `make()` evaluated once per device (with that device current) and cached; a device id
// outside [0, kMaxDevices) is not cached.  Two threads may both evaluate `make()` the
// first time, which is harmless for the idempotent settings kept here.
template <typename F>
inline int per_device(std::atomic<int> (&slot)[kMaxDevices], F make) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return make();
  int v = slot[dev].load(std::memory_order_acquire);
  if (v == 0) {
    v = make();   // 0 means "not known yet": a failed query is retried on the next call
    slot[dev].store(v, std::memory_order_release);
  }
  return v;
}

struct Shape {
  int B, L, Hq, Hkv, d, n, w, pool, dtype;
  __host__ __device__ int G() const { return Hq / Hkv; }
  __host__ __device__ int C() const { return n - w; }
  __host__ __device__ int R() const { return (Hq / Hkv) * w; }      // window rows per KV head
  __host__ __device__ int64_t units() const { return (int64_t)B * L * Hkv; }
  __host__ __device__ int64_t segments() const { return (int64_t)B * L; }
  int esize() const { return dtype == KV_BF16 ? 2 : 4; }
};

// ----------------------------- scoring -------------------------------------
struct ScorePlan {
  int path;             // 0 = CUDA-core (SIMT), 1 = tcgen05
  int chunk1, nchunk1;  // pass-1 keys per CTA and CTAs per unit
  int chunk2, nchunk2;  // pass-2 candidates per CTA and CTAs per unit
  size_t off_part, off_lse, off_vbar, off_end;
};
ScorePlan score_plan(const Shape& s, int mode);
cudaError_t launch_score(const Shape& s, int mode, int group, const void* q_win, const void* k,
                         const void* v, const void* w_o, int D, float* scores, float* crit,
                         char* ws, const ScorePlan& p, cudaStream_t st);

// CriticalKV's ||(V W_O)_j||_1 alone (tcgen05 kernel where the shape allows); `ws` is a
// scoring workspace (only its error word is used).
cudaError_t launch_crit_norm(const Shape& s, const void* v, const void* w_o, int D, float* crit,
                             char* ws, cudaStream_t st);

// Every query head's window term (kind KV_TERMS_MEAN_POOLED or KV_TERMS_L2) into
// terms [units][G][C]; `p` is the scoring plan of the shape (its LSE scratch is used).
cudaError_t launch_window_terms(const Shape& s, int kind, const void* q_win, const void* k,
                                float* terms, char* ws, const ScorePlan& p, cudaStream_t st);
// The norm kernel with one W_O block per query head ([L][Hq][d][D]), each query head's norm
// weighted by its window term (+ eps): mode 1 L1 norms, group mean (KV_PROJ_CRIT_GQA);
// mode 2 L2 norms, group sum (KV_PROJ_LAPROX).  bf16, d = 128 (crit_tc_supported).
bool crit_tc_supported(const Shape& s, int D);
cudaError_t launch_proj_tc(const Shape& s, int mode, const void* v, const void* w_o, int D,
                           const float* terms, float eps, float* out, char* ws,
                           cudaStream_t st);

// After the tcgen05 scoring kernel: LAVa's V-bar factor (vbar != nullptr) and the keys whose
// pooling window crosses a range boundary (from the halo copies of both ranges).
cudaError_t launch_score_fixup(const float* halo, const float* vbar, int64_t units, int Pg,
                               int Tu, int C, int G, int r, int group_max, int terms,
                               float* scores, cudaStream_t st);

// ----------------------------- allocation ----------------------------------
struct AllocPlan {
  int nchunkE;            // sweep CTAs per segment
  int64_t union_per_cta;  // candidate keys one sweep CTA can list
  size_t off_bprime, off_epart, off_gbin, off_zero, off_union, off_end;
};
AllocPlan alloc_plan(const Shape& s);
// layer_cap (nullable, entropy mode only): [B][L] the most rows each layer may keep.
cudaError_t launch_allocate(const Shape& s, const float* scores, const int64_t* budget,
                            int entropy_mode, const int32_t* layer_cap, uint32_t an, uint32_t ad,
                            int32_t* layer_budget, int32_t* head_budget, char* ws,
                            const AllocPlan& p, cudaStream_t st);

// layer_budget[seg] = sum over the segment's Hkv heads of head_budget.
cudaError_t launch_layer_sums(const int32_t* head_budget, int64_t segments, int Hkv,
                              int32_t* layer_budget, cudaStream_t st);

// ----------------------------- compaction ----------------------------------
struct CompactPlan {
  size_t off_flags, off_union, off_end;
  int64_t flag_words;   // per head, when CriticalKV stage-1 flags are needed
};
CompactPlan compact_plan(const Shape& s, bool critical);
// kappa_given: crit holds the stage-2 key itself instead of ||(V W_O)_j||_1.  row_base
// (nullable device pointer): the first output row (0 when null).
cudaError_t launch_compact(const Shape& s, const void* k, const void* v, const float* scores,
                           const float* crit, uint32_t can, uint32_t cad, float ceps,
                           bool kappa_given, const int32_t* head_budget, int reserve,
                           int32_t* kept, int64_t* cu, int32_t* lens, void* kf, void* vf,
                           int64_t cap, char* ws, const CompactPlan& p, cudaStream_t st,
                           const int64_t* row_base = nullptr);

// StreamingLLM preset: sinks and the most recent candidates fill each head's budget.
cudaError_t launch_compact_streaming(const Shape& s, const void* k, const void* v, int sinks,
                                     const int32_t* head_budget, int reserve, int32_t* kept,
                                     int64_t* cu, int32_t* lens, void* kf, void* vf, int64_t cap,
                                     char* ws, cudaStream_t st);

// ----------------------------- re-compaction --------------------------------
// Workspace of kv_recompact: the header, then one int32 per source row (the rows each head
// keeps, listed at the head's own source offsets).
size_t recompact_ws_bytes(int64_t src_rows);
// src_kept == nullptr: the source is the uncompacted [B][L][Hkv][n][d] K/V (head h's rows
// [h*n, (h+1)*n) hold positions 0..n-1); src_rows = its row count either way.
cudaError_t launch_recompact(const Shape& s, const float* scores, const int32_t* head_budget,
                             const int32_t* src_kept, const int64_t* src_cu,
                             const int32_t* src_lens, const void* src_k, const void* src_v,
                             int64_t src_rows, int reserve, const int64_t* row_base,
                             int32_t* kept, int64_t* cu, int32_t* lens, void* kf, void* vf,
                             int64_t cap, char* ws, cudaStream_t st);

// ----------------------------- decode --------------------------------------
struct DecodePlan {
  int64_t max_chunks;   // flat-row chunks (one CTA each) the launch may use
  int64_t part_slots;   // partials the part region holds
  size_t off_part, off_map, off_work, off_tick, off_end;
};
DecodePlan decode_plan(const Shape& s);
cudaError_t launch_decode(const Shape& s, const void* q, const void* kn, const void* vn,
                          void* kf, void* vf, const int64_t* cu, int32_t* lens, int64_t cap,
                          float scale, void* out, char* ws, const DecodePlan& p,
                          cudaStream_t st);

// Decode with one CTA per KV head (decode_head.cu): rows of 256 bytes, G <= 8, and at most
// this many flat rows per head on average (beyond it the row-balanced split of decode.cu
// evens out uneven heads better).
constexpr int64_t kDecodeHeadRowsMax = 1024;
bool decode_head_supported(const Shape& s, int64_t cap);
cudaError_t launch_decode_head(const Shape& s, const void* q, const void* kn, const void* vn,
                               void* kf, void* vf, const int64_t* cu, int32_t* lens,
                               int64_t cap, float scale, void* out, WsHeader* hdr,
                               cudaStream_t st);

// Decode with the used rows of all heads split evenly across CTAs (decode_split.cu): rows of
// 256 bytes, G <= 4, at most kDecodeSplitHeadsMax heads and a flat capacity within int32.
constexpr int64_t kDecodeSplitHeadsMax = 1024;
// Flat rows per head up to which the default choice is one CTA per head (when the heads fit
// one wave), and up to which it is the split (when they do not).
constexpr int64_t kDecodeHeadShortRows = 256;
constexpr int64_t kDecodeSplitRowsMax = 1536;
constexpr int64_t kDecodeSplitFewRowsMax = 8192;   // when the heads fit one wave
bool decode_split_supported(const Shape& s, int64_t cap);
cudaError_t launch_decode_split(const Shape& s, const void* q, const void* kn, const void* vn,
                                void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                int64_t cap, float scale, void* out, float* part,
                                int64_t part_slots, uint32_t* tick, WsHeader* hdr,
                                cudaStream_t st);

// Decode with one CTA per head and the rows of the longest heads spread over the CTAs left,
// in parts of one ring fill (decode_parts.cu): rows of 256 bytes, G <= 4, at most
// kDecodePartsHeadsMax heads, a flat capacity within int32 and a partial slot per head and
// per extra part.
constexpr int64_t kDecodePartsHeadsMax = 512;
bool decode_parts_supported(const Shape& s, int64_t cap, int64_t part_slots);
cudaError_t launch_decode_parts(const Shape& s, const void* q, const void* kn, const void* vn,
                                void* kf, void* vf, const int64_t* cu, int32_t* lens,
                                int64_t cap, float scale, void* out, float* part,
                                int64_t part_slots, uint32_t* tick, WsHeader* hdr,
                                cudaStream_t st);

int num_sms();
// Largest dynamic + static shared memory one CTA may opt in to.
size_t max_smem_optin();
// Adds n to the library's running count of kernel launches (kv_kernel_launches()).
void count_launches(int n);

}  // namespace kv
