// C ABI of libkvevict: argument validation, workspace layout, dispatch.
// Every check here runs on the host before anything is enqueued.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "kv_internal.cuh"

namespace kv {

int current_device() {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

int num_sms() {
  static std::atomic<int> slot[kMaxDevices];
  return per_device(slot, []() {
    int v = 0;
    const int dev = current_device();
    if (dev >= 0 && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        v > 0)
      return v;
    return 148;
  });
}

size_t max_smem_optin() {
  static std::atomic<int> slot[kMaxDevices];
  return (size_t)per_device(slot, []() {
    int v = 0;
    const int dev = current_device();
    if (dev >= 0 &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
        v > 0)
      return v;
    return 48 * 1024;
  });
}

static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to every op.  Returns false on an invalid shape.
static bool shape_ok(const kv_shape* sh, Shape* out) {
  if (sh == nullptr) return false;
  Shape s{sh->batch, sh->layers, sh->hq, sh->hkv, sh->d, sh->n, sh->w, sh->pool, sh->dtype};
  if (s.B < 0 || s.L < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.d <= 0 || s.n < 0 || s.w < 0) return false;
  if (s.Hq % s.Hkv != 0) return false;
  if (s.d % 8 != 0) return false;
  if (s.w > s.n) return false;
  if (s.pool < 1 || s.pool % 2 == 0) return false;
  if (s.dtype != KV_BF16 && s.dtype != KV_F32) return false;
  *out = s;
  return true;
}

// Limits of the kernels as built (valid shapes outside them are KV_ERR_UNSUPPORTED).
static bool shape_supported(const Shape& s) {
  if (s.G() > 8) return false;
  if (s.d > 128) return false;
  if (s.R() > 256) return false;
  if (s.Hkv > 256) return false;
  if ((int64_t)s.Hkv * s.n >= (int64_t)1 << 31) return false;
  return true;
}

static kv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KV_OK : KV_ERR_CUDA; }

// The shape of a model-wide selection (kv_allocate layer_entropy_mode 2): the L layers of a
// sequence as one layer of L * Hkv heads.  Scores [B][L][Hkv][C] and head budgets
// [B][L][Hkv] already have that layout.  False when it exceeds the kernels' limits.
static bool model_wide_shape(const Shape& s, Shape* m) {
  *m = s;
  m->L = 1;
  m->Hq = s.Hq * s.L;
  m->Hkv = s.Hkv * s.L;
  return s.L > 0 && shape_supported(*m);
}

// Scratch of flat_decode_attn_noalloc: one fixed array per device, never allocated at run
// time.  Host code must not pass the symbol itself to a kernel (on the host it names a
// host-side stand-in); the device address comes from cudaGetSymbolAddress, looked up once
// per device with that device current.
static __device__ __align__(256) char g_decode_noalloc_scratch[KV_DECODE_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[256] = {};

static cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace kv

using namespace kv;

extern "C" {

size_t kv_workspace_size(int op, const kv_shape* shape) {
  Shape s;
  if (!shape_ok(shape, &s)) return 0;
  switch (op) {
    case KV_OP_SCORE: {
      const ScorePlan a = score_plan(s, KV_SCORE_LAVA);
      const ScorePlan b = score_plan(s, KV_SCORE_CRITICAL);
      return a.off_end > b.off_end ? a.off_end : b.off_end;
    }
    case KV_OP_ALLOCATE: {
      size_t need = alloc_plan(s).off_end;
      Shape m;
      if (model_wide_shape(s, &m)) {   // room for layer_entropy_mode 2 as well
        const size_t w2 = alloc_plan(m).off_end + align_up((size_t)s.B * sizeof(int32_t), 256);
        if (w2 > need) need = w2;
      }
      return need;
    }
    case KV_OP_COMPACT: return compact_plan(s, true).off_end;
    case KV_OP_DECODE: return decode_plan(s).off_end;
    default: return 0;
  }
}

kv_status kv_score(const kv_shape* shape, int mode, int group, const void* q_win, const void* k,
                   const void* v, const void* w_o, int32_t model_dim, float* scores,
                   float* crit_norm, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (mode < KV_SCORE_ADA || mode > KV_SCORE_CRITICAL) return KV_ERR_INVALID_ARG;
  if (group != KV_GROUP_MEAN && group != KV_GROUP_MAX) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  if (s.n == 0 || s.w == 0) return KV_ERR_INVALID_ARG;
  if (q_win == nullptr || k == nullptr || scores == nullptr) return KV_ERR_INVALID_ARG;
  if (!aligned16(q_win) || !aligned16(k) || !aligned16(scores)) return KV_ERR_INVALID_ARG;
  if (mode != KV_SCORE_ADA && (v == nullptr || !aligned16(v))) return KV_ERR_INVALID_ARG;
  if (mode == KV_SCORE_CRITICAL) {
    if (w_o == nullptr || crit_norm == nullptr || !aligned16(w_o) || !aligned16(crit_norm))
      return KV_ERR_INVALID_ARG;
    if (model_dim <= 0 || model_dim % 8 != 0) return KV_ERR_INVALID_ARG;
  }
  if (!shape_supported(s)) return KV_ERR_UNSUPPORTED;
  const ScorePlan p = score_plan(s, mode);
  if (ws_bytes < p.off_end) return KV_ERR_WORKSPACE;
  return cuda_status(launch_score(s, mode, group, q_win, k, v, w_o, model_dim, scores,
                                  crit_norm, static_cast<char*>(ws), p,
                                  static_cast<cudaStream_t>(stream)));
}

kv_status kv_crit_norm(const kv_shape* shape, const void* v, const void* w_o, int32_t model_dim,
                       float* crit_norm, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (s.units() == 0 || s.C() <= 0) return KV_OK;
  if (v == nullptr || w_o == nullptr || crit_norm == nullptr) return KV_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(w_o) || !aligned16(crit_norm)) return KV_ERR_INVALID_ARG;
  if (model_dim <= 0 || model_dim % 8 != 0) return KV_ERR_INVALID_ARG;
  if (!shape_supported(s)) return KV_ERR_UNSUPPORTED;
  if (ws_bytes < kWsHeader) return KV_ERR_WORKSPACE;
  return cuda_status(launch_crit_norm(s, v, w_o, model_dim, crit_norm, static_cast<char*>(ws),
                                      static_cast<cudaStream_t>(stream)));
}

kv_status kv_allocate(const kv_shape* shape, const float* scores, const int64_t* budget,
                      int layer_entropy_mode, uint32_t alpha_num, uint32_t alpha_den,
                      int32_t* layer_budget, int32_t* head_budget, void* ws, size_t ws_bytes,
                      void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (layer_entropy_mode < 0 || layer_entropy_mode > 2) return KV_ERR_INVALID_ARG;
  if (alpha_den == 0 || alpha_num > alpha_den || alpha_den > 65536u) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  if (scores == nullptr || budget == nullptr || layer_budget == nullptr || head_budget == nullptr)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(scores) || !aligned16(budget) || !aligned16(layer_budget) ||
      !aligned16(head_budget))
    return KV_ERR_INVALID_ARG;
  if (layer_entropy_mode == 2) {
    // one selection over every layer of a sequence, then each layer's sum of head budgets
    Shape m;
    if (!shape_supported(s) || !model_wide_shape(s, &m)) return KV_ERR_UNSUPPORTED;
    const AllocPlan pm = alloc_plan(m);
    if (ws_bytes < pm.off_end + align_up((size_t)s.B * sizeof(int32_t), 256))
      return KV_ERR_WORKSPACE;
    char* w = static_cast<char*>(ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_allocate(m, scores, budget, 0, nullptr, alpha_num, alpha_den,
                                    reinterpret_cast<int32_t*>(w + pm.off_end), head_budget, w,
                                    pm, st);
    if (e == cudaSuccess) e = launch_layer_sums(head_budget, s.segments(), s.Hkv, layer_budget, st);
    return cuda_status(e);
  }
  if (!shape_supported(s) || (layer_entropy_mode && s.L > 1024)) return KV_ERR_UNSUPPORTED;
  const AllocPlan p = alloc_plan(s);
  if (ws_bytes < p.off_end) return KV_ERR_WORKSPACE;
  return cuda_status(launch_allocate(s, scores, budget, layer_entropy_mode, nullptr, alpha_num,
                                     alpha_den, layer_budget, head_budget,
                                     static_cast<char*>(ws), p,
                                     static_cast<cudaStream_t>(stream)));
}

kv_status kv_allocate_capped(const kv_shape* shape, const float* scores, const int64_t* budget,
                             const int32_t* layer_cap, uint32_t alpha_num, uint32_t alpha_den,
                             int32_t* layer_budget, int32_t* head_budget, void* ws,
                             size_t ws_bytes, void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (alpha_den == 0 || alpha_num > alpha_den || alpha_den > 65536u) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  if (scores == nullptr || budget == nullptr || layer_cap == nullptr || layer_budget == nullptr ||
      head_budget == nullptr)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(scores) || !aligned16(budget) || !aligned16(layer_cap) ||
      !aligned16(layer_budget) || !aligned16(head_budget))
    return KV_ERR_INVALID_ARG;
  if (!shape_supported(s) || s.L > 1024) return KV_ERR_UNSUPPORTED;
  const AllocPlan p = alloc_plan(s);
  if (ws_bytes < p.off_end) return KV_ERR_WORKSPACE;
  return cuda_status(launch_allocate(s, scores, budget, 1, layer_cap, alpha_num, alpha_den,
                                     layer_budget, head_budget, static_cast<char*>(ws), p,
                                     static_cast<cudaStream_t>(stream)));
}

// Argument checks of a compaction (kv_compact, kv_compact_kappa): KV_OK or the error.
static kv_status kv_compact_check(const Shape& s, const void* k, const void* v,
                                  const float* scores, const float* crit_norm,
                                  uint32_t crit_alpha_num, uint32_t crit_alpha_den,
                                  float crit_eps, const int32_t* head_budget, int32_t reserve,
                                  int32_t* kept_idx, int64_t* cu_off, int32_t* lens,
                                  void* k_flat, void* v_flat, int64_t flat_capacity_rows,
                                  void* ws) {
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (reserve < 0 || flat_capacity_rows < 0) return KV_ERR_INVALID_ARG;
  if (k == nullptr || v == nullptr || scores == nullptr || head_budget == nullptr ||
      kept_idx == nullptr || cu_off == nullptr || lens == nullptr || k_flat == nullptr ||
      v_flat == nullptr)
    return KV_ERR_INVALID_ARG;
  const void* ptrs[] = {k, v, scores, head_budget, kept_idx, cu_off, lens, k_flat, v_flat};
  for (const void* q : ptrs)
    if (!aligned16(q)) return KV_ERR_INVALID_ARG;
  if (crit_norm != nullptr) {
    if (!aligned16(crit_norm)) return KV_ERR_INVALID_ARG;
    if (crit_alpha_den == 0 || crit_alpha_num > crit_alpha_den || crit_alpha_den > 65536u)
      return KV_ERR_INVALID_ARG;
    if (!(crit_eps >= 0.0f) || std::isinf(crit_eps)) return KV_ERR_INVALID_ARG;
  }
  // The smallest flat buffer any valid budgets can need: every head keeps its window.
  if (flat_capacity_rows < s.units() * (int64_t)(s.w + reserve)) return KV_ERR_CAPACITY;
  if (!shape_supported(s)) return KV_ERR_UNSUPPORTED;
  return KV_OK;
}

kv_status kv_compact(const kv_shape* shape, const void* k, const void* v, const float* scores,
                     const float* crit_norm, uint32_t crit_alpha_num, uint32_t crit_alpha_den,
                     float crit_eps, const int32_t* head_budget, int32_t reserve,
                     int32_t* kept_idx, int64_t* cu_off, int32_t* lens, void* k_flat,
                     void* v_flat, int64_t flat_capacity_rows, void* ws, size_t ws_bytes,
                     void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (reserve < 0 || flat_capacity_rows < 0) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  const kv_status st = kv_compact_check(s, k, v, scores, crit_norm, crit_alpha_num,
                                        crit_alpha_den, crit_eps, head_budget, reserve, kept_idx,
                                        cu_off, lens, k_flat, v_flat, flat_capacity_rows, ws);
  if (st != KV_OK) return st;
  const CompactPlan p = compact_plan(s, crit_norm != nullptr);
  if (ws_bytes < p.off_end) return KV_ERR_WORKSPACE;
  return cuda_status(launch_compact(s, k, v, scores, crit_norm, crit_alpha_num, crit_alpha_den,
                                    crit_eps, false, head_budget, reserve, kept_idx, cu_off,
                                    lens, k_flat, v_flat, flat_capacity_rows,
                                    static_cast<char*>(ws), p,
                                    static_cast<cudaStream_t>(stream)));
}

kv_status kv_compact_streaming(const kv_shape* shape, const void* k, const void* v,
                               int32_t sinks, const int32_t* head_budget, int32_t reserve,
                               int32_t* kept_idx, int64_t* cu_off, int32_t* lens, void* k_flat,
                               void* v_flat, int64_t flat_capacity_rows, void* ws,
                               size_t ws_bytes, void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (sinks < 0) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (reserve < 0 || flat_capacity_rows < 0) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  // the checks of kv_compact; the scores are not read (any aligned pointer will do)
  const kv_status st = kv_compact_check(s, k, v, reinterpret_cast<const float*>(head_budget),
                                        nullptr, 1, 2, 0.0f, head_budget, reserve, kept_idx,
                                        cu_off, lens, k_flat, v_flat, flat_capacity_rows, ws);
  if (st != KV_OK) return st;
  if (ws_bytes < kWsHeader) return KV_ERR_WORKSPACE;
  return cuda_status(launch_compact_streaming(s, k, v, sinks, head_budget, reserve, kept_idx,
                                              cu_off, lens, k_flat, v_flat, flat_capacity_rows,
                                              static_cast<char*>(ws),
                                              static_cast<cudaStream_t>(stream)));
}

kv_status kv_compact_kappa(const kv_shape* shape, const void* k, const void* v,
                           const float* scores, const float* kappa, uint32_t crit_alpha_num,
                           uint32_t crit_alpha_den, const int32_t* head_budget, int32_t reserve,
                           int32_t* kept_idx, int64_t* cu_off, int32_t* lens, void* k_flat,
                           void* v_flat, int64_t flat_capacity_rows, void* ws, size_t ws_bytes,
                           void* stream) {
  if (kappa == nullptr) return KV_ERR_INVALID_ARG;
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  // the argument checks of kv_compact, with kappa in the norm's place
  const kv_status st = kv_compact_check(s, k, v, scores, kappa, crit_alpha_num, crit_alpha_den,
                                        0.0f, head_budget, reserve, kept_idx, cu_off, lens,
                                        k_flat, v_flat, flat_capacity_rows, ws);
  if (st != KV_OK) return st;
  const CompactPlan p = compact_plan(s, true);
  if (ws_bytes < p.off_end) return KV_ERR_WORKSPACE;
  return cuda_status(launch_compact(s, k, v, scores, kappa, crit_alpha_num, crit_alpha_den, 0.0f,
                                    true, head_budget, reserve, kept_idx, cu_off, lens, k_flat,
                                    v_flat, flat_capacity_rows, static_cast<char*>(ws), p,
                                    static_cast<cudaStream_t>(stream)));
}

kv_status kv_window_terms(const kv_shape* shape, int kind, const void* q_win, const void* k,
                          float* terms, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (kind != KV_TERMS_MEAN_POOLED && kind != KV_TERMS_L2) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  if (s.n == 0 || s.w == 0) return KV_ERR_INVALID_ARG;
  if (q_win == nullptr || k == nullptr || terms == nullptr) return KV_ERR_INVALID_ARG;
  if (!aligned16(q_win) || !aligned16(k) || !aligned16(terms)) return KV_ERR_INVALID_ARG;
  if (!shape_supported(s)) return KV_ERR_UNSUPPORTED;
  const ScorePlan p = score_plan(s, KV_SCORE_ADA);
  if (ws_bytes < p.off_end) return KV_ERR_WORKSPACE;
  return cuda_status(launch_window_terms(s, kind, q_win, k, terms, static_cast<char*>(ws), p,
                                         static_cast<cudaStream_t>(stream)));
}

kv_status kv_proj_score(const kv_shape* shape, int kind, const void* v, const void* w_o,
                        int32_t model_dim, const float* terms, float eps, float* out, void* ws,
                        size_t ws_bytes, void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (kind != KV_PROJ_CRIT_GQA && kind != KV_PROJ_LAPROX) return KV_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || std::isinf(eps)) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (s.units() == 0 || s.C() <= 0) return KV_OK;
  if (v == nullptr || w_o == nullptr || terms == nullptr || out == nullptr)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(w_o) || !aligned16(terms) || !aligned16(out))
    return KV_ERR_INVALID_ARG;
  if (model_dim <= 0 || model_dim % 8 != 0) return KV_ERR_INVALID_ARG;
  if (!shape_supported(s) || !crit_tc_supported(s, model_dim)) return KV_ERR_UNSUPPORTED;
  if (ws_bytes < kWsHeader) return KV_ERR_WORKSPACE;
  return cuda_status(launch_proj_tc(s, kind == KV_PROJ_CRIT_GQA ? 1 : 2, v, w_o, model_dim,
                                    terms, kind == KV_PROJ_CRIT_GQA ? eps : 0.0f, out,
                                    static_cast<char*>(ws), static_cast<cudaStream_t>(stream)));
}

// Argument checks of a decode step; on KV_OK, `s` and `p` hold its shape and workspace plan.
static kv_status decode_check(const kv_shape* shape, const void* q, const void* k_new,
                              const void* v_new, const void* k_flat, const void* v_flat,
                              const int64_t* cu_off, const int32_t* lens,
                              int64_t flat_capacity_rows, float softmax_scale, const void* out,
                              Shape* s, DecodePlan* p) {
  if (!shape_ok(shape, s)) return KV_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return KV_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KV_ERR_INVALID_ARG;
  if (flat_capacity_rows < 0) return KV_ERR_INVALID_ARG;
  if (s->units() == 0) {
    *p = DecodePlan{};
    return KV_OK;
  }
  if (q == nullptr || k_flat == nullptr || v_flat == nullptr || cu_off == nullptr ||
      lens == nullptr || out == nullptr)
    return KV_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k_flat, v_flat, cu_off, lens, out};
  for (const void* x : ptrs)
    if (!aligned16(x)) return KV_ERR_INVALID_ARG;
  if (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))) return KV_ERR_INVALID_ARG;
  if (!shape_supported(*s) || s->G() * s->d > 1024) return KV_ERR_UNSUPPORTED;
  *p = decode_plan(*s);
  return KV_OK;
}

size_t kv_recompact_workspace_size(int64_t src_capacity_rows) {
  if (src_capacity_rows < 0) return 0;
  return recompact_ws_bytes(src_capacity_rows);
}

kv_status kv_recompact(const kv_shape* shape, const float* scores, const int32_t* head_budget,
                       const int32_t* src_kept, const int64_t* src_cu, const int32_t* src_lens,
                       const void* src_k, const void* src_v, int64_t src_capacity_rows,
                       int32_t reserve, const int64_t* row_base, int32_t* kept_idx,
                       int64_t* cu_off, int32_t* lens, void* k_flat, void* v_flat,
                       int64_t flat_capacity_rows, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  if (!shape_ok(shape, &s)) return KV_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  if (reserve < 0 || flat_capacity_rows < 0 || src_capacity_rows < 0) return KV_ERR_INVALID_ARG;
  if (s.units() == 0) return KV_OK;
  const bool full = src_kept == nullptr;   // the source is the uncompacted K/V
  if (full != (src_cu == nullptr) || full != (src_lens == nullptr)) return KV_ERR_INVALID_ARG;
  if (scores == nullptr || head_budget == nullptr || src_k == nullptr || src_v == nullptr ||
      kept_idx == nullptr || cu_off == nullptr || lens == nullptr || k_flat == nullptr ||
      v_flat == nullptr)
    return KV_ERR_INVALID_ARG;
  // the rows move as 16-byte vectors; every table is read and written element by element,
  // so slices of per-layer tables need only their element's alignment
  const void* rows[] = {src_k, src_v, k_flat, v_flat};
  for (const void* x : rows)
    if (!aligned16(x)) return KV_ERR_INVALID_ARG;
  auto al = [](const void* x, uintptr_t a) {
    return x == nullptr || (reinterpret_cast<uintptr_t>(x) & (a - 1)) == 0;
  };
  if (!al(scores, 4) || !al(head_budget, 4) || !al(src_kept, 4) || !al(src_cu, 8) ||
      !al(src_lens, 4) || !al(row_base, 8) || !al(kept_idx, 4) || !al(cu_off, 8) ||
      !al(lens, 4))
    return KV_ERR_INVALID_ARG;
  if (src_k == k_flat || src_v == v_flat) return KV_ERR_INVALID_ARG;
  if (!shape_supported(s)) return KV_ERR_UNSUPPORTED;
  const int64_t src_rows = full ? s.units() * (int64_t)s.n : src_capacity_rows;
  if (src_rows >= ((int64_t)1 << 31)) return KV_ERR_UNSUPPORTED;
  if (ws_bytes < recompact_ws_bytes(src_rows)) return KV_ERR_WORKSPACE;
  return cuda_status(launch_recompact(s, scores, head_budget, src_kept, src_cu, src_lens, src_k,
                                      src_v, src_rows, reserve, row_base, kept_idx, cu_off, lens,
                                      k_flat, v_flat, flat_capacity_rows,
                                      static_cast<char*>(ws),
                                      static_cast<cudaStream_t>(stream)));
}

kv_status flat_decode_attn(const kv_shape* shape, const void* q, const void* k_new,
                           const void* v_new, void* k_flat, void* v_flat, const int64_t* cu_off,
                           int32_t* lens, int64_t flat_capacity_rows, float softmax_scale,
                           void* out, void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  Shape s;
  DecodePlan p;
  const kv_status st = decode_check(shape, q, k_new, v_new, k_flat, v_flat, cu_off, lens,
                                    flat_capacity_rows, softmax_scale, out, &s, &p);
  if (st != KV_OK || s.units() == 0) return st;
  if (ws_bytes < p.off_end) return KV_ERR_WORKSPACE;
  return cuda_status(launch_decode(s, q, k_new, v_new, k_flat, v_flat, cu_off, lens,
                                   flat_capacity_rows, softmax_scale, out,
                                   static_cast<char*>(ws), p, static_cast<cudaStream_t>(stream)));
}

kv_status kv_check_device_status(void* ws, void* stream, uint32_t* info) {
  if (ws == nullptr || !aligned16(ws)) return KV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader h;
  if (cudaMemcpyAsync(&h, ws, 8, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KV_ERR_CUDA;
  if (h.err == 0) {
    if (info) *info = 0;
    return KV_OK;
  }
  if (info) *info = h.err;
  if (cudaMemsetAsync(ws, 0, 8, st) != cudaSuccess) return KV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KV_ERR_CUDA;
  return KV_ERR_DEVICE_CHECK;
}

kv_status flat_decode_attn_noalloc(const kv_shape* shape, const void* q, const void* k_new,
                                   const void* v_new, void* k_flat, void* v_flat,
                                   const int64_t* cu_off, int32_t* lens,
                                   int64_t flat_capacity_rows, float softmax_scale, void* out,
                                   void* stream) {
  Shape s;
  DecodePlan p;
  const kv_status st = decode_check(shape, q, k_new, v_new, k_flat, v_flat, cu_off, lens,
                                    flat_capacity_rows, softmax_scale, out, &s, &p);
  if (st != KV_OK || s.units() == 0) return st;
  // A decode whose plan needs more than the fixed array is refused before anything is
  // enqueued.
  if (p.off_end > (size_t)KV_DECODE_NOALLOC_SCRATCH_BYTES) return KV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return KV_ERR_CUDA;
  char* ws = static_cast<char*>(scratch);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // The array starts at zero when the library is loaded, but it is shared by every call and
  // no caller reads its error word back.  So each call clears, on its own stream, what the
  // decode kernels need at zero: the error word (a check that fired in an earlier call must
  // not linger) and the tickets and counter of the one-launch kernels (the split and the
  // heads in parts), which share one region.  Those return to zero at the end of every
  // complete launch; clearing them here also undoes a launch that was cut short or raced
  // with an overlapping call.  The partials, the chunk map and the work counter are written
  // before they are read in every launch.  A memset allocates nothing.
  if (cudaMemsetAsync(ws, 0, kWsHeader, cs) != cudaSuccess ||
      cudaMemsetAsync(ws + p.off_tick, 0, p.off_end - p.off_tick, cs) != cudaSuccess)
    return KV_ERR_CUDA;
  return cuda_status(launch_decode(s, q, k_new, v_new, k_flat, v_flat, cu_off, lens,
                                   flat_capacity_rows, softmax_scale, out, ws, p, cs));
}

uint64_t kv_kernel_launches(void) { return (uint64_t)g_launches.load(); }

const char* kv_status_string(kv_status status) {
  switch (status) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KV_ERR_WORKSPACE: return "workspace too small";
    case KV_ERR_CAPACITY: return "flat buffer capacity too small";
    case KV_ERR_CUDA: return "CUDA error";
    case KV_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

}  // extern "C"
