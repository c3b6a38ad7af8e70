/*
 * kvevict.h -- C ABI of the GB300 (sm_103a) head-adaptive KV-cache eviction pass
 * and the flat variable-length decode attention that runs over its result.
 *
 * Method (cited by page title and section):
 *   "Ada-KV: Optimizing KV Cache Eviction by Adaptive Budget Allocation for
 *    Efficient LLM Inference": Algorithm 1 (adaptive budget allocation),
 *    Algorithm 2 (integration with SnapKV-style observation-window scoring),
 *    the flat cache layout with a custom cache-update kernel and variable-length
 *    attention, and the GQA group-mean criterion.
 *   "LAVa: Layer-wise KV Cache Eviction with Dynamic Budget Allocation":
 *    Definition 1 (LAVa score), head-flattened layer-wise eviction,
 *    uncertainty (entropy) based layer budgets, GQA group max.
 *   "CriticalKV: Optimizing KV Cache Eviction from an Output Perturbation
 *    Perspective": two-stage greedy selection with (A + eps) * ||(V W^O)_j||_1,
 *    plugged into Ada-KV.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor arguments are DEVICE pointers, contiguous, head-major, and
 *   16-byte aligned.  `d` must be a multiple of 8.  Violations return
 *   KV_ERR_INVALID_ARG before anything is enqueued.
 * - The caller owns every buffer.  The library allocates nothing, frees
 *   nothing and never synchronises implicitly: all work is enqueued on
 *   `stream` (a cudaStream_t passed as void*; NULL is the legacy default
 *   stream).  Inputs are read-only.
 * - Calls run on the device current on the calling thread.  A process may drive
 *   several devices: launch settings are kept per device.
 * - `ws` is a caller-provided device workspace of at least
 *   kv_workspace_size(op, shape) bytes for the op it is passed to.  Its first
 *   256 bytes hold a device error word.  Zero the whole workspace once before
 *   its first use; the library keeps the error word sticky across calls until
 *   kv_check_device_status() reads and clears it.  Calls that share one
 *   workspace must be ordered on one stream.
 * - Notation: B = batch (sequences), L = layers, Hq / Hkv = query / KV heads
 *   (Hq a multiple of Hkv, G = Hq/Hkv, query head q uses KV head q / G),
 *   d = head dim, n = prefix length, w = observation window (the last w
 *   positions), C = n - w candidate positions, pool = max-pool width (odd).
 * - Ties in every Top-k are broken by total orders: layer-wide
 *   (score desc, head asc, position asc); per head (score desc, position asc).
 *   Scores must be finite and >= 0 (they are, by construction).
 */
#ifndef KVEVICT_H_
#define KVEVICT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KV_API __attribute__((visibility("default")))
#else
#define KV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment or parameter        */
  KV_ERR_UNSUPPORTED = 2,   /* valid but not built for this shape / dtype        */
  KV_ERR_WORKSPACE = 3,     /* ws too small                                      */
  KV_ERR_CAPACITY = 4,      /* flat buffer too small for what the shape implies  */
  KV_ERR_CUDA = 5,          /* a CUDA launch or runtime call failed              */
  KV_ERR_DEVICE_CHECK = 6   /* a device-side check fired (see kv_check_device_status) */
} kv_status;

typedef enum { KV_BF16 = 0, KV_F32 = 1 } kv_dtype;
typedef enum { KV_SCORE_ADA = 0, KV_SCORE_LAVA = 1, KV_SCORE_CRITICAL = 2 } kv_score_mode;
typedef enum { KV_GROUP_MEAN = 0, KV_GROUP_MAX = 1 } kv_group_reduce;
typedef enum { KV_OP_SCORE = 0, KV_OP_ALLOCATE = 1, KV_OP_COMPACT = 2, KV_OP_DECODE = 3 } kv_op;
typedef enum { KV_TERMS_MEAN_POOLED = 0, KV_TERMS_L2 = 1 } kv_terms_kind;
typedef enum { KV_PROJ_CRIT_GQA = 0, KV_PROJ_LAPROX = 1 } kv_proj_kind;

/* Shape of one eviction problem: B sequences x L layers of one model. */
typedef struct {
  int32_t batch, layers, hq, hkv, d, n, w, pool;
  int32_t dtype;            /* kv_dtype: element type of q_win, k, v, w_o, q, k_new, v_new, out */
} kv_shape;

/* Bytes of device workspace `op` needs for `shape` (0 for an invalid shape). */
KV_API size_t kv_workspace_size(int op, const kv_shape* shape);

/*
 * kv_score -- observation-window scores of every candidate position.
 *
 * Ada-KV Algorithm 2 (scoring steps), LAVa Definition 1, CriticalKV's
 * projected-value norm.  For every (b, l, KV head g):
 *   z[q,t,j] = q_win[q,t] . k[g,j] / sqrt(d), causal: window row t sees j <= n-w+t
 *   P[q,t,:] = softmax_j z[q,t,:]                         (over all visible keys)
 *   a[q,j]   = (1/w) sum_t P[q,t,j]                        j < C
 *   p[q,j]   = max over |j'-j| <= pool/2, 0 <= j' < C of a[q,j']
 *   s[g,j]   = mean (KV_GROUP_MEAN) or max (KV_GROUP_MAX) over the G query heads
 *   LAVA:      s[g,j] *= max_k ||v[g,k]||_1
 *   CRITICAL:  crit_norm[g,j] = || v[g,j] W_O[l,g] ||_1  (the sum runs over D = model_dim)
 *
 * q_win     [B][L][Hq][w][d]    dtype
 * k, v      [B][L][Hkv][n][d]   dtype   (v is read by LAVA and CRITICAL only; may be NULL otherwise)
 * w_o       [L][Hkv][d][D]      dtype   CRITICAL only, else NULL; model_dim = D (multiple of 8)
 * scores    [B][L][Hkv][C]      float32 out
 * crit_norm [B][L][Hkv][C]      float32 out, CRITICAL only, else NULL
 */
KV_API kv_status kv_score(const kv_shape* shape, int mode, int group,
                   const void* q_win, const void* k, const void* v,
                   const void* w_o, int32_t model_dim,
                   float* scores, float* crit_norm,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * kv_crit_norm -- CriticalKV's projected-value norm on its own
 * ("CriticalKV: Optimizing KV Cache Eviction from an Output Perturbation Perspective",
 * key designs: the perturbation bound weighs each entry by the L1 norm of its value row
 * projected through the output matrix).  The same values kv_score writes to crit_norm in
 * KV_SCORE_CRITICAL mode, for callers that score with another mode first or time the two
 * apart:  crit_norm[b][l][g][j] = || v[b][l][g][j] W_O[l][g] ||_1  for j < C.
 *
 * v         [B][L][Hkv][n][d]   dtype
 * w_o       [L][Hkv][d][D]      dtype, model_dim = D (multiple of 8)
 * crit_norm [B][L][Hkv][C]      float32 out
 * ws        a workspace of at least kv_workspace_size(KV_OP_SCORE, shape) bytes (only its
 *           error word is used; 256 bytes suffice)
 */
KV_API kv_status kv_crit_norm(const kv_shape* shape, const void* v, const void* w_o,
                              int32_t model_dim, float* crit_norm, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * kv_window_terms -- every query head's observation-window term, before any reduction over
 * its group: the per-query-head inputs of the scores below that need one W_O block per
 * query head.  For every (b, l, query head q) and candidate j < C, with P the causal window
 * attention of kv_score:
 *   KV_TERMS_MEAN_POOLED: max-pool (width pool) of (1/w) sum_t P[q,t,j]  -- the per-head
 *       score of Ada-KV Algorithm 2 (kv_score's KV_GROUP_MEAN is its group mean);
 *   KV_TERMS_L2: sqrt(sum_t P[q,t,j]^2), no pooling -- ||A[:, j]||_2 of LaProx Algorithm 1.
 * q_win [B][L][Hq][w][d], k [B][L][Hkv][n][d]; terms [B][L][Hq][C] float32 out.
 * ws: a kv_workspace_size(KV_OP_SCORE, shape) workspace.  CUDA-core kernels.
 */
KV_API kv_status kv_window_terms(const kv_shape* shape, int kind, const void* q_win,
                                 const void* k, float* terms, void* ws, size_t ws_bytes,
                                 void* stream);

/*
 * kv_proj_score -- a score per KV head and candidate from the value rows projected through
 * one W_O block per query head ([L][Hq][d][D]: query head q's rows of the output
 * projection), each query head weighted by its window term (kv_window_terms):
 *   KV_PROJ_CRIT_GQA: out[g][j] = (1/G) sum_{q in g} (terms[q][j] + eps) * ||v[g][j] W_O[q]||_1
 *       -- CriticalKV's stage-2 key (A_j + eps) * ||(V W^O)_j||_1 ("CriticalKV", two-stage
 *       greedy selection) with W^O split per query head and Ada-KV's group mean over GQA;
 *       terms of kind KV_TERMS_MEAN_POOLED.  Feed it to kv_compact_kappa.
 *   KV_PROJ_LAPROX: out[g][j] = sum_{q in g} terms[q][j] * ||v[g][j] W_O[q]||_2 (eps unused)
 *       -- LaProx's p[i] = ||A[:, i]||_2 * ||H[i, :]||_2, H = V W_O (Algorithm 1), summed over
 *       the group's query heads; terms of kind KV_TERMS_L2.  Select with kv_allocate
 *       (layer_entropy_mode 2, alpha 0) and kv_compact.
 * v [B][L][Hkv][n][d], w_o [L][Hq][d][D] (model_dim = D, a multiple of 8), terms
 * [B][L][Hq][C], out [B][L][Hkv][C] float32.  tcgen05 kernel: bf16, d = 128 only (others
 * KV_ERR_UNSUPPORTED).  ws: 256 bytes (the error word).
 */
KV_API kv_status kv_proj_score(const kv_shape* shape, int kind, const void* v, const void* w_o,
                               int32_t model_dim, const float* terms, float eps, float* out,
                               void* ws, size_t ws_bytes, void* stream);

/*
 * kv_allocate -- per-head budgets (Ada-KV Algorithm 1 + safeguard; LAVa layer budgets).
 *
 * layer_entropy_mode = 0: budget [B][L] int64 is the layer budget B including
 *   the w*Hkv window rows.  B' = B - w*Hkv must lie in [0, Hkv*C].
 * layer_entropy_mode = 2: budget [B] int64 is one total over the L layers of a
 *   sequence (all windows included), selected model-wide ("Reformulating KV cache
 *   eviction for long-context LLM inference" (LaProx), Algorithm 1: one TopK over every
 *   head of every layer): the top total - L*w*Hkv candidates of all L*Hkv heads at once
 *   by (score desc, layer asc, head asc, position asc), counted per head, then the blend
 *   with alpha over all L*Hkv heads (LaProx: alpha = 0).  layer_budget[b][l] is the sum
 *   of layer l's head budgets.  Needs L*Hkv <= 256 and L*Hkv*n < 2^31.
 * layer_entropy_mode = 1: budget [B] int64 is one total over the L layers of a
 *   sequence (including all windows).  Each layer's selectable share of
 *   R = total - L*w*Hkv is proportional to its score entropy
 *   e_l = -sum s^ ln s^ / (Hkv*n), s^ = s / sum s over the layer; layers capped
 *   at Hkv*C give their overflow to the others; floors plus one unit each to
 *   the largest fractional parts (ties to the lower layer); all-zero entropies
 *   split uniformly.
 * Then per layer: f_g = number of head-g entries among the layer-wide top B'
 *   scores, and the safeguard blend with alpha = alpha_num/alpha_den, the
 *   weight of the UNIFORM share (alpha = 1: uniform SnapKV budgets; the
 *   Ada-KV page's own alpha' maps to alpha = 1 - alpha'):
 *     X_g = a*B' + (b-a)*Hkv*f_g,  B_g = floor(X_g / (b*Hkv)),
 *     the B' - sum B_g leftover units go to the largest X_g mod (b*Hkv), ties to the lower head.
 *   sum_g B_g = B' exactly and B_g >= floor(alpha*B'/Hkv).
 *
 * scores       [B][L][Hkv][C] float32 (from kv_score)
 * budget       [B][L] or [B]  int64 (device)
 * layer_budget [B][L]         int32 out: B_l including the window rows
 * head_budget  [B][L][Hkv]    int32 out: B_g + w, the kept length of head g
 * An out-of-range budget sets the device error word and is clamped.
 */
KV_API kv_status kv_allocate(const kv_shape* shape, const float* scores, const int64_t* budget,
                      int layer_entropy_mode, uint32_t alpha_num, uint32_t alpha_den,
                      int32_t* layer_budget, int32_t* head_budget,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * kv_allocate_capped -- LAVa layer budgets with a ceiling per layer, for the online
 * layer-wise prefill ("LAVa: Layer-wise KV Cache Eviction with Dynamic Budget Allocation",
 * online prefill and layer budget adjustment: after layer l is prefilled, the layers below
 * it are compressed again with the same scores and budgets that shrink as more layers
 * share the memory).
 *
 * The entropy split of kv_allocate's layer_entropy_mode = 1 over the L layers of `shape`,
 * except that layer l keeps at most layer_cap[b][l] rows (window included): a layer whose
 * proportional share exceeds its cap is fixed at the cap and the rest re-split, floors plus
 * largest remainders as before.  When the layers cannot hold the selectable total together,
 * every layer keeps its cap (no device check).  Then the per-head counts and the blend with
 * alpha as in kv_allocate (LAVa: alpha = 0).
 *
 * Stage t of the cascade (layers 0..t-1 prefilled, B = 1): shape.layers = t, scores of
 * layers 0..t-1 (contiguous), budget [1] the sequence's total, layer_cap [t] the previous
 * stage's layer_budget for layers 0..t-2 and at least Hkv*n for layer t-1.  layer_cap and
 * layer_budget must not be the same array (the caps are read while budgets are written).
 *
 * scores       [B][L][Hkv][C] float32
 * budget       [B] int64 total per sequence (all windows included)
 * layer_cap    [B][L] int32
 * layer_budget [B][L] int32 out, head_budget [B][L][Hkv] int32 out (B_g + w)
 * ws           a kv_workspace_size(KV_OP_ALLOCATE, shape) workspace
 */
KV_API kv_status kv_allocate_capped(const kv_shape* shape, const float* scores,
                                    const int64_t* budget, const int32_t* layer_cap,
                                    uint32_t alpha_num, uint32_t alpha_den,
                                    int32_t* layer_budget, int32_t* head_budget,
                                    void* ws, size_t ws_bytes, void* stream);

/*
 * kv_compact -- per-head Top-B_g selection and the flat cache gather
 * (Ada-KV Algorithm 2, selection and concatenation of the window; the flat
 * layout that concatenates every head of a layer into one tensor;
 * CriticalKV two-stage selection when crit_norm != NULL).
 *
 * Head g of (b, l) keeps B_g = head_budget - w positions: the top B_g by
 * (score desc, position asc); with crit_norm: stage 1 keeps the top
 * floor(crit_alpha_num * B_g / crit_alpha_den) by score, stage 2 the top
 * remaining by kappa = (score + crit_eps) * crit_norm, formed in float32.
 * Kept positions are written in ascending order, followed by the window
 * positions C..n-1.
 *
 * Flat layout: one buffer holds every (b, l, g) back to back in that order.
 * Head (b,l,g) owns rows [cu_off[b][l][g], cu_off[b][l][g+1]), of size
 * head_budget + reserve; its first lens = head_budget rows are filled, the
 * reserve rows are left for decode appends.  cu_off[b][l][Hkv] ==
 * cu_off[b][l+1][0] and the last entry is the total row count, which fits in
 * flat_capacity_rows when that is sum over (b,l) of (B_l + Hkv*reserve).
 *
 * k, v        [B][L][Hkv][n][d] dtype
 * scores      [B][L][Hkv][C] float32; crit_norm same shape or NULL
 * head_budget [B][L][Hkv] int32 (from kv_allocate)
 * kept_idx    [flat_capacity_rows] int32 out: source position of each flat row, -1 for reserve rows
 * cu_off      [B][L][Hkv+1] int64 out
 * lens        [B][L][Hkv] int32 out
 * k_flat, v_flat [flat_capacity_rows][d] dtype out
 * Rows past flat_capacity_rows are never written; the device error word is set instead.
 */
KV_API kv_status kv_compact(const kv_shape* shape, const void* k, const void* v,
                     const float* scores, const float* crit_norm,
                     uint32_t crit_alpha_num, uint32_t crit_alpha_den, float crit_eps,
                     const int32_t* head_budget, int32_t reserve,
                     int32_t* kept_idx, int64_t* cu_off, int32_t* lens,
                     void* k_flat, void* v_flat, int64_t flat_capacity_rows,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * kv_compact_streaming -- the sliding-window baseline as a budget preset (Ada-KV arXiv page,
 * Parameters: StreamingLLM keeps 4 sink tokens and the most recent window's cache): head g
 * keeps its first min(sinks, B_g) positions and the most recent B_g - min(sinks, B_g)
 * candidates before the window, then the window C..n-1, in ascending order; no scores are
 * read.  B_g = head_budget - w, as from kv_allocate (alpha = 1 gives the uniform per-head
 * budgets of a fixed-window policy whatever the scores).  Layout, outputs and checks as
 * kv_compact (sinks >= 0; the default of the page is 4).  ws: 256 bytes (error word).
 */
KV_API kv_status kv_compact_streaming(const kv_shape* shape, const void* k, const void* v,
                                      int32_t sinks, const int32_t* head_budget, int32_t reserve,
                                      int32_t* kept_idx, int64_t* cu_off, int32_t* lens,
                                      void* k_flat, void* v_flat, int64_t flat_capacity_rows,
                                      void* ws, size_t ws_bytes, void* stream);

/*
 * kv_compact_kappa -- kv_compact's CriticalKV two-stage selection with the stage-2 key
 * given: stage 1 keeps the top floor(crit_alpha * B_g) by score, stage 2 the rest by
 * kappa[b][l][g][j] itself (desc, position asc), for keys computed elsewhere such as
 * kv_proj_score's KV_PROJ_CRIT_GQA.  Arguments, layout and checks as kv_compact, with kappa
 * in crit_norm's place and no eps.
 */
KV_API kv_status kv_compact_kappa(const kv_shape* shape, const void* k, const void* v,
                                  const float* scores, const float* kappa,
                                  uint32_t crit_alpha_num, uint32_t crit_alpha_den,
                                  const int32_t* head_budget, int32_t reserve,
                                  int32_t* kept_idx, int64_t* cu_off, int32_t* lens,
                                  void* k_flat, void* v_flat, int64_t flat_capacity_rows,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * kv_recompact -- a smaller per-head Top-B_g chosen among the rows a flat cache still holds,
 * gathered into another flat buffer (LAVa, online prefill and layer budget adjustment: the
 * layers already compressed are compressed again with the same scores; Ada-KV Algorithm 2's
 * per-head selection and window).
 *
 * Source: a flat cache as kv_compact / kv_recompact write it (src_kept, src_cu, src_lens,
 * src_k, src_v; head h holds src_lens[h] rows from src_cu), or, with src_kept, src_cu and
 * src_lens all NULL, the uncompacted K/V [B][L][Hkv][n][d] (head h holds all n positions).
 * For every head: a row whose position p (its src_kept entry) is a candidate, 0 <= p < C,
 * competes by (scores[b][l][g][p] desc, p asc); every other row -- the window positions
 * C..n-1, and rows with no position (-1, e.g. decode appends) -- is always kept.  The head
 * keeps head_budget[h] rows in all (at most the rows it holds, at least its forced rows),
 * in source order (ascending positions), and they are gathered with their positions.
 *
 * Since Top-B sets of one total order are nested, re-selecting a smaller budget among the
 * rows kept by an earlier selection on the same scores gives the same rows as selecting
 * among all candidates.  On a cache that decode steps have appended to (their rows carry
 * position -1), the same call is a re-eviction: the appended rows and the window stay, and
 * the prefill rows make room by their prefill scores (CriticalKV notes, limitations: how to
 * re-select as entries join the cache during decoding is left open there).
 *
 * Output layout as in kv_compact, starting at row *row_base (row_base a device pointer to
 * one int64, 16-byte alignment not required, 8 bytes required; NULL = row 0): head h owns
 * rows [cu_off[h], cu_off[h] + lens[h] + reserve).  Pointing row_base at the last cu_off
 * entry of an earlier call appends after that call's rows without a host round trip.
 *
 * scores     [B][L][Hkv][C] float32
 * head_budget[B][L][Hkv] int32 (kv_allocate / kv_allocate_capped's head_budget)
 * src_capacity_rows: rows of src_k / src_v (ignored for the uncompacted source)
 * kept_idx, cu_off [B][L][Hkv+1], lens, k_flat, v_flat: outputs; k_flat / v_flat must not be
 *   the source buffers (the source is read while the output is written)
 * ws         at least kv_recompact_workspace_size(src rows) bytes (src rows = B*L*Hkv*n for
 *            the uncompacted source), zeroed once before its first use
 * head_budget out of range sets DEV check 4 (clamped); rows past flat_capacity_rows set
 * check 2 and are not written.  Modes without a second stage only (no CriticalKV norm).
 * Alignment: src_k, src_v, k_flat, v_flat 16 bytes; the tables only their element's
 * (scores, head_budget, src_kept, src_lens, kept_idx, lens 4 bytes; src_cu, cu_off,
 * row_base 8 bytes), so that one layer's slice of a [B][L] table can be passed.
 */
KV_API size_t kv_recompact_workspace_size(int64_t src_capacity_rows);
KV_API kv_status kv_recompact(const kv_shape* shape, const float* scores,
                              const int32_t* head_budget, const int32_t* src_kept,
                              const int64_t* src_cu, const int32_t* src_lens,
                              const void* src_k, const void* src_v, int64_t src_capacity_rows,
                              int32_t reserve, const int64_t* row_base, int32_t* kept_idx,
                              int64_t* cu_off, int32_t* lens, void* k_flat, void* v_flat,
                              int64_t flat_capacity_rows, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * flat_decode_attn -- one decode step of attention over the flat cache
 * (Ada-KV formal model: append k, v, then A = softmax(q K^T * scale), o = A V;
 * variable-length attention over the uneven per-head lengths).
 *
 * If k_new/v_new are given, row cu_off[b][l][g] + lens[b][l][g] of k_flat /
 * v_flat is written first and lens grows by one (the new token attends to
 * itself); with no reserve row left the device error word is set and that
 * head attends without the append.  Then for every query head q of KV head g:
 *   out[b][l][q] = sum_{r < lens} softmax_r(q . k_flat[cu + r] * softmax_scale) v_flat[cu + r]
 * with float32 accumulation.  A head with lens == 0 writes zeros.
 *
 * q            [B][L][Hq][d] dtype
 * k_new, v_new [B][L][Hkv][d] dtype, or both NULL
 * k_flat, v_flat, cu_off, lens as written by kv_compact (lens is updated in place)
 * flat_capacity_rows: rows of k_flat / v_flat; rows at or past it are never read or written
 *   (an append that would land there sets the device error word instead)
 * out          [B][L][Hq][d] dtype
 * `shape.n` bounds the head length (lens <= n + reserve); `w` and `pool` are unused.
 * The workspace holds counters that each call uses and leaves at zero (the reason for
 * zeroing a workspace once before its first use).
 */
KV_API kv_status flat_decode_attn(const kv_shape* shape, const void* q,
                           const void* k_new, const void* v_new,
                           void* k_flat, void* v_flat, const int64_t* cu_off, int32_t* lens,
                           int64_t flat_capacity_rows, float softmax_scale, void* out,
                           void* ws, size_t ws_bytes, void* stream);

/*
 * flat_decode_attn_noalloc -- the same decode step as flat_decode_attn, for callers that
 * cannot allocate device memory.  (The method's pages have no counterpart: this is a
 * deployment convenience of this library.)
 *
 * Some callers own no allocator at the point where they run a decode step: a serving loop
 * whose device memory was planned once at start-up and may not grow, an engine plugin that
 * is handed only its input and output buffers when it is enqueued, or code that issues work
 * while a stream is being captured, where allocation calls are not allowed.  This entry
 * point takes no workspace.  Its split-K scratch is a fixed array of
 * KV_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the library; every GPU that loads
 * the library holds that array until the process exits.  Nothing here calls cudaMalloc,
 * cudaFree or any allocating routine.
 *
 * Arguments, results and validation are those of flat_decode_attn without `ws`/`ws_bytes`.
 * - A shape whose decode needs more scratch than the fixed array (kv_workspace_size
 *   (KV_OP_DECODE, shape) > KV_DECODE_NOALLOC_SCRATCH_BYTES) is rejected with
 *   KV_ERR_WORKSPACE before anything is enqueued.
 * - The first call on each device looks up that device's copy of the array (with the
 *   device current) and caches it; make that first call before any stream capture.
 * - Every call on a device shares the one array and leaves its last contents there.  Each
 *   call first clears, on its own stream (cudaMemsetAsync, which allocates nothing), the
 *   parts the decode kernels need at zero: the error word and the tickets and counter of the
 *   one-launch decode kernels (rows split across CTAs, or heads in parts).
 *   The rest (partials, chunk map, work counter) is written before it is read.
 *   Calls whose kernels overlap on the GPU (different streams without ordering between
 *   them) race on the array and can return wrong outputs: order them on one stream, or use
 *   flat_decode_attn with separate workspaces.  A later, correctly ordered call is not
 *   affected by such a race, since it clears the tickets again.
 * - Device-side checks (an append with no reserve row left) behave as in flat_decode_attn
 *   (the append is skipped and lens is not advanced) but are not reported: there is no
 *   workspace for kv_check_device_status to read.
 */
#define KV_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)
KV_API kv_status flat_decode_attn_noalloc(const kv_shape* shape, const void* q,
                                          const void* k_new, const void* v_new,
                                          void* k_flat, void* v_flat, const int64_t* cu_off,
                                          int32_t* lens, int64_t flat_capacity_rows,
                                          float softmax_scale, void* out, void* stream);

/* Synchronises `stream`, reads the device error word of `ws` and clears it.
 * Returns KV_OK or KV_ERR_DEVICE_CHECK (KV_ERR_CUDA if the copy fails).
 * `info` (nullable) receives the first recorded check code. */
KV_API kv_status kv_check_device_status(void* ws, void* stream, uint32_t* info);

/* Number of kernels the library has launched in this process so far (all calls, all
 * streams); the difference across a region counts that region's launches. */
KV_API uint64_t kv_kernel_launches(void);

/* Static description of a status code. */
KV_API const char* kv_status_string(kv_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVEVICT_H_ */
