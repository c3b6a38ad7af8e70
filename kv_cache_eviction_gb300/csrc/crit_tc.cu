// CriticalKV output-projection norm on the 5th-generation tensor cores.
//
// CriticalKV ("Main experiments": the two-stage selection keeps the rest of the budget by
// (A_j + eps) * ||(V W_O)_j||_1): for every key j of a (sequence, layer, KV head) unit,
//   crit[j] = sum_{c < D} | sum_{e < d} V[j, e] * W_O[l, g][e, c] |,
// the L1 norm of the key's value row projected by that head's block of the output
// projection.  Per unit this is a (C x d) x (d x D) product, 2 * C * d * D flops, which is
// why it runs on tcgen05 while the rest of the pass is bandwidth-bound.
//
// Layout.  One work item = two 128-key tiles of V (256 keys, M = 2 x 128) against all
// D / 128 tiles of W_O (N = 128 each, K = d = 128).  V tiles are K-major (a key's d values
// are contiguous); W_O is stored [d][D] (c contiguous), so its tiles are the MN-major B
// operand as loaded: TMA boxes of 64 c x 128 e with 128-byte swizzling.  Both 128-row MMAs
// of an item read the same W_O tile, which comes from L2 (1 MiB per (layer, KV head),
// shared by every item of the B sequences).  Each N tile's two accumulators sit in TMEM
// (2 x 128 columns, double-buffered); the epilogue folds |x| of each row into one running
// sum per key, so the C x D product is never stored.
//
// Roles (384 threads): warp 0 = TMA producer, warp 1 = MMA issuer, warp 2 = TMEM
// allocator, warp 3 idle, warps 4..11 = epilogue (warp 4 + 4h + q: accumulator h, TMEM
// lanes 32q..32q+31).  Persistent: one CTA per SM takes items b, b + grid, ...  Every wait
// is bounded; on a timeout the CTA records DEV_WAIT_TIMEOUT, lets its copies and MMAs in
// flight finish (bounded) and frees its TMEM.
#include <cudaTypedefs.h>

#include <mutex>

#include "kv_internal.cuh"
#include "tc_ptx.cuh"

namespace kv {
namespace {

using namespace ptx;

constexpr int kCThreads = 384;
constexpr int kCEpiWarps = 8;
constexpr uint32_t kBox = 128 * 128;                // 128 rows x 128 bytes
constexpr uint32_t kTile = 2 * kBox;                // 128 x 128 bf16
constexpr int kBStages = 3;
constexpr uint32_t kOffA = 0;                       // 2 buffers x 2 tiles
constexpr uint32_t kOffB = 4 * kTile;               // kBStages tiles
constexpr uint32_t kOffTail = kOffB + kBStages * kTile;
constexpr uint32_t kTmemCols = 512;                 // 2 buffers x (2 x 128) fp32 columns

struct __align__(8) CTail {
  uint64_t afull[2], aempty[2];
  uint64_t bfull[kBStages], bempty[kBStages];
  uint64_t tfull[2], tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr uint32_t kCSmem = kOffTail + sizeof(CTail) + 1024;
static_assert(kCSmem <= 232448, "shared memory budget of one CTA");

// Shared-memory descriptor of an MN-major bf16 operand written by TMA with 128-byte
// swizzling: 64 elements along MN per 128-byte row, one row per K index, 8-row (1024-byte)
// swizzle atoms stacked along K (stride `sbo`), the next 64 MN elements `lbo` bytes on.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t dsc = 0;
  dsc |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  dsc |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  dsc |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  dsc |= (uint64_t)1 << 46;
  dsc |= (uint64_t)2 << 61;
  return dsc;
}

struct CritParams {
  int C, D, NT;          // candidates per unit, model dim, D / 128 tiles
  int LHkv;              // layers x KV heads
  int64_t units, pairs;  // units and 256-key items per unit
  float* crit;           // [units][C]
  WsHeader* hdr;
  // Per query head (mode != 0): W_O holds one [d][D] block per query head, Gq of them per
  // unit; the epilogue weighs query head q's norm by terms[unit][q][key] (+ eps) and sums,
  // times `scale`.  mode 1: L1 norms (GQA-exact CriticalKV), mode 2: L2 norms (LaProx).
  int mode, Gq;
  const float* terms;    // [units][Gq][C]
  float eps, scale;
};

__global__ void __launch_bounds__(kCThreads, 1)
crit_tc_kernel(const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap wmap,
               const CritParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  CTail* tl = reinterpret_cast<CTail*>(smem + kOffTail);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nitems = p.units * p.pairs;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tl->afull[b], 1);
      mbar_init(&tl->aempty[b], 1);
      mbar_init(&tl->tfull[b], 1);
      mbar_init(&tl->tempty[b], kCEpiWarps);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&tl->bfull[s], 1);
      mbar_init(&tl->bempty[s], 1);
    }
    mbar_init(&tl->drain, 1);
    tl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&wmap);
  }
  if (warp == 2) {
    tmem_alloc(&tl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort_flag = &tl->abort_flag;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      uint32_t li = 0, gb = 0;
      uint32_t afill[2] = {}, bfill[kBStages] = {};
      bool ok = true;
      for (int64_t it = blockIdx.x; it < nitems && ok; it += gridDim.x, ++li) {
        const int64_t u = it / p.pairs;
        const int key0 = (int)(it - u * p.pairs) * 256;
        const int lg = (int)(u % p.LHkv);
        const int ab = li & 1;
        if (!mbar_wait(&tl->aempty[ab], ((li >> 1) & 1) ^ 1) || *abort_flag) { ok = false; break; }
        ++afill[ab];
        mbar_arrive_expect_tx(&tl->afull[ab], 2 * kTile);
        unsigned char* A = smem + kOffA + ab * 2 * kTile;
        for (int h = 0; h < 2; ++h) {
          tma_load_3d(A + h * kTile, &vmap, &tl->afull[ab], 0, key0 + 128 * h, (int)u);
          tma_load_3d(A + h * kTile + kBox, &vmap, &tl->afull[ab], 64, key0 + 128 * h, (int)u);
        }
        for (int nt = 0; nt < p.NT * p.Gq; ++nt, ++gb) {
          const int s = gb % kBStages;
          if (!mbar_wait(&tl->bempty[s], ((gb / kBStages) & 1) ^ 1) || *abort_flag) {
            ok = false;
            break;
          }
          ++bfill[s];
          mbar_arrive_expect_tx(&tl->bfull[s], kTile);
          unsigned char* B = smem + kOffB + s * kTile;
          // tile nt: query head nt / NT of the unit's group, output columns (nt % NT) * 128
          const int blk = lg * p.Gq + nt / p.NT, col = (nt % p.NT) * 128;
          tma_load_3d(B, &wmap, &tl->bfull[s], col, 0, blk);
          tma_load_3d(B + kBox, &wmap, &tl->bfull[s], col + 64, 0, blk);
        }
      }
      if (!ok) {
        raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 0x200u + 1);
        *abort_flag = 1;
        // let the copies already issued land before the CTA exits
        for (int b = 0; b < 2; ++b)
          if (afill[b]) mbar_wait(&tl->afull[b], (afill[b] - 1) & 1, 20000000ull);
        for (int s = 0; s < kBStages; ++s)
          if (bfill[s]) mbar_wait(&tl->bfull[s], (bfill[s] - 1) & 1, 20000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      // kind::f16, bf16 x bf16 -> fp32, M = N = 128, A K-major, B MN-major
      const uint32_t idesc = idesc_bf16_f32(128, 128) | (1u << 16);
      uint32_t li = 0, gb = 0, gt = 0;
      bool ok = true;
      for (int64_t it = blockIdx.x; it < nitems && ok; it += gridDim.x, ++li) {
        const int ab = li & 1;
        if (!mbar_wait(&tl->afull[ab], (li >> 1) & 1) || *abort_flag) { ok = false; break; }
        const uint32_t aaddr = smem_u32(smem + kOffA + ab * 2 * kTile);
        for (int nt = 0; nt < p.NT * p.Gq; ++nt, ++gb, ++gt) {
          const int s = gb % kBStages, tb = gt & 1;
          if (!mbar_wait(&tl->bfull[s], (gb / kBStages) & 1) ||
              !mbar_wait(&tl->tempty[tb], ((gt >> 1) & 1) ^ 1) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t baddr = smem_u32(smem + kOffB + s * kTile);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // A: 16 K elements = 32 bytes along the swizzled 128-byte rows of box kk / 4;
            // B: 16 K rows = two 1024-byte swizzle atoms
            const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;
            const uint64_t bd = sdesc_sw128_mn(baddr + kk * 2048, kBox, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              mma_bf16(tmem + tb * 256 + h * 128, sdesc_sw128(aaddr + h * kTile + aoff), bd,
                       idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&tl->bempty[s]);
          mma_commit(&tl->tfull[tb]);
        }
        if (!ok) break;
        mma_commit(&tl->aempty[ab]);
      }
      if (!ok) {
        raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 0x200u + 2);
        *abort_flag = 1;
      }
      // every MMA issued has completed before TMEM is freed
      mma_commit(&tl->drain);
      mbar_wait(&tl->drain, 0, 20000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------ epilogue ----------------------------------
    const int ew = warp - 4, q = ew & 3, h = ew >> 2;
    uint32_t gt = 0;
    bool ok = true;
    for (int64_t it = blockIdx.x; it < nitems && ok; it += gridDim.x) {
      const int64_t u = it / p.pairs;
      const int key = (int)(it - u * p.pairs) * 256 + 128 * h + 32 * q + lane;
      float acc0 = 0.f, acc1 = 0.f, comb = 0.f;
      for (int nt = 0; nt < p.NT * p.Gq; ++nt, ++gt) {
        const int tb = gt & 1;
        const bool landed = mbar_wait(&tl->tfull[tb], (gt >> 1) & 1) && !*abort_flag;
        if (__any_sync(0xffffffffu, !landed)) { ok = false; break; }   // the whole warp
        tc_fence_after();
        const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + tb * 256 + h * 128;
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {
          uint32_t r[32];
          tmem_ld32(base + cq * 32, r);
          tmem_ld_wait(r);
          if (p.mode == 2) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float x0 = __uint_as_float(r[c]), x1 = __uint_as_float(r[c + 1]);
              acc0 = fmaf(x0, x0, acc0);
              acc1 = fmaf(x1, x1, acc1);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              acc0 += fabsf(__uint_as_float(r[c]));
              acc1 += fabsf(__uint_as_float(r[c + 1]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->tempty[tb]);
        if (p.mode != 0 && nt % p.NT == p.NT - 1) {
          // query head nt / NT is complete: its weighted norm joins the key's sum
          const int qh = nt / p.NT;
          const float nrm = p.mode == 2 ? sqrtf(acc0 + acc1) : acc0 + acc1;
          const float wt = key < p.C ? p.terms[(u * p.Gq + qh) * p.C + key] + p.eps : 0.f;
          comb = fmaf(wt, nrm, comb);
          acc0 = acc1 = 0.f;
        }
      }
      if (!ok) break;
      if (key < p.C) p.crit[u * p.C + key] = p.mode == 0 ? acc0 + acc1 : comb * p.scale;
    }
    if (!ok) {
      raise_dev(p.hdr, DEV_WAIT_TIMEOUT, 0x200u + 3);
      *abort_flag = 1;
    }
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 crit_encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D bf16 map [z][y][x] with 128-byte swizzled boxes of 64 x-elements by 128 y-rows.
bool make_map_3d(CUtensorMap* map, const void* base, uint64_t x, uint64_t y, uint64_t z) {
  auto fn = crit_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {x, y, z};
  const cuuint64_t strides[2] = {x * 2, x * y * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool crit_tc_supported(const Shape& s, int D) {
  return s.dtype == KV_BF16 && s.d == 128 && D >= 8 && D % 8 == 0 && s.C() >= 1 &&
         s.n <= (1 << 30);
}

cudaError_t launch_crit_tc(const Shape& s, const void* v, const void* w_o, int D, float* crit,
                           char* ws, cudaStream_t st) {
  return launch_proj_tc(s, 0, v, w_o, D, nullptr, 0.f, crit, ws, st);
}

cudaError_t launch_proj_tc(const Shape& s, int mode, const void* v, const void* w_o, int D,
                           const float* terms, float eps, float* crit, char* ws,
                           cudaStream_t st) {
  const int64_t units = s.units();
  const int Gq = mode == 0 ? 1 : s.G();
  CUtensorMap vm, wm;
  if (!make_map_3d(&vm, v, 128, (uint64_t)s.n, (uint64_t)units) ||
      !make_map_3d(&wm, w_o, (uint64_t)D, 128, (uint64_t)s.L * s.Hkv * Gq))
    return cudaErrorInvalidValue;
  CritParams prm{};
  prm.mode = mode;
  prm.Gq = Gq;
  prm.terms = terms;
  prm.eps = eps;
  // GQA-exact CriticalKV: the group mean; LaProx: the sum over the group
  prm.scale = mode == 1 ? 1.0f / (float)Gq : 1.0f;
  prm.C = s.C();
  prm.D = D;
  prm.NT = (int)cdiv(D, 128);
  prm.LHkv = s.L * s.Hkv;
  prm.units = units;
  prm.pairs = cdiv(s.C(), 256);
  prm.crit = crit;
  prm.hdr = reinterpret_cast<WsHeader*>(ws);
  cudaError_t e =
      cudaFuncSetAttribute(crit_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms();
  if (grid > units * prm.pairs) grid = units * prm.pairs;
  crit_tc_kernel<<<(unsigned)grid, kCThreads, kCSmem, st>>>(vm, wm, prm);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace kv
