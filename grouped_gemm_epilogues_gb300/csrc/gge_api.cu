// Host side of libgge.so: argument validation, launch planning, TMA tensor
// maps and the C ABI declared in include/gge.h.
//
// The checks follow the pages' rules (quack/dense_gemm_sm90.py,
// GemmSm90.is_valid_dtypes and the wrapper's major / alignment handling):
// 16-bit A and B of the same type, or two 8-bit types in K-major layout; the
// contiguous dimension 16-byte aligned.  Everything here runs before the
// launch; nothing allocates or synchronises.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gge.h"
#include "gge_launch.h"
#include "gge_params.h"
#include "gge_sched.cuh"

namespace gge {
namespace {

constexpr int kTileM = 128;
constexpr int kRowBytesHost = 128;
constexpr int kMaxSmemOptin = 232448;  // 227 KiB per block on sm_100 / sm_103
constexpr int kCtrlBytesHost = 1024;
constexpr int kEpiWarpsHost = 8;          // epilogue warps of the TMA variants (4 with gathers)
constexpr int kMaxGroupsHost = 1024;
constexpr int kIdxChunkHost = 2048;       // gather-K index entries staged in shared memory
constexpr size_t kWorkspaceBytes = 256;
// the split last wave's tickets (one int32 per tail tile, CTA, epilogue warp and chunk)
// follow the status words in a region of their own: no other call writes there,
// so a ticket is never mistaken for another call's data
constexpr size_t kTicketBytes = 16384;
constexpr size_t kMapSlotsHost = 16;     // varlen-K tensor-map slots per CTA (kernel kMapSlots)
constexpr size_t kMapSlotBytesHost = 256;
constexpr int kMaxStages = 8;            // fewer stages than map slots
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int64_t kMaxExtent = (int64_t(1) << 31) - 1;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    RelaxedCaptureMode relaxed;  // the first call may run inside a stream capture
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

int elem_bytes(int32_t dt) {
  switch (dt) {
    case GGE_BF16: case GGE_F16: return 2;
    case GGE_E4M3: case GGE_E5M2: return 1;
    case GGE_F32: return 4;
    default: return 0;
  }
}

bool is16(int32_t dt) { return dt == GGE_BF16 || dt == GGE_F16; }
bool is8(int32_t dt) { return dt == GGE_E4M3 || dt == GGE_E5M2; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gge_status check_view(const gge_tensor& t) {
  // an empty view (no elements) may carry a NULL pointer: it is never dereferenced
  const bool empty = (t.rows == 0 || t.cols == 0);
  if ((t.ptr == nullptr && !empty) || t.reserved != 0) return GGE_ERR_INVALID_ARG;
  if (elem_bytes(t.dtype) == 0) return GGE_ERR_INVALID_ARG;
  if (t.rows < 0 || t.cols < 0 || t.batch < 1) return GGE_ERR_INVALID_ARG;
  if (t.rows > kMaxExtent || t.cols > kMaxExtent || t.batch > kMaxExtent) return GGE_ERR_UNSUPPORTED;
  if (t.stride_row < 0 || t.stride_col < 0 || t.stride_batch < 0) return GGE_ERR_INVALID_ARG;
  if (!aligned16(t.ptr)) return GGE_ERR_ALIGNMENT;
  return GGE_OK;
}

// An output / C view: [M, N, L] N-major with 16-byte aligned rows and batches.
gge_status check_mn(const gge_tensor* t, int64_t M, int64_t N, int64_t L, bool is_output) {
  gge_status s = check_view(*t);
  if (s != GGE_OK) return s;
  if (t->dtype != GGE_BF16 && t->dtype != GGE_F16 && t->dtype != GGE_F32) return GGE_ERR_UNSUPPORTED;
  if (t->rows != M || t->cols != N || t->batch != L) return GGE_ERR_INVALID_ARG;
  if (N > 1 && t->stride_col != 1) return GGE_ERR_UNSUPPORTED;  // N-major only
  const int es = elem_bytes(t->dtype);
  if (M > 1 && t->stride_row < N) return GGE_ERR_INVALID_ARG;
  if ((t->stride_row * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
  if (L > 1 && (t->stride_batch * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
  (void)is_output;
  return GGE_OK;
}

enum class Form { Plain, Varlen, Gather, GatherVarlen, VarlenK, GatherK };

struct Plan {
  Params p;
  CUtensorMap tmA, tmB;
  int bn;
  int cg;  // CTAs per tile: 1, or 2 for a CTA pair (cta_group::2)
  bool gather;
  LaunchShape shape;
  int64_t M, N, K, L;
  bool empty;  // nothing to compute
  int band;
  // split last wave (plain problems): whole-tile count and units, so that a call
  // whose workspace is too small can run unsplit
  int64_t tiles = 0;
  int units = 0;
};

// Workspace layout: the status words; the split last wave's tickets; then either
// the split's partial accumulators (one 128 x BN fp32 block per tail tile, slice
// and CTA) or, for varlen-K and gather-K, the per-CTA tensor-map slots.  Each
// region starts 256-byte aligned.
constexpr size_t kTailBase = kWorkspaceBytes + kTicketBytes;
size_t tail_workspace(const Plan& pl) {
  if (pl.p.tail_tiles <= 0) return 0;
  const int64_t blocks = static_cast<int64_t>(pl.p.tail_tiles) * pl.p.tail_splits * pl.cg;
  return kTailBase + static_cast<size_t>(blocks) * kTileM * pl.bn * sizeof(float);
}
constexpr size_t kTicketsPerWarpHost = 4;  // one per epilogue warp and 32-column chunk
bool tickets_fit(const Plan& pl) {
  return static_cast<size_t>(pl.p.tail_tiles) * pl.cg * kEpiWarpsHost * kTicketsPerWarpHost * 4 <=
         kTicketBytes;
}

CUtensorMapDataType tmap_type(int es) {
  return es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
}

// Encoded tensor maps are cached (keyed by everything that goes into them), so
// repeated calls on the same buffers skip the driver call.
struct TmapKey {
  void* ptr;
  uint64_t d0, d1, d2, s1, s2;
  uint32_t b0, b1;
  int es;
  bool operator==(const TmapKey& o) const {
    return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && s1 == o.s1 && s2 == o.s2 &&
           b0 == o.b0 && b1 == o.b1 && es == o.es;
  }
};

struct TmapCache {
  static constexpr int kEntries = 64;
  std::mutex mu;
  TmapKey key[kEntries];
  CUtensorMap map[kEntries];
  uint64_t used[kEntries] = {};  // 0: empty; else last-use tick
  uint64_t tick = 0;
};

TmapCache& tmap_cache() {
  static TmapCache c;
  return c;
}

gge_status encode_3d(CUtensorMap* m, void* ptr, int es, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1) {
  const TmapKey k{ptr, d0, d1, d2, s1_bytes, s2_bytes, b0, b1, es};
  TmapCache& c = tmap_cache();
  {
    std::lock_guard<std::mutex> g(c.mu);
    for (int i = 0; i < TmapCache::kEntries; ++i) {
      if (c.used[i] != 0 && c.key[i] == k) {
        c.used[i] = ++c.tick;
        *m = c.map[i];
        return GGE_OK;
      }
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return GGE_ERR_CUDA;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, tmap_type(es), 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return GGE_ERR_CUDA;
  std::lock_guard<std::mutex> g(c.mu);
  int victim = 0;
  for (int i = 0; i < TmapCache::kEntries; ++i)
    if (c.used[i] < c.used[victim]) victim = i;  // an empty slot (0) or the least recent
  c.key[victim] = k;
  c.map[victim] = *m;
  c.used[victim] = ++c.tick;
  return GGE_OK;
}

uint64_t batch_stride_bytes(const gge_tensor& t, int es) {
  if (t.batch > 1) return static_cast<uint64_t>(t.stride_batch) * es;
  // a single batch: any legal stride (never stepped over)
  uint64_t s = static_cast<uint64_t>(std::max<int64_t>(t.rows, 1)) *
               static_cast<uint64_t>(std::max<int64_t>(t.stride_row, 1)) * es;
  return (s + 15) / 16 * 16;
}

// The same for an M- / N-major view, whose K columns are stride_col apart.
uint64_t mn_batch_stride_bytes(const gge_tensor& t, int es) {
  if (t.batch > 1) return static_cast<uint64_t>(t.stride_batch) * es;
  uint64_t s = static_cast<uint64_t>(std::max<int64_t>(t.cols, 1)) *
               static_cast<uint64_t>(std::max<int64_t>(t.stride_col, 1)) * es;
  return (s + 15) / 16 * 16;
}

// ---- the kernel variants: (BN, gather, CTAs per tile)

int variant_threads(int bn, bool gather, int cg) {
  if (gather && cg == 2) return kernel_threads<256, true, 2>();
  if (gather) return bn == 128 ? kernel_threads<128, true, 1>() : kernel_threads<256, true, 1>();
  if (cg == 2) {
    switch (bn) {
      case 224: return kernel_threads<224, false, 2>();
      case 192: return kernel_threads<192, false, 2>();
      case 160: return kernel_threads<160, false, 2>();
      default: return kernel_threads<256, false, 2>();
    }
  }
  if (bn == 64) return kernel_threads<64, false, 1>();
  return bn == 128 ? kernel_threads<128, false, 1>() : kernel_threads<256, false, 1>();
}

int variant_units_uncached(int bn, bool gather, int cg, size_t smem, int cluster);

// Resident CTAs (pairs) per device for a variant and shared-memory size, cached.
int variant_units(int bn, bool gather, int cg, size_t smem, int cluster) {
  struct Entry { int dev, bn, cg; bool gather; size_t smem; int cluster, units; };
  static std::mutex mu;
  static Entry cache[64];
  static int n = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < n; ++i) {
      const Entry& e = cache[i];
      if (e.dev == dev && e.bn == bn && e.cg == cg && e.gather == gather && e.smem == smem &&
          e.cluster == cluster)
        return e.units;
    }
  }
  int units;
  {
    RelaxedCaptureMode relaxed;  // the first query may run inside a stream capture
    units = variant_units_uncached(bn, gather, cg, smem, cluster);
  }
  if (units > 0) {
    std::lock_guard<std::mutex> g(mu);
    if (n < 64) cache[n++] = Entry{dev, bn, cg, gather, smem, cluster, units};
  }
  return units;
}

int variant_units_uncached(int bn, bool gather, int cg, size_t smem, int cluster) {
  if (gather && cg == 2) return max_active_units<256, true, 2>(smem, cluster);
  if (gather)
    return bn == 128 ? max_active_units<128, true, 1>(smem, 1) : max_active_units<256, true, 1>(smem, 1);
  if (cg == 2) {
    switch (bn) {
      case 224: return max_active_units<224, false, 2>(smem, cluster);
      case 192: return max_active_units<192, false, 2>(smem, cluster);
      case 160: return max_active_units<160, false, 2>(smem, cluster);
      default: return max_active_units<256, false, 2>(smem, cluster);
    }
  }
  if (bn == 64) return max_active_units<64, false, 1>(smem, 1);
  return bn == 128 ? max_active_units<128, false, 1>(smem, 1) : max_active_units<256, false, 1>(smem, 1);
}

cudaError_t variant_launch(const Plan& pl, cudaStream_t st) {
  if (pl.gather && pl.cg == 2) return launch_gemm<256, true, 2>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
  if (pl.gather)
    return pl.bn == 128 ? launch_gemm<128, true, 1>(pl.tmA, pl.tmB, pl.p, pl.shape, st)
                        : launch_gemm<256, true, 1>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
  if (pl.cg == 2) {
    switch (pl.bn) {
      case 224: return launch_gemm<224, false, 2>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
      case 192: return launch_gemm<192, false, 2>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
      case 160: return launch_gemm<160, false, 2>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
      default: return launch_gemm<256, false, 2>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
    }
  }
  if (pl.p.out_trans) {  // swap_ab: the transposed-output instances (one-CTA tiles)
    if (pl.bn == 64) return launch_gemm<64, false, 1, true>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
    return pl.bn == 128 ? launch_gemm<128, false, 1, true>(pl.tmA, pl.tmB, pl.p, pl.shape, st)
                        : launch_gemm<256, false, 1, true>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
  }
  if (pl.bn == 64) return launch_gemm<64, false, 1>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
  return pl.bn == 128 ? launch_gemm<128, false, 1>(pl.tmA, pl.tmB, pl.p, pl.shape, st)
                      : launch_gemm<256, false, 1>(pl.tmA, pl.tmB, pl.p, pl.shape, st);
}

// Relative time of a pair tile of width bn: tensor-core time per 16-deep MMA
// step (math bn/2 cycles per SM) plus the operand bytes it fetches (measured
// ~6.5 cycles per KiB: A 4 KiB + B 16*bn bytes per SM).
double pair_tile_cost(int bn) { return 0.6 * bn + 26.0; }

// Pair tile width with the least (rounds x tile cost) for `units` resident pairs.
int choose_pair_bn(int64_t tiles_m, int64_t N, int64_t L, int64_t units) {
  static const int kWidths[] = {256, 224, 192, 160};
  int best = 256;
  double best_cost = 0.0;
  for (int bn : kWidths) {
    const int64_t tiles = tiles_m * ((N + bn - 1) / bn) * L;
    const int64_t rounds = (tiles + units - 1) / units;
    const double cost = static_cast<double>(rounds) * pair_tile_cost(bn);
    if (bn == 256 || cost < best_cost * 0.97) {  // prefer the widest tile unless clearly better
      if (bn == 256 || cost < best_cost) { best = bn; best_cost = cost; }
    }
  }
  return best;
}

// Validate and plan.  `encode` = build tensor maps (needs the CUDA driver).
gge_status make_plan(const gge_gemm_args* a, Form form, const int32_t* a_idx,
                     const int32_t* cu, int32_t G, bool want_act, bool act_entry, bool encode,
                     Plan* out, bool dact = false) {
  if (a == nullptr || out == nullptr) return GGE_ERR_INVALID_ARG;
  Plan& pl = *out;
  std::memset(&pl, 0, sizeof(pl));
  Params& p = pl.p;
  const gge_config* cfg = a->config;
  // swap_ab (the pages' GemmConfig.swap_ab): run D^T = B A^T, i.e. the kernel's A is
  // the caller's B and its rows are the caller's N; the epilogue stores transposed
  const bool swap = cfg && (cfg->flags & FLAG_SWAP_AB);
  gge_gemm_args swapped;
  if (swap) {
    if (form != Form::Plain) return GGE_ERR_UNSUPPORTED;
    swapped = *a;
    swapped.A = a->B;
    swapped.B = a->A;
    a = &swapped;
  }
  const bool varlen = (form == Form::Varlen || form == Form::GatherVarlen);
  const bool gk = (form == Form::GatherK);  // varlen-K with A gathered along K
  const bool gather = (form == Form::Gather || form == Form::GatherVarlen || gk);
  const bool vk = (form == Form::VarlenK || gk);
  pl.gather = gather;

  if (a->act < GGE_ACT_NONE || a->act > GGE_ACT_RELU_SQ) return GGE_ERR_INVALID_ARG;
  if (cfg && (cfg->flags & FLAG_RESERVED)) return GGE_ERR_UNSUPPORTED;
  // one dynamic scheduler at a time: the atomic counter or cluster launch control
  const bool clc = cfg && (cfg->flags & FLAG_CLC_SCHED);
  if (clc && (cfg->flags & FLAG_DYNAMIC_SCHED)) return GGE_ERR_INVALID_ARG;
  // the pages' batch_idx_permute: batched plain problems only (the varlen and
  // gather forms order their groups by the group table)
  const int32_t* perm = cfg ? cfg->batch_idx_permute : nullptr;
  if (perm != nullptr && form != Form::Plain) return GGE_ERR_UNSUPPORTED;
  if (dact) {
    // backward epilogue: C = pre-activation and D = dx are required, PostAct optional
    if (a->C == nullptr || a->D == nullptr || a->act == GGE_ACT_NONE) return GGE_ERR_INVALID_ARG;
  } else if (act_entry) {
    if (a->PostAct == nullptr) return GGE_ERR_INVALID_ARG;
  } else if (!want_act) {
    if (a->PostAct != nullptr || a->act != GGE_ACT_NONE) return GGE_ERR_INVALID_ARG;
  }
  if (!dact && a->PostAct == nullptr && a->act != GGE_ACT_NONE) return GGE_ERR_INVALID_ARG;
  if (a->D == nullptr && a->PostAct == nullptr) return GGE_ERR_INVALID_ARG;

  gge_status s = check_view(a->A);
  if (s != GGE_OK) return s;
  s = check_view(a->B);
  if (s != GGE_OK) return s;
  const int32_t adt = a->A.dtype, bdt = a->B.dtype;
  const bool f8 = is8(adt);
  if (!(is16(adt) || is8(adt))) return GGE_ERR_UNSUPPORTED;
  if (is16(adt) && bdt != adt) return GGE_ERR_UNSUPPORTED;
  if (f8 && !is8(bdt)) return GGE_ERR_UNSUPPORTED;
  if (gather && f8) return GGE_ERR_UNSUPPORTED;
  const int es = elem_bytes(adt);

  // shapes from the output
  const gge_tensor* o = a->D ? a->D : a->PostAct;
  // the kernel's problem: M x N per batch (swapped: the caller's N x M)
  const int64_t M = swap ? o->cols : o->rows, N = swap ? o->rows : o->cols, L = o->batch;
  const int64_t out_rows = o->rows, out_cols = o->cols;  // the caller's [M, N]
  // gather-K: A is the source X^T [M, K_src]; the contraction runs over B's columns
  const int64_t K = gk ? a->B.cols : a->A.cols;
  if (M < 0 || N < 0 || K < 0) return GGE_ERR_INVALID_ARG;
  if (a->D) { s = check_mn(a->D, out_rows, out_cols, L, true); if (s != GGE_OK) return s; }
  if (a->PostAct) { s = check_mn(a->PostAct, out_rows, out_cols, L, true); if (s != GGE_OK) return s; }
  if (a->C) { s = check_mn(a->C, out_rows, out_cols, L, false); if (s != GGE_OK) return s; }
  // the caller's output rows are stored in whole 16-byte pieces
  if (out_cols % 8 != 0) return GGE_ERR_UNSUPPORTED;
  // epilogue staging per warp: a 32 x 32 chunk of the widest output
  const int out_es = std::max(a->D ? elem_bytes(a->D->dtype) : 0,
                              a->PostAct ? elem_bytes(a->PostAct->dtype) : 0);
  const bool direct = cfg && (cfg->flags & FLAG_DIRECT_STORES);
  const int out_stage = direct ? 0 : 32 * 32 * out_es;

  // A: [M, K, La] K-major, or M-major (16-bit, TMA-loaded A only); B: [N, K, Lb]
  // K- or N-major (16-bit).  With K == 0 neither is read.
  bool a_mn = false, b_mn = false;
  if (a->B.rows != N || a->B.cols != K) return GGE_ERR_INVALID_ARG;
  if (gk) {
    // the source [M, K_src, 1]: M-major 16-bit, read in 16-byte pieces of 8 rows of M
    if (f8) return GGE_ERR_UNSUPPORTED;
    if (a->A.rows != M || a->A.batch != 1) return GGE_ERR_INVALID_ARG;
    if (M % 8 != 0) return GGE_ERR_UNSUPPORTED;
    if (K > 0 && a->A.cols < 1) return GGE_ERR_INVALID_ARG;
    if (M > 1 && a->A.stride_row != 1) return GGE_ERR_UNSUPPORTED;
    if (a->A.cols > 1 && a->A.stride_col < M) return GGE_ERR_INVALID_ARG;
    if ((a->A.stride_col * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
    a_mn = true;
  }
  if (K > 0) {
    if (gk) {
      // checked above
    } else if (K == 1 || a->A.stride_col == 1) {
      if (a->A.rows > 1 && a->A.stride_row < K) return GGE_ERR_INVALID_ARG;
      if ((a->A.stride_row * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
    } else if (a->A.stride_row == 1 && !gather) {
      a_mn = true;
      if (f8) return GGE_ERR_UNSUPPORTED;  // 8-bit operands must be K-major
      if (a->A.stride_col < a->A.rows) return GGE_ERR_INVALID_ARG;
      if ((a->A.stride_col * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
    } else {
      return GGE_ERR_UNSUPPORTED;
    }
    if (a->A.batch > 1 && (a->A.stride_batch * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
    if (K == 1 || a->B.stride_col == 1) {
      if (N > 1 && a->B.stride_row < K) return GGE_ERR_INVALID_ARG;
      if ((a->B.stride_row * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
    } else if (a->B.stride_row == 1) {
      b_mn = true;
      if (f8) return GGE_ERR_UNSUPPORTED;  // 8-bit operands must be K-major
      if (a->B.stride_col < N) return GGE_ERR_INVALID_ARG;
      if ((a->B.stride_col * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
    } else {
      return GGE_ERR_UNSUPPORTED;
    }
    if (a->B.batch > 1 && (a->B.stride_batch * es) % 16 != 0) return GGE_ERR_ALIGNMENT;
  }

  if (vk) {
    // A [M, total_K], B [N, total_K], outputs [G, M, N]
    if (cu == nullptr) return GGE_ERR_INVALID_ARG;
    if (G < 1 || G > kMaxGroupsHost) return GGE_ERR_UNSUPPORTED;
    if (L != G) return GGE_ERR_INVALID_ARG;
    if (a->A.rows != M || a->A.batch != 1 || a->B.batch != 1) return GGE_ERR_INVALID_ARG;
  } else if (varlen) {
    if (cu == nullptr) return GGE_ERR_INVALID_ARG;
    if (G < 1 || G > kMaxGroupsHost) return GGE_ERR_UNSUPPORTED;
    if (L != 1) return GGE_ERR_INVALID_ARG;
    if (a->B.batch != G) return GGE_ERR_INVALID_ARG;
    if (!gather && (a->A.rows != M || a->A.batch != 1)) return GGE_ERR_INVALID_ARG;
  } else {
    if (a->B.batch != L) return GGE_ERR_INVALID_ARG;
    if (!gather && (a->A.rows != M || a->A.batch != L)) return GGE_ERR_INVALID_ARG;
    // the permutation is copied to shared memory (the group tables' space)
    if (perm != nullptr && L > kMaxGroupsHost) return GGE_ERR_UNSUPPORTED;
  }
  if (gather) {
    if (a_idx == nullptr) return GGE_ERR_INVALID_ARG;
    if (a->A.batch != 1) return GGE_ERR_INVALID_ARG;
    if (!gk && K > 0 && a->A.rows < 1) return GGE_ERR_INVALID_ARG;  // nothing to gather from
    if (!gk && (K * es) % 16 != 0) return GGE_ERR_UNSUPPORTED;  // whole 16-byte chunks along K
  }

  // tile shape: 128 x BN on one CTA, or 256 x BN on a CTA pair
  // (swap_ab runs on one-CTA tiles: its kernel N is the caller's small M)
  int cg = cfg && cfg->cta_group ? cfg->cta_group
                                 : ((!gather && !swap && N > 128 && M >= 256) ? 2 : 1);
  if (swap && cg != 1) return GGE_ERR_UNSUPPORTED;
  // gather-A runs on one CTA or a CTA pair (256 x 256 tiles); gather-K on one CTA
  if (cg == 2 && gk) return GGE_ERR_UNSUPPORTED;
  if (cg != 1 && cg != 2) return GGE_ERR_UNSUPPORTED;
  int bn = cfg && cfg->tile_n ? cfg->tile_n : 0;
  if (cg == 1) {
    if (bn == 0) {
      bn = (N <= 64 && !gather) ? 64 : (N <= 128 ? 128 : 256);
      // fewer 256-wide tiles than CTAs the GPU holds: 128-wide tiles spread the
      // problem over twice as many (measured on skinny problems: 128 x 8192 x 8192
      // 40.8 -> 32.8 us, 64 x 4096 x 8192 26.3 -> 20.7 us)
      if (bn == 256 && !varlen && !vk) {
        int64_t ctas = cfg && cfg->num_ctas > 0 ? cfg->num_ctas : (encode ? sm_count() : 0);
        const int64_t tiles256 = (M + kTileM - 1) / kTileM * ((N + 255) / 256) * L;
        if (ctas > 0 && tiles256 < ctas) bn = 128;
      }
    }
    if (bn != 128 && bn != 256 && !(bn == 64 && !gather)) return GGE_ERR_UNSUPPORTED;
  } else {
    if (bn == 0) {
      bn = 256;
      // narrower tiles even out the last wave; N-major B stages 64-column chunks
      if (!b_mn && !varlen && !vk && !gather) {
        int64_t units = cfg && cfg->num_ctas > 0 ? cfg->num_ctas / 2 : 0;
        if (units <= 0 && encode) {
          // the 256-wide plan: as many stages of (128 + 128) rows as fit, at most kMaxStages
          const int fixed256 = 1024 + kCtrlBytesHost + kEpiWarpsHost * out_stage;
          const int st256 = (kTileM + 128) * kRowBytesHost;
          const size_t smem256 =
              fixed256 + std::min(kMaxStages, (kMaxSmemOptin - fixed256) / st256) * st256;
          units = variant_units(256, false, 2, smem256, 2);
        }
        if (units > 0) bn = choose_pair_bn((M + 2 * kTileM - 1) / (2 * kTileM), N, L, units);
      }
    }
    if (bn != 256 && bn != 224 && bn != 192 && bn != 160) return GGE_ERR_UNSUPPORTED;
    if ((b_mn || gather) && bn != 256) return GGE_ERR_UNSUPPORTED;
  }
  pl.bn = bn;
  pl.cg = cg;
  const int tile_m = kTileM * cg;
  const int bk = kRowBytesHost / es;
  const int stage_bytes = (kTileM + bn / cg) * kRowBytesHost;
  // the varlen group tables, then (gather-K) the staged source-row indices
  // (batch_idx_permute: the permutation, then a 1024-bit table of the batches seen
  // and a flag, where the kernel's group tables would sit)
  const int varlen_bytes = ((varlen || vk) ? 2 * 4 * (kMaxGroupsHost + 1)
                                           : (perm ? 4 * (kMaxGroupsHost + 1) + 4 * 33 : 0)) +
                           (gk ? 16 + 4 * kIdxChunkHost : 0);  // + alignment padding
  const int epi_warps = gather ? kEpiWarpsHost / 2 : kEpiWarpsHost;
  const int fixed = 1024 + kCtrlBytesHost + varlen_bytes + epi_warps * out_stage;
  int stages = (kMaxSmemOptin - fixed) / stage_bytes;
  stages = std::min(stages, kMaxStages);
  if (cfg && cfg->stages > 0) stages = std::min(stages, cfg->stages);
  if (stages < 2) return GGE_ERR_UNSUPPORTED;

  pl.M = M; pl.N = N; pl.K = K; pl.L = L;
  const int64_t tiles_n = (N + bn - 1) / bn;
  const int64_t tiles_m = (M + tile_m - 1) / tile_m;
  pl.empty = (M == 0 || N == 0 || L == 0);

  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.L = static_cast<int32_t>(L);
  p.bk = bk;
  p.k_tiles = static_cast<int32_t>((K + bk - 1) / bk);
  p.stages = stages;
  p.tiles_n = static_cast<int32_t>(tiles_n);
  p.tiles_n_div = FastDivmod::create(tiles_n > 0 ? static_cast<int32_t>(tiles_n) : 1);
  p.batch_perm = perm;
  int64_t num_tiles = 0;
  if (!varlen) {
    num_tiles = tiles_m * tiles_n * L;
    if (num_tiles > kMaxExtent) return GGE_ERR_UNSUPPORTED;
    p.num_tiles = static_cast<int32_t>(num_tiles);
    if (vk) {
      p.k_groups = G;
      p.cu_seqlens_k = cu;
      // a K-major operand's TMA boxes (and gather-K's B copies) start on 16-byte
      // boundaries of its rows; gather-K's A is always M-major
      p.k_align = (a_mn && b_mn) ? 1 : 16 / es;
    }
  } else {
    p.num_groups = G;
    p.cu_seqlens = cu;
    // upper bound on the tile count (the exact count is formed on the device)
    num_tiles = (M / tile_m + G) * tiles_n;
    p.num_tiles = -1;
  }
  if (gather) {
    p.a_idx = a_idx;
    p.a_src = static_cast<const uint8_t*>(a->A.ptr);
    if (gk) {  // index k selects column a_idx[k] of the source: a contiguous M vector
      p.a_src_ld = a->A.stride_col * es;
      p.a_src_rows = static_cast<int32_t>(a->A.cols);
    } else {
      p.a_src_ld = a->A.stride_row * es;
      p.a_src_rows = static_cast<int32_t>(a->A.rows);
      p.k_bytes = static_cast<int32_t>(K * es);
    }
  }
  p.b_src = static_cast<const uint8_t*>(a->B.ptr);
  p.b_ld = (b_mn ? a->B.stride_col : a->B.stride_row) * es;
  // epilogue
  if (a->D) {
    p.d = a->D->ptr; p.ldd = a->D->stride_row; p.sbd = a->D->stride_batch; p.d_dtype = a->D->dtype;
  }
  if (a->PostAct) {
    p.post = a->PostAct->ptr; p.ldp = a->PostAct->stride_row; p.sbp = a->PostAct->stride_batch;
    p.p_dtype = a->PostAct->dtype;
  }
  if (a->C) {
    p.c = a->C->ptr; p.ldc = a->C->stride_row; p.sbc = a->C->stride_batch; p.c_dtype = a->C->dtype;
  }
  p.act = a->act;
  p.dact = dact ? 1 : 0;
  p.out_trans = swap ? 1 : 0;
  p.out_stage_bytes = out_stage;
  p.alpha = a->alpha;
  p.beta = a->beta;
  p.alpha_dev = a->alpha_dev;
  p.beta_dev = a->beta_dev;
  // instruction descriptor: f32 accumulator, operand formats, A / B major, N >> 3, M >> 4
  const uint32_t afmt = f8 ? (adt == GGE_E5M2 ? 1u : 0u) : (adt == GGE_BF16 ? 1u : 0u);
  const uint32_t bfmt = f8 ? (bdt == GGE_E5M2 ? 1u : 0u) : (bdt == GGE_BF16 ? 1u : 0u);
  p.idesc = (1u << 4) | (afmt << 7) | (bfmt << 10) | ((a_mn ? 1u : 0u) << 15) |
            ((b_mn ? 1u : 0u) << 16) |
            ((static_cast<uint32_t>(bn) >> 3) << 17) | ((static_cast<uint32_t>(tile_m) >> 4) << 24);
  p.f8 = f8 ? 1 : 0;
  p.a_mn_major = a_mn ? 1 : 0;
  p.b_mn_major = b_mn ? 1 : 0;
  p.flags = cfg ? cfg->flags : 0;
  p.tile_counts = cfg ? cfg->tile_counts : nullptr;
  p.timeout_ns = (cfg && cfg->timeout_ns) ? cfg->timeout_ns : kDefaultTimeoutNs;

  // launch shape: a persistent grid of at most one CTA (pair) per resident slot
  pl.shape.smem = static_cast<size_t>(fixed + stages * stage_bytes);
  pl.shape.threads = variant_threads(bn, pl.gather, cg);
  pl.shape.cluster = cg;
  const int unit_ctas = pl.shape.cluster;
  int units_cap = cfg && cfg->num_ctas > 0 ? std::max(1, cfg->num_ctas / unit_ctas) : -1;
  if (encode) {
    const int resident = variant_units(bn, pl.gather, cg, pl.shape.smem, pl.shape.cluster);
    if (resident <= 0) return GGE_ERR_CUDA;
    units_cap = units_cap > 0 ? std::min(units_cap, resident) : resident;
  }
  pl.shape.grid =
      units_cap > 0 ? unit_ctas * static_cast<int>(std::min<int64_t>(num_tiles, units_cap)) : -1;
  // cluster launch control: one cluster per tile (those not launched yet are taken over)
  if (clc) {
    if (num_tiles * unit_ctas > kMaxExtent) return GGE_ERR_UNSUPPORTED;
    pl.shape.grid = unit_ctas * static_cast<int>(num_tiles);
  }
  if (!varlen) {
    // raster: bands of m-tiles (or of n-tiles), the band width the caller's or the
    // one that keeps a wave's operand footprint smallest for the units in use
    const bool along_n = cfg && (cfg->flags & FLAG_RASTER_N);
    const int band = cfg && cfg->raster_band > 0
                         ? cfg->raster_band
                         : (units_cap > 0 ? auto_band(units_cap, tile_m, bn, along_n) : 8);
    p.sched = PlainSchedule::create(static_cast<int32_t>(tiles_m), static_cast<int32_t>(tiles_n),
                                    static_cast<int32_t>(L), band, along_n);
    pl.band = p.sched.band;
  }
  // split the last, partly filled wave along K (plain problems, fixed schedule)
  pl.tiles = num_tiles;
  pl.units = units_cap;
  const int32_t flags = cfg ? cfg->flags : 0;
  if (!varlen && !vk && !gather && K > 0 && units_cap > 0 &&
      !(flags & (FLAG_DYNAMIC_SCHED | FLAG_NO_SPLIT | FLAG_CLC_SCHED))) {
    const TailSplit ts = plan_tail_split(num_tiles, units_cap, p.k_tiles);
    if (ts.tail > 0) {
      p.full_tiles = ts.full;
      p.tail_tiles = ts.tail;
      p.tail_splits = ts.splits;
      const int64_t work = static_cast<int64_t>(ts.full) + static_cast<int64_t>(ts.tail) * ts.splits;
      p.num_tiles = static_cast<int32_t>(work);
      pl.shape.grid = unit_ctas * static_cast<int>(std::min<int64_t>(work, units_cap));
    }
  }
  if (pl.empty || !encode) return GGE_OK;
  if (pl.shape.grid <= 0) pl.empty = true;  // e.g. varlen with no rows
  if (pl.empty) return GGE_OK;

  // tensor maps (never read when K == 0)
  if (K > 0) {
    if (gather) {
      // A rows are copied by the gather warps: no tensor map
    } else if (!a_mn) {
      s = encode_3d(&pl.tmA, a->A.ptr, es, K, a->A.rows, a->A.batch,
                    static_cast<uint64_t>(a->A.stride_row) * es, batch_stride_bytes(a->A, es), bk,
                    kTileM);
      if (s != GGE_OK) return s;
    } else {
      s = encode_3d(&pl.tmA, a->A.ptr, es, a->A.rows, K, a->A.batch,
                    static_cast<uint64_t>(a->A.stride_col) * es, mn_batch_stride_bytes(a->A, es),
                    64, bk);
      if (s != GGE_OK) return s;
    }
    if (!b_mn) {
      s = encode_3d(&pl.tmB, a->B.ptr, es, K, N, a->B.batch,
                    static_cast<uint64_t>(a->B.stride_row) * es, batch_stride_bytes(a->B, es), bk,
                    bn / cg);
    } else {
      s = encode_3d(&pl.tmB, a->B.ptr, es, N, K, a->B.batch,
                    static_cast<uint64_t>(a->B.stride_col) * es, mn_batch_stride_bytes(a->B, es),
                    64, bk);
    }
    if (s != GGE_OK) return s;
  }
  return GGE_OK;
}

size_t varlen_k_workspace(const Plan& pl) {
  return kTailBase + static_cast<size_t>(std::max(pl.shape.grid, 0)) * kMapSlotsHost *
                         kMapSlotBytesHost;
}

gge_status check_workspace(void* ws, size_t bytes) {
  if (ws == nullptr) return bytes == 0 ? GGE_OK : GGE_ERR_WORKSPACE;
  if (bytes < kWorkspaceBytes) return GGE_ERR_WORKSPACE;
  if (!aligned16(ws)) return GGE_ERR_ALIGNMENT;
  return GGE_OK;
}

gge_status run(const gge_gemm_args* a, Form form, const int32_t* a_idx, const int32_t* cu,
               int32_t G, bool want_act, bool act_entry, void* ws, size_t ws_bytes,
               gge_stream_t stream, bool dact = false) {
  gge_status s = check_workspace(ws, ws_bytes);
  if (s != GGE_OK) return s;
  // the dynamic tile scheduler keeps its claim counter in the workspace
  if (a != nullptr && a->config != nullptr && (a->config->flags & FLAG_DYNAMIC_SCHED) &&
      ws == nullptr)
    return GGE_ERR_WORKSPACE;
  Plan pl;
  s = make_plan(a, form, a_idx, cu, G, want_act, act_entry, true, &pl, dact);
  if (s != GGE_OK) return s;
  if (pl.empty) return GGE_OK;
  if (pl.p.k_groups > 0) {
    // varlen-K and gather-K: per-CTA tensor-map slots follow the ticket region (the
    // kernel writes the clipped maps of ragged groups there)
    if (ws == nullptr || ws_bytes < varlen_k_workspace(pl)) return GGE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GGE_ERR_ALIGNMENT;
    pl.p.kmaps = static_cast<uint8_t*>(ws) + kTailBase;
  }
  pl.p.status = static_cast<int32_t*>(ws);
  if (pl.p.tail_tiles > 0) {
    if (ws != nullptr && ws_bytes >= tail_workspace(pl) && tickets_fit(pl) &&
        (reinterpret_cast<uintptr_t>(ws) & 255u) == 0) {
      uint8_t* base = static_cast<uint8_t*>(ws);
      pl.p.tail_tickets = reinterpret_cast<int32_t*>(base + kWorkspaceBytes);
      pl.p.partials = reinterpret_cast<float*>(base + kTailBase);
    } else {
      // not enough workspace for the partial sums: run the last wave unsplit
      pl.p.tail_tiles = 0;
      pl.p.num_tiles = static_cast<int32_t>(pl.tiles);
      pl.shape.grid = pl.shape.cluster * static_cast<int>(std::min<int64_t>(pl.tiles, pl.units));
    }
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = variant_launch(pl, st);
  return e == cudaSuccess ? GGE_OK : GGE_ERR_CUDA;
}

}  // namespace

int32_t validate_op(const gge_gemm_args* args, int32_t op, int32_t num_groups) {
  static const int32_t dummy = 0;
  Plan pl;
  const bool act_entry = args != nullptr && args->PostAct != nullptr;
  switch (op) {
    case GGE_OP_GEMM:
      return make_plan(args, Form::Plain, nullptr, nullptr, 0, act_entry, act_entry, false, &pl);
    case GGE_OP_DACT:
      return make_plan(args, Form::Plain, nullptr, nullptr, 0, true, false, false, &pl, true);
    case GGE_OP_VARLEN_M:
      return make_plan(args, Form::Varlen, nullptr, &dummy, num_groups, true, false, false, &pl);
    case GGE_OP_GATHER_A:
      return make_plan(args, num_groups > 0 ? Form::GatherVarlen : Form::Gather, &dummy,
                       num_groups > 0 ? &dummy : nullptr, num_groups, true, false, false, &pl);
    case GGE_OP_VARLEN_K:
      return make_plan(args, Form::VarlenK, nullptr, &dummy, num_groups, true, false, false, &pl);
    case GGE_OP_GATHER_K:
      return make_plan(args, Form::GatherK, &dummy, &dummy, num_groups, true, false, false, &pl);
    default:
      return GGE_ERR_INVALID_ARG;
  }
}

}  // namespace gge

using gge::Form;

extern "C" {

size_t gge_workspace_size(const gge_gemm_args* args, int32_t num_groups) {
  (void)args;
  (void)num_groups;
  // room for the split last wave of any plain problem: the tickets and at most
  // one partial block (128 x 256 fp32) per CTA the GPU can hold
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    return gge::kWorkspaceBytes;
  }
  return gge::kTailBase + static_cast<size_t>(sms) * gge::kTileM * 256 * sizeof(float);
}

gge_status gge_gemm(const gge_gemm_args* args, void* ws, size_t ws_bytes, gge_stream_t stream) {
  return gge::run(args, Form::Plain, nullptr, nullptr, 0, false, false, ws, ws_bytes, stream);
}

gge_status gge_gemm_act(const gge_gemm_args* args, void* ws, size_t ws_bytes,
                        gge_stream_t stream) {
  return gge::run(args, Form::Plain, nullptr, nullptr, 0, true, true, ws, ws_bytes, stream);
}

gge_status gge_gemm_dact(const gge_gemm_args* args, void* ws, size_t ws_bytes,
                         gge_stream_t stream) {
  return gge::run(args, Form::Plain, nullptr, nullptr, 0, true, false, ws, ws_bytes, stream, true);
}

gge_status gge_gemm_varlen_m(const gge_gemm_args* args, const int32_t* cu_seqlens_m,
                             int32_t num_groups, void* ws, size_t ws_bytes, gge_stream_t stream) {
  return gge::run(args, Form::Varlen, nullptr, cu_seqlens_m, num_groups, true, false, ws, ws_bytes,
                  stream);
}

gge_status gge_gemm_gather_a(const gge_gemm_args* args, const int32_t* a_idx,
                             const int32_t* cu_seqlens_m, int32_t num_groups, void* ws,
                             size_t ws_bytes, gge_stream_t stream) {
  const Form f = cu_seqlens_m ? Form::GatherVarlen : Form::Gather;
  return gge::run(args, f, a_idx, cu_seqlens_m, num_groups, true, false, ws, ws_bytes, stream);
}

size_t gge_workspace_size_varlen_k(const gge_gemm_args* args, int32_t num_groups) {
  // a launch has at most one CTA per SM (each CTA takes most of an SM's shared memory)
  (void)args;
  (void)num_groups;
  const int sms = gge::sm_count();
  if (sms <= 0) return 0;
  return gge::kTailBase + static_cast<size_t>(sms) * gge::kMapSlotsHost * gge::kMapSlotBytesHost;
}

gge_status gge_gemm_varlen_k(const gge_gemm_args* args, const int32_t* cu_seqlens_k,
                             int32_t num_groups, void* ws, size_t ws_bytes, gge_stream_t stream) {
  return gge::run(args, Form::VarlenK, nullptr, cu_seqlens_k, num_groups, true, false, ws,
                  ws_bytes, stream);
}

gge_status gge_gemm_gather_k(const gge_gemm_args* args, const int32_t* a_idx,
                             const int32_t* cu_seqlens_k, int32_t num_groups, void* ws,
                             size_t ws_bytes, gge_stream_t stream) {
  return gge::run(args, Form::GatherK, a_idx, cu_seqlens_k, num_groups, true, false, ws, ws_bytes,
                  stream);
}

gge_status gge_read_device_status(void* ws, gge_stream_t stream, int32_t* detail) {
  if (ws == nullptr) return GGE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return GGE_ERR_CUDA;
  int32_t h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return GGE_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof(h)) != cudaSuccess) return GGE_ERR_CUDA;
  if (detail) {
    detail[0] = h[1];
    detail[1] = h[2];
  }
  switch (h[0]) {
    case 0: return GGE_OK;
    case gge::DEV_TIMEOUT: return GGE_ERR_TIMEOUT;
    case gge::DEV_INDEX_RANGE: return GGE_ERR_INDEX_RANGE;
    default: return GGE_ERR_CUDA;
  }
}

const char* gge_status_string(gge_status s) {
  switch (s) {
    case GGE_OK: return "ok";
    case GGE_ERR_INVALID_ARG: return "invalid argument";
    case GGE_ERR_UNSUPPORTED: return "unsupported configuration";
    case GGE_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case GGE_ERR_WORKSPACE: return "workspace missing or too small";
    case GGE_ERR_CUDA: return "CUDA error";
    case GGE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case GGE_ERR_INDEX_RANGE: return "gather index or group offset out of range";
    default: return "unknown status";
  }
}

void gge_fastdivmod_params(int32_t divisor, uint32_t* multiplier, uint32_t* shift) {
  const gge::FastDivmod f = gge::FastDivmod::create(divisor);
  if (multiplier) *multiplier = f.multiplier;
  if (shift) *shift = f.shift;
}

int32_t gge_fastdivmod_div(int32_t divisor, int32_t n) {
  return gge::FastDivmod::create(divisor).div(n);
}

int32_t gge_schedule_map(int32_t tiles_m, int32_t tiles_n, int32_t batches, int32_t band,
                         int32_t along_n, int32_t count, int32_t* out) {
  const gge::PlainSchedule s =
      gge::PlainSchedule::create(tiles_m, tiles_n, batches, band, along_n != 0);
  for (int32_t t = 0; t < count && t < s.num_tiles; ++t) {
    int32_t l, mb, nb;
    s.map(t, l, mb, nb);
    out[3 * t] = l;
    out[3 * t + 1] = mb;
    out[3 * t + 2] = nb;
  }
  return s.num_tiles;
}

gge_status gge_plan(const gge_gemm_args* args, int32_t num_groups, int32_t form,
                    gge_plan_info* out) {
  if (out == nullptr) return GGE_ERR_INVALID_ARG;
  if (form != GGE_FORM_DEFAULT && form != GGE_FORM_GATHER_A && form != GGE_FORM_VARLEN_K &&
      form != GGE_FORM_GATHER_K)
    return GGE_ERR_INVALID_ARG;
  gge::Plan pl;
  const bool gather = form == GGE_FORM_GATHER_A || form == GGE_FORM_GATHER_K;
  const Form f = form == GGE_FORM_VARLEN_K  ? Form::VarlenK
                 : form == GGE_FORM_GATHER_K ? Form::GatherK
                 : gather ? (num_groups > 0 ? Form::GatherVarlen : Form::Gather)
                          : (num_groups > 0 ? Form::Varlen : Form::Plain);
  // a dummy non-null index pointer lets the shape checks run
  static const int32_t dummy = 0;
  const gge_status s = gge::make_plan(args, f, gather ? &dummy : nullptr,
                                      num_groups > 0 ? &dummy : nullptr, num_groups, true, false,
                                      false, &pl);
  if (s != GGE_OK) return s;
  out->tile_m = gge::kTileM * pl.cg;
  out->tile_n = pl.bn;
  out->tile_k = pl.p.bk;
  out->stages = pl.p.stages;
  out->num_tiles = pl.p.num_groups > 0 ? -1 : static_cast<int32_t>(pl.tiles);  // varlen-M: on the device
  out->grid = pl.shape.grid;
  out->threads = pl.shape.threads;
  out->smem_bytes = static_cast<int32_t>(pl.shape.smem);
  out->raster_band = pl.band;
  out->raster_along_n = pl.p.sched.along_n;
  out->cta_group = pl.cg;
  out->tail_tiles = pl.p.tail_tiles;
  out->tail_splits = pl.p.tail_tiles > 0 ? pl.p.tail_splits : 1;
  return GGE_OK;
}

const char* gge_version(void) { return "gge 0.1.0 (sm_103a, tcgen05)"; }

}  // extern "C"
