// Autotuning over the library's launch shapes, after the pages' GemmConfig
// search space (quack-kernels 0.2.0 diff, quack/gemm_config.py,
// get_all_configs): every candidate is timed on the caller's stream with CUDA
// events and the fastest is kept, per problem, in an in-process cache.
//
// The candidates are the shapes the kernels have: one CTA per 128 x 128 or
// 128 x 256 tile, or a CTA pair per 256 x {256, 224, 192, 160} tile, times the
// raster of plain problems (bands of m-tiles of the automatic width or 8, or
// bands of n-tiles: the pages' raster_order / max_swizzle_size), times staged
// or direct epilogue stores.  The pages' cooperative / ping-pong choice
// has no counterpart (the accumulator is double-buffered in TMEM instead), and
// their cluster shapes correspond to the one-CTA / CTA-pair choice.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>

#include "../../include/gge.h"
#include "gge_launch.h"

namespace {

constexpr int kMaxCandidates = 64;

bool plain_op(int32_t op) { return op == GGE_OP_GEMM || op == GGE_OP_DACT; }
// CTA pairs: every form but gather-K; with gathered A rows, 256-wide tiles only
bool pair_shape_ok(int32_t op, int tile_n) {
  if (op == GGE_OP_GATHER_K) return false;
  return op != GGE_OP_GATHER_A || tile_n == 256;
}

// All candidates the planner accepts, in a fixed order.
int32_t enumerate(const gge_gemm_args* args, int32_t op, int32_t num_groups, gge_config* out,
                  int32_t max) {
  if (args == nullptr) return 0;
  gge_config base{};
  if (args->config != nullptr) base = *args->config;
  base.flags &= ~gge::FLAG_SWAP_AB;
  const gge_tensor* o = args->D ? args->D : args->PostAct;
  const int64_t out_m = o ? o->rows : 0, out_n = o ? o->cols : 0;
  struct Shape { int cg, tile_n; };
  static const Shape kShapes[] = {{2, 256}, {2, 224}, {2, 192}, {2, 160}, {1, 256}, {1, 128},
                                  {1, 64}};
  struct Raster { int band; bool along_n; };
  static const Raster kRasters[] = {{0, false}, {8, false}, {0, true}};
  const int n_rasters = plain_op(op) ? 3 : 1;
  // swap_ab (the pages' GemmConfig.swap_ab) is searched for plain problems whose M
  // is small next to N: the swapped problem's tile width covers the small M
  const bool try_swap = plain_op(op) && out_m > 0 && out_m <= 256 && out_m < out_n;
  int32_t n = 0;
  for (int swap = 0; swap < (try_swap ? 2 : 1); ++swap) {
    const int64_t width = swap ? out_m : out_n;  // the kernel's N
    for (const Shape& sh : kShapes) {
      if (sh.cg == 2 && !pair_shape_ok(op, sh.tile_n)) continue;
      if (sh.tile_n == 64 && width > 128) continue;  // 64-wide tiles only for narrow outputs
      // swapped candidates: the automatic raster and staged stores only
      for (int b = 0; b < (swap ? 1 : n_rasters); ++b) {
        for (int direct = 0; direct < (swap ? 1 : 2); ++direct) {
          gge_config c = base;
          c.cta_group = sh.cg;
          c.tile_n = sh.tile_n;
          c.raster_band = kRasters[b].band;
          int32_t f = direct ? (base.flags | gge::FLAG_DIRECT_STORES)
                             : (base.flags & ~gge::FLAG_DIRECT_STORES);
          if (n_rasters > 1)
            f = kRasters[b].along_n ? (f | gge::FLAG_RASTER_N) : (f & ~gge::FLAG_RASTER_N);
          if (swap) f |= gge::FLAG_SWAP_AB;
          c.flags = f;
          gge_gemm_args a = *args;
          a.config = &c;
          if (gge::validate_op(&a, op, num_groups) != GGE_OK) continue;
          if (n < max && out != nullptr) out[n] = c;
          ++n;
        }
      }
    }
  }
  return n;
}

gge_status launch(const gge_gemm_args* a, int32_t op, const int32_t* idx, const int32_t* cu,
                  int32_t g, void* ws, size_t ws_bytes, gge_stream_t st) {
  switch (op) {
    case GGE_OP_GEMM:
      return a->PostAct ? gge_gemm_act(a, ws, ws_bytes, st) : gge_gemm(a, ws, ws_bytes, st);
    case GGE_OP_DACT: return gge_gemm_dact(a, ws, ws_bytes, st);
    case GGE_OP_VARLEN_M: return gge_gemm_varlen_m(a, cu, g, ws, ws_bytes, st);
    case GGE_OP_GATHER_A: return gge_gemm_gather_a(a, idx, cu, g, ws, ws_bytes, st);
    case GGE_OP_VARLEN_K: return gge_gemm_varlen_k(a, cu, g, ws, ws_bytes, st);
    case GGE_OP_GATHER_K: return gge_gemm_gather_k(a, idx, cu, g, ws, ws_bytes, st);
    default: return GGE_ERR_INVALID_ARG;
  }
}

void add_tensor(std::string& k, const gge_tensor* t) {
  char buf[160];
  if (t == nullptr) {
    k += "|-";
    return;
  }
  // shapes, dtype and which strides are unit (the layout), not the addresses
  std::snprintf(buf, sizeof(buf), "|%d:%lldx%lldx%lld:%d%d", t->dtype,
                static_cast<long long>(t->rows), static_cast<long long>(t->cols),
                static_cast<long long>(t->batch), t->stride_row == 1 ? 1 : 0,
                t->stride_col == 1 ? 1 : 0);
  k += buf;
}

// The cache key: device, op, groups, every operand's shape / dtype / layout,
// the activation, and the parts of the caller's config the search keeps.
std::string key_of(const gge_gemm_args* a, int32_t op, int32_t g) {
  int dev = -1;
  cudaGetDevice(&dev);
  char buf[96];
  std::snprintf(buf, sizeof(buf), "%d|%d|%d|%d", dev, op, g, a->act);
  std::string k = buf;
  add_tensor(k, &a->A);
  add_tensor(k, &a->B);
  add_tensor(k, a->C);
  add_tensor(k, a->D);
  add_tensor(k, a->PostAct);
  if (a->config != nullptr) {
    std::snprintf(buf, sizeof(buf), "|f%d|n%d|s%d", a->config->flags, a->config->num_ctas,
                  a->config->stages);
    k += buf;
  }
  return k;
}

std::mutex g_mu;
std::map<std::string, gge_config>& cache() {
  static std::map<std::string, gge_config> m;
  return m;
}

}  // namespace

extern "C" {

int32_t gge_tune_candidates(const gge_gemm_args* args, int32_t op, int32_t num_groups,
                            gge_config* out, int32_t max) {
  return enumerate(args, op, num_groups, out, max);
}

gge_status gge_autotune(const gge_gemm_args* args, int32_t op, const int32_t* idx,
                        const int32_t* cu, int32_t num_groups, void* ws, size_t ws_bytes,
                        gge_stream_t stream, int32_t reps, gge_config* best, float* best_ms) {
  if (args == nullptr || best == nullptr || reps < 1) return GGE_ERR_INVALID_ARG;
  gge_config cand[kMaxCandidates];
  const int32_t n = std::min<int32_t>(enumerate(args, op, num_groups, cand, kMaxCandidates),
                                      kMaxCandidates);
  if (n == 0) return static_cast<gge_status>(gge::validate_op(args, op, num_groups));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return GGE_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return GGE_ERR_CUDA;
  }
  gge_status status = GGE_OK;
  float best_t = -1.f;
  for (int32_t i = 0; i < n && status == GGE_OK; ++i) {
    gge_gemm_args a = *args;
    a.config = &cand[i];
    gge_status s = launch(&a, op, idx, cu, num_groups, ws, ws_bytes, stream);  // warm-up
    if (s == GGE_ERR_INVALID_ARG || s == GGE_ERR_UNSUPPORTED) continue;
    if (s != GGE_OK) { status = s; break; }
    if (cudaEventRecord(e0, st) != cudaSuccess) { status = GGE_ERR_CUDA; break; }
    for (int32_t r = 0; r < reps && s == GGE_OK; ++r)
      s = launch(&a, op, idx, cu, num_groups, ws, ws_bytes, stream);
    if (s != GGE_OK) { status = s; break; }
    float ms = 0.f;
    if (cudaEventRecord(e1, st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
      status = GGE_ERR_CUDA;
      break;
    }
    ms /= static_cast<float>(reps);
    if (best_t < 0.f || ms < best_t) {
      best_t = ms;
      *best = cand[i];
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (status != GGE_OK) return status;
  if (best_t < 0.f) return GGE_ERR_UNSUPPORTED;  // every candidate was rejected
  if (best_ms != nullptr) *best_ms = best_t;
  std::lock_guard<std::mutex> g(g_mu);
  cache()[key_of(args, op, num_groups)] = *best;
  return GGE_OK;
}

gge_status gge_tuned_config(const gge_gemm_args* args, int32_t op, int32_t num_groups,
                            gge_config* out) {
  if (args == nullptr || out == nullptr) return GGE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_mu);
  auto it = cache().find(key_of(args, op, num_groups));
  if (it == cache().end()) return GGE_ERR_INVALID_ARG;
  // the search's launch shape with this caller's own pointers and limit
  gge_config c = it->second;
  const gge_config* mine = args->config;
  c.tile_counts = mine ? mine->tile_counts : nullptr;
  c.timeout_ns = mine ? mine->timeout_ns : 0;
  c.batch_idx_permute = mine ? mine->batch_idx_permute : nullptr;
  *out = c;
  return GGE_OK;
}

}  // extern "C"
