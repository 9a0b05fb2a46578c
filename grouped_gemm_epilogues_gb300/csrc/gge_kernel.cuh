// Persistent, warp-specialised GEMM with a fused epilogue for sm_103a.
//
//   D       = alpha * A * B^T + beta * C          (rounded to D's dtype)
//   PostAct = act(alpha * A * B^T + beta * C)     (act on the unrounded fp32 value)
//
// after quack/dense_gemm_sm90.py (GemmSm90) and quack/gemm_act_sm90.py
// (GemmActSm90.epi_visit_acc_subtile), rebuilt for the 5th-generation
// tensor core instead of Hopper warpgroup MMA:
//
//   warps 0-7  epilogue: TMEM -> registers (tcgen05.ld), alpha / beta / C /
//              activation in fp32, round, and store D and PostAct through a
//              per-warp shared-memory transpose (row-contiguous stores).  Warp w
//              owns TMEM lanes 32(w%4)..+31 (tile rows) and every other
//              32-column chunk (warps 0-3 and every chunk in the gather forms).
//   warp  8    TMEM allocator and MMA issuer (one elected lane): tcgen05.mma
//              128 x BN x 16 (x32 for 8-bit) from shared memory into a
//              double-buffered fp32 TMEM accumulator, so the epilogue of
//              tile i overlaps the main loop of tile i+1 (this replaces the
//              pages' ping-pong warpgroups).  (warp 4 in the gather forms)
//   warp  9    TMA producer: A and B k-tiles into an S-stage shared-memory
//              ring (128-byte swizzle), one mbarrier pair per stage.
//   warp 10    varlen-K: writes each ragged group's clipped tensor maps ahead
//              of the producer (otherwise idle).
//   warps 5-8  (gather forms) row gathers with 16-byte cp.async into the same
//              swizzled layouts, B by TMA (GemmSm90.load_AB_gather_A, and the
//              gather along K of varlen-K).
//
// With CG = 2 a cluster of two CTAs (a CTA pair) computes a 256 x BN tile
// (BN = 256, 224, 192 or 160; narrower tiles even out the last wave):
// each CTA stages its own 128 rows of A and half of the BN columns of B, the
// leader CTA issues tcgen05.mma.cta_group::2 over both CTAs' shared memory,
// and each CTA's TMEM receives its own 128 accumulator rows.  The pair halves
// the B bytes each SM stages per FLOP, so a stage is 32 KiB instead of 48 KiB
// and six stages fit.
//
// Every CTA (pair) walks the same static persistent schedule (tile t, t + grid, ...),
// or claims tiles from an atomic counter; tile coordinates come from
// FastDivmod (plain) or from a per-group tile prefix sum in shared memory
// (varlen-M, VarlenMTileScheduler's role).  On plain problems a last wave that
// is at most half full is split along K: its tiles' K-slices run on otherwise
// idle units, which leave fp32 partial sums in the workspace; whichever unit
// finishes a tile's slices last adds them up and runs the epilogue
// (plan_tail_split).  No unit ever waits for another one.
//
// Launches use programmatic dependent launch: a CTA sets up its shared memory
// and TMEM, then waits (griddepcontrol.wait) for the previous kernel in the
// stream before touching global memory, and lets the next launch start as
// soon as SMs free up.
//
// Every mbarrier wait is bounded by
// Params::timeout_ns of %globaltimer; on expiry the kernel records
// DEV_TIMEOUT in the status words, raises a shared abort flag so that every
// role leaves its loop, lets copies in flight land, frees its TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gge_params.h"
#include "gge_ptx.cuh"

namespace gge {

constexpr int kBM = 128;           // tile rows = TMEM lanes
constexpr int kRowBytes = 128;     // bytes of K per stage row (one swizzle span)

constexpr int kGatherWarps = 4;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kMaxGroups = 1024;   // varlen groups held in shared memory
// gather-K: source-row indices of up to this many K rows (32 k-tiles) are staged
// in shared memory at a time
constexpr int kIdxChunk = 2048;
constexpr int kCtrlBytes = 1024;   // barriers, flags and the tile ring (bytes 0..255),
                                   // the varlen-K tensor-map scratch (256..511) and
                                   // map-slot barriers (512..767)
constexpr int kMapScratch = 256;
constexpr int kMapBars = 512;
constexpr int kClcBar = 768;       // cluster launch control: its barrier and (at +16) the
                                   // 16-byte response
constexpr int kRelayWord = 800;    // gathering pair: the word the peer's relay stores into
constexpr int kSchedDepth = 4;     // tile indices in flight between the fetching warp and the rest
constexpr int kTicketsPerWarp = 4; // split tail: one ticket per epilogue warp and 32-column chunk
constexpr int kMapSlots = 16;      // varlen-K: tensor-map copies per CTA (> pipeline stages)
constexpr int kMapSlotBytes = 256; // one A and one B tensor map
// barriers for up to 8 stages, the TMEM slot, the abort flag and the tile ring
static_assert(8 * (2 * 8 + 5 + 2 * kSchedDepth) + 8 + 4 * kSchedDepth <= kMapScratch,
              "control block overlaps the tensor-map scratch");
static_assert(kMapBars + 16 * kMapSlots <= kClcBar, "map-slot barriers overflow");
static_assert(kClcBar + 32 <= kRelayWord && kRelayWord + 4 <= kCtrlBytes, "control block overflow");

template <int BN, bool GATHER, int CG>
struct KernelCfg {
  static constexpr int kTileM = kBM * CG;        // rows of one (pair) tile
  static constexpr int kBRows = BN / CG;         // B rows staged by each CTA
  static constexpr int kABytes = kBM * kRowBytes;
  static constexpr int kBBytes = kBRows * kRowBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // epilogue warps: two per TMEM lane quadrant (one in the gather forms, whose
  // four copy warps need the registers), then the MMA warp, then the producer
  // warp(s): one TMA warp and the map warp, or the gather warps
  static constexpr int kEpiWarps = GATHER ? 4 : 8;
  static constexpr int kMmaWarp = kEpiWarps;
  static constexpr int kLoadWarp = kEpiWarps + 1;
  // TMA forms: one more warp writes the varlen-K tensor maps ahead of the producer
  static constexpr int kMapWarp = kLoadWarp + 1;
  static constexpr int kWarps = GATHER ? kLoadWarp + kGatherWarps : kLoadWarp + 2;
  static constexpr int kThreads = kWarps * 32;
  // two accumulator buffers of BN columns; the allocation is the next power of two
  static constexpr int kTmemCols = (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN: a multiple of 32 in [64, 256]");
  static_assert(kBRows % 8 == 0, "B rows per CTA must fill 8-row swizzle atoms");
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
  static_assert(GATHER || (BN / 32 + kEpiWarps / 4 - 1) / (kEpiWarps / 4) <= kTicketsPerWarp,
                "split-tail tickets: one per epilogue warp and chunk (the gather forms never split)");
};

// Shared-memory matrix descriptor for a K-major (or N-major) operand staged
// with the 128-byte swizzle: start address, leading / stride byte offsets
// (>> 4), descriptor version 1, swizzle mode 2 (128B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
         (uint64_t(2) << 61);
}

struct TileCoord {
  int32_t m_row0;     // first output row of the tile (global row in varlen form)
  int32_t row_limit;  // rows >= this are not written (batch end / group end)
  int32_t n0;
  int32_t batch;      // batch index (plain) or group index (varlen)
  int32_t a_batch;    // third TMA coordinate of A
  int32_t b_batch;    // third TMA coordinate of B
};

struct Shared {
  uint32_t full, empty, tfull, tempty;  // barrier array bases (shared addresses)
  uint32_t map_full, map_empty;         // varlen-K map-slot barriers (kMapSlots each)
  volatile int32_t* abort;
  const int32_t* prefix;  // varlen-M: tile prefix [G+1]; varlen-K: group K ends [G];
                          // plain with batch_idx_permute: the permutation [L]
  const int32_t* cu;      // varlen-M: cu_seqlens copy [G+1]; varlen-K: group K starts [G]
  int32_t* idx;           // gather-K: staged source-row indices [kIdxChunk]
};

template <int BN, int TILE_M>
__device__ __forceinline__ TileCoord tile_coord(int32_t t, const Params& p, const Shared& sh) {
  TileCoord tc;
  if (p.num_groups > 0) {
    int lo = 0, hi = p.num_groups;  // prefix[lo] <= t < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sh.prefix[mid] <= t) lo = mid; else hi = mid;
    }
    int32_t mb, nb;
    p.tiles_n_div.divmod(t - sh.prefix[lo], mb, nb);
    tc.m_row0 = sh.cu[lo] + mb * TILE_M;
    tc.row_limit = min(sh.cu[lo + 1], p.M);
    tc.n0 = nb * BN;
    tc.batch = lo;
    tc.a_batch = 0;
    tc.b_batch = lo;
  } else {
    // a split tail item computes a slice of tile full_tiles + (t - full_tiles) / tail_splits
    const int32_t tt =
        (p.tail_tiles > 0 && t >= p.full_tiles) ? p.full_tiles + (t - p.full_tiles) / p.tail_splits : t;
    int32_t l, mb, nb;
    p.sched.map(tt, l, mb, nb);
    if (p.batch_perm != nullptr) l = sh.prefix[l];  // checked copy of batch_idx_permute
    tc.m_row0 = mb * TILE_M;
    tc.row_limit = p.M;
    tc.n0 = nb * BN;
    tc.batch = l;
    // varlen-K operands are single [rows, total_K] matrices
    tc.a_batch = p.k_groups > 0 ? 0 : l;
    tc.b_batch = tc.a_batch;
  }
  return tc;
}

// The K columns a tile contracts: [k0, k_end) in k-tiles of bk.  `ragged`: a
// varlen-K group whose length is not a whole number of MMA K-steps, so its
// last step must read zeros past k_end (through a tensor map clipped at k_end);
// every other range is cut exactly by issuing only the K-steps it covers.
struct KRange {
  int32_t k0, k_end, tiles;
  bool ragged;
};

__device__ __forceinline__ int32_t mma_kstep(const Params& p) { return p.f8 ? 32 : 16; }

// K range of work item t (batch / group `batch`): all of K, a varlen-K group's
// columns, or one K-slice of a split tail tile (k-tiles s k_tiles / S ..
// (s + 1) k_tiles / S of slice s).
__device__ __forceinline__ KRange k_range(const Params& p, const Shared& sh, int32_t batch,
                                          int32_t t) {
  if (p.k_groups == 0) {
    if (p.tail_tiles > 0 && t >= p.full_tiles) {
      const int32_t sl = (t - p.full_tiles) % p.tail_splits;
      const int32_t kt0 = sl * p.k_tiles / p.tail_splits;
      const int32_t kt1 = (sl + 1) * p.k_tiles / p.tail_splits;
      return KRange{kt0 * p.bk, min(p.K, kt1 * p.bk), kt1 - kt0, false};
    }
    return KRange{0, p.K, p.k_tiles, false};
  }
  const int32_t lo = sh.cu[batch], hi = sh.prefix[batch];
  return KRange{lo, hi, (hi - lo + p.bk - 1) / p.bk, ((hi - lo) & (mma_kstep(p) - 1)) != 0};
}

// Serpentine K (config flag bit 10, plain and varlen-M TMA forms): work items of
// odd waves (item / units) walk their k-tiles backwards, so that a wave starts
// on the k-slices of A and B that the previous wave read last and are still
// in L2.  The direction depends only on the item, so results are reproducible.
__device__ __forceinline__ bool k_reversed(const Params& p, int32_t t, int32_t units) {
  return (p.flags & FLAG_K_SERPENTINE) && p.k_groups == 0 && ((t / units) & 1);
}

// MMA K-steps of k-tile kt (4 per full k-tile; the last one stops at k_end).
__device__ __forceinline__ int32_t ksteps_of(const Params& p, const KRange& kr, int32_t kt) {
  const int32_t left = kr.k_end - (kr.k0 + kt * p.bk);
  const int32_t step = mma_kstep(p);
  return min(4, (left + step - 1) / step);
}

__device__ __forceinline__ void record_status(const Params& p, int32_t code, int32_t where,
                                              int32_t tile) {
  if (p.status != nullptr) {
    if (atomicCAS(p.status, 0, code) == 0) {
      p.status[1] = where;
      p.status[2] = tile;
    }
  }
}

// Slow path of a bounded mbarrier wait: wait until the phase completes, the
// CTA aborts, or timeout_ns of %globaltimer pass (then record and abort).
// `sleep`: probe with the sleeping try_wait (the thread issues nothing until the
// phase completes) instead of short polls.  Measured: sleeping waits for the
// epilogue's accumulator (long waits, many warps) are ~0.5 % faster under the
// power cap; for the copy warps' and MMA warp's short stage waits they cost up
// to 2.5 % (gather-K), so those poll.
static __device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             int32_t* status, volatile int32_t* abort,
                                             int32_t where, int32_t tile, bool cluster_scope,
                                             bool sleep) {
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (sleep) {
      if (cluster_scope ? ptx::mbar_try_wait_cluster_sleep(bar, parity)
                        : ptx::mbar_try_wait_sleep(bar, parity))
        return true;
    } else {
#pragma unroll 1
      for (int i = 0; i < 32; ++i)
        if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
          return true;
    }
    if (*abort) return false;
    if (ptx::globaltimer() - t0 > timeout_ns) {
      if (status != nullptr && atomicCAS(status, 0, DEV_TIMEOUT) == 0) {
        status[1] = where;
        status[2] = tile;
      }
      *abort = 1;
      return false;
    }
  }
}

// Bounded wait on an mbarrier phase.  Returns false on abort or timeout.
// CLUSTER: acquire at cluster scope (barriers that the peer CTA signals).
// SLEEP: the slow path sleeps in try_wait instead of polling.
template <bool CLUSTER = false, bool SLEEP = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Params& p,
                                           const Shared& sh, int32_t where, int32_t tile) {
  if (CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
    return true;
  return wait_phase_slow(bar, parity, p.timeout_ns, p.status, sh.abort, where, tile, CLUSTER,
                         SLEEP);
}

// ------------------------------------------------------------- tile stream
// Every role walks the same tile sequence.  Static: unit, unit + units, ...
// Dynamic (quack/dense_gemm_sm90.py's tile_count_semaphore): after its first
// tile, the fetching warp (the producer; the leader's producer for a pair)
// claims tiles from an atomic counter in the workspace and hands each index to
// the other warps (and the peer CTA) through a small shared-memory ring.
// Cluster launch control (the later gemm_sm90.py's use_clc_persistence, which
// the pages gate on Blackwell): the grid has one cluster per tile; after its
// own tile, a cluster's fetching warp cancels a cluster that has not been
// launched yet and takes over its tile, until no cluster is left to cancel.
// One cancellation request is kept in flight, issued as soon as the previous
// answer is in, so its latency hides behind the current tile.  An index >=
// num_tiles ends every role's loop.
struct TileSched {
  int32_t unit, units;
  int32_t* counter;      // workspace claim counter (dynamic)
  uint32_t full, empty;  // ring barriers (kSchedDepth each)
  uint32_t ring;         // int32 ring[kSchedDepth]
  bool dyn;              // indices pass through the ring (atomic counter or CLC)
};

// The fetching warp's lane 0, cluster launch control: the tile of item i.
// (its barrier and response sit at fixed offsets of the control block)
__device__ __forceinline__ uint32_t clc_bar_addr(const Shared& sh) {
  return sh.map_full + (kClcBar - kMapBars);
}

__device__ __forceinline__ int32_t clc_next(const TileSched& ts, int i, const Params& p,
                                                const Shared& sh, int32_t num_tiles, int cg) {
  const uint32_t bar = clc_bar_addr(sh), resp = bar + 16;
  int32_t t = ts.unit;
  if (i > 0) {
    // the answer to the request issued at item i - 1 (request r completes phase r & 1)
    t = 0x7fffffff;
    if (wait_phase(bar, static_cast<uint32_t>(i - 1) & 1u, p, sh, 13, i)) {
      int32_t x = 0;
      if (ptx::clc_query(resp, x)) t = x / cg;
    }
  }
  if (t < num_tiles) {  // ask for the next one now (none after a refusal: the grid is done)
    ptx::mbar_arrive_expect_tx(bar, 16);
    ptx::clc_try_cancel(resp, bar);
  }
  return t;
}

template <int CG>
__device__ __forceinline__ int32_t sched_fetch(const TileSched& ts, int i, const Params& p,
                                               const Shared& sh, int32_t num_tiles) {
  if (!ts.dyn) return ts.unit + i * ts.units;
  const int slot = i % kSchedDepth;
  const uint32_t ph = static_cast<uint32_t>(i / kSchedDepth) & 1u;
  const bool ok = wait_phase<CG == 2>(ts.empty + 8 * slot, ph ^ 1u, p, sh, 7, i);
  if (!__all_sync(0xffffffffu, ok)) return 0x7fffffff;
  int32_t t = 0;
  if ((threadIdx.x & 31) == 0) {
    if (p.flags & FLAG_CLC_SCHED) t = clc_next(ts, i, p, sh, num_tiles, CG);
    else t = (i == 0) ? ts.unit : ts.units + atomicAdd(ts.counter, 1);
    const uint32_t slot_addr = ts.ring + 4 * slot;
    ptx::st_shared_u32(slot_addr, static_cast<uint32_t>(t));
    if (CG == 2) ptx::st_shared_cluster_u32(ptx::mapa(slot_addr, 1), static_cast<uint32_t>(t));
    ptx::mbar_arrive(ts.full + 8 * slot);
    if (CG == 2) ptx::mbar_arrive_cluster(ptx::mapa(ts.full + 8 * slot, 1));
  }
  return __shfl_sync(0xffffffffu, t, 0);
}

template <int CG>
__device__ __forceinline__ int32_t sched_next(const TileSched& ts, int i, const Params& p,
                                              const Shared& sh) {
  if (!ts.dyn) return ts.unit + i * ts.units;
  const int slot = i % kSchedDepth;
  const uint32_t ph = static_cast<uint32_t>(i / kSchedDepth) & 1u;
  const bool ok = wait_phase<CG == 2>(ts.full + 8 * slot, ph, p, sh, 7, i);
  if (!__all_sync(0xffffffffu, ok)) return 0x7fffffff;
  const int32_t t = static_cast<int32_t>(ptx::ld_shared_u32(ts.ring + 4 * slot));
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {  // this warp is done with the slot (the leader's ring owns it)
    if (CG == 1) ptx::mbar_arrive(ts.empty + 8 * slot);
    else ptx::mbar_arrive_remote(ptx::mapa(ts.empty + 8 * slot, 0));
  }
  return t;
}

// ------------------------------------------------------------- epilogue math

// exp(-2u) for gelu_tanh's u = sqrt(2/pi) (x + 0.044715 x^3): with exp(y) = 2^(y log2 e)
// the exponent is x (k0 + k1 x^2), the three constant factors folded into k0 and k1.
__device__ __forceinline__ float gelu_exp_m2u(float x) {
  constexpr float k0 = static_cast<float>(-2.0 * 0.7978845608028654 * 1.4426950408889634);
  constexpr float k1 = static_cast<float>(-2.0 * 0.7978845608028654 * 1.4426950408889634 *
                                          0.044715);
  return ptx::ex2_approx(x * fmaf(k1, x * x, k0));
}

// exp(-x) as 2^(-x log2 e).
__device__ __forceinline__ float exp_neg(float x) {
  constexpr float kNegLog2e = static_cast<float>(-1.4426950408889634);
  return ptx::ex2_approx(x * kNegLog2e);
}

// The activation of one value; ACT is fixed at compile time.
template <int ACT>
__device__ __forceinline__ float act_one(float x) {
  if constexpr (ACT == ACT_RELU) {
    return (x <= 0.f) ? 0.f : x;  // NaN propagates, -0 -> +0
  } else if constexpr (ACT == ACT_GELU_TANH) {
    // 0.5 x (1 + tanh u) written as x / (1 + exp(-2u)): no cancellation in the tail;
    // one base-2 exponential, one reciprocal and five FP32 operations a value
    return x * ptx::rcp_approx(1.f + gelu_exp_m2u(x));
  } else if constexpr (ACT == ACT_SILU) {
    return x * ptx::rcp_approx(1.f + exp_neg(x));
  } else if constexpr (ACT == ACT_RELU_SQ) {
    return (x <= 0.f) ? 0.f : x * x;
  } else {
    return x;
  }
}

// act'(x) for the backward epilogue.
template <int ACT>
__device__ __forceinline__ float dact_one(float x) {
  if constexpr (ACT == ACT_RELU) {
    return (x > 0.f) ? 1.f : 0.f;
  } else if constexpr (ACT == ACT_RELU_SQ) {
    return (x <= 0.f) ? 0.f : 2.f * x;
  } else if constexpr (ACT == ACT_GELU_TANH) {
    // s = sigmoid(2u) = (1 + tanh u) / 2 and 1 - tanh^2 u = 4 s (1 - s)
    const float s = ptx::rcp_approx(1.f + gelu_exp_m2u(x));
    const float du = 0.7978845608028654f * fmaf(3.f * 0.044715f * x, x, 1.f);
    return fmaf(2.f * x * s * (1.f - s), du, s);
  } else if constexpr (ACT == ACT_SILU) {
    const float s = ptx::rcp_approx(1.f + exp_neg(x));
    return s * fmaf(x, 1.f - s, 1.f);
  } else {
    return 1.f;
  }
}

// The activation's choice is made once per 32-value chunk, outside the value
// loop: switched per value, the unrolled loop kept every activation's
// arithmetic in the instruction stream.
template <int ACT>
__device__ __forceinline__ void act_chunk_t(float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = act_one<ACT>(v[j]);
}

__device__ __forceinline__ void act_chunk(int act, float (&v)[32]) {
  switch (act) {
    case ACT_RELU: act_chunk_t<ACT_RELU>(v); break;
    case ACT_GELU_TANH: act_chunk_t<ACT_GELU_TANH>(v); break;
    case ACT_SILU: act_chunk_t<ACT_SILU>(v); break;
    case ACT_RELU_SQ: act_chunk_t<ACT_RELU_SQ>(v); break;
    default: break;
  }
}

// y = act'(x) * dout over a chunk.
template <int ACT>
__device__ __forceinline__ void dact_chunk_t(const float (&x)[32], const uint32_t (&dout)[32],
                                             float (&y)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) y[j] = dact_one<ACT>(x[j]) * __uint_as_float(dout[j]);
}

__device__ __forceinline__ void dact_chunk(int act, const float (&x)[32],
                                           const uint32_t (&dout)[32], float (&y)[32]) {
  switch (act) {
    case ACT_RELU: dact_chunk_t<ACT_RELU>(x, dout, y); break;
    case ACT_GELU_TANH: dact_chunk_t<ACT_GELU_TANH>(x, dout, y); break;
    case ACT_SILU: dact_chunk_t<ACT_SILU>(x, dout, y); break;
    case ACT_RELU_SQ: dact_chunk_t<ACT_RELU_SQ>(x, dout, y); break;
    default: dact_chunk_t<ACT_NONE>(x, dout, y); break;
  }
}

__device__ __forceinline__ int dtype_bytes(int dt) { return dt == DT_F32 ? 4 : 2; }

// Raw bits of one thread's 32 columns of a 16-bit C, loaded one chunk ahead.
// (An fp32 C is read where it is used: holding two chunks of it would cost 32
// more registers than the epilogue has.)
struct CRegs {
  uint4 w[4];
};

// Address of C[row, col0] of batch `batch`.  TR (swap_ab): the caller's C holds
// the kernel's element (row, col) at [col][row].
template <bool TR = false>
__device__ __forceinline__ const char* c_ptr(const Params& p, int32_t row, int32_t col0,
                                             int32_t batch) {
  const int64_t out_batch = (p.num_groups > 0) ? 0 : batch;
  const int64_t off = TR ? static_cast<int64_t>(col0) * p.ldc + row
                         : static_cast<int64_t>(row) * p.ldc + col0;
  return static_cast<const char*>(p.c) + (out_batch * p.sbc + off) * dtype_bytes(p.c_dtype);
}

// Issue the loads of a 16-bit C[row, col0 .. col0+32) (no arithmetic: the
// values are used one chunk later, so the load latency hides behind that
// chunk's work).  TR: the 32 values sit one caller row apart; each load
// instruction of the warp still reads 32 consecutive elements.
template <bool TR = false>
__device__ __forceinline__ void load_c_chunk(const Params& p, int32_t row, int32_t col0,
                                             int32_t batch, CRegs& c) {
  if (p.c_dtype == DT_F32) return;
  if constexpr (TR) {
    const uint16_t* base = reinterpret_cast<const uint16_t*>(c_ptr<true>(p, row, col0, batch));
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t lo = (col0 + 2 * i < p.N) ? __ldg(base + (2 * i) * p.ldc) : 0u;
      const uint32_t hi = (col0 + 2 * i + 1 < p.N) ? __ldg(base + (2 * i + 1) * p.ldc) : 0u;
      w[i] = lo | (hi << 16);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) c.w[g] = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
  } else {
    const uint4* base = reinterpret_cast<const uint4*>(c_ptr(p, row, col0, batch));
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (col0 + 8 * i < p.N) c.w[i] = __ldg(base + i);
  }
}

// Eight values of C (group g of 8 columns of the chunk) as fp32: from the
// prefetched registers (16-bit C), or read now through `crow` (fp32 C; NULL
// for a row that does not exist).  CDT is C's dtype.
template <int CDT, bool TR>
__device__ __forceinline__ void c_values8(const CRegs& c, const Params& p, const char* crow,
                                          int32_t col0, int g, float (&out)[8]) {
  if constexpr (CDT == DT_F32 && TR) {
    // `crow` points at the caller's C[col0][row]: the chunk's columns are rows of C
    const float* cc = reinterpret_cast<const float*>(crow);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      out[i] = (cc != nullptr && col0 + 8 * g + i < p.N) ? __ldg(cc + (8 * g + i) * p.ldc) : 0.f;
  } else if constexpr (CDT == DT_F32) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (crow != nullptr && col0 + 8 * g < p.N) {
      a = __ldg(reinterpret_cast<const float4*>(crow) + 2 * g);
      b = __ldg(reinterpret_cast<const float4*>(crow) + 2 * g + 1);
    }
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
  } else {
    const uint32_t w[4] = {c.w[g].x, c.w[g].y, c.w[g].z, c.w[g].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f;
      if constexpr (CDT == DT_BF16)
        f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      else
        f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
}

// v += beta * C over the chunk (C's dtype chosen once, outside the value loops).
template <int CDT, bool TR>
__device__ __forceinline__ void add_beta_c_t(const CRegs& c, const Params& p, const char* crow,
                                             int32_t col0, float beta, float (&v)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float cv[8];
    c_values8<CDT, TR>(c, p, crow, col0, g, cv);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[8 * g + j] = fmaf(beta, cv[j], v[8 * g + j]);
  }
}

template <bool TR>
__device__ __forceinline__ void add_beta_c(const CRegs& c, const Params& p, const char* crow,
                                           int32_t col0, float beta, float (&v)[32]) {
  if (p.c_dtype == DT_F32) add_beta_c_t<DT_F32, TR>(c, p, crow, col0, beta, v);
  else if (p.c_dtype == DT_BF16) add_beta_c_t<DT_BF16, TR>(c, p, crow, col0, beta, v);
  else add_beta_c_t<DT_F16, TR>(c, p, crow, col0, beta, v);
}

// All 32 values of C as fp32 (the backward epilogue's pre-activation).
template <int CDT, bool TR>
__device__ __forceinline__ void c_values32_t(const CRegs& c, const Params& p, const char* crow,
                                             int32_t col0, float (&x)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float cv[8];
    c_values8<CDT, TR>(c, p, crow, col0, g, cv);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[8 * g + j] = cv[j];
  }
}

template <bool TR>
__device__ __forceinline__ void c_values32(const CRegs& c, const Params& p, const char* crow,
                                           int32_t col0, float (&x)[32]) {
  if (p.c_dtype == DT_F32) c_values32_t<DT_F32, TR>(c, p, crow, col0, x);
  else if (p.c_dtype == DT_BF16) c_values32_t<DT_BF16, TR>(c, p, crow, col0, x);
  else c_values32_t<DT_F16, TR>(c, p, crow, col0, x);
}

// Two fp32 values as one 32-bit word of a 16-bit output type (RNE).
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// A lane's 32 values as 16 words of the 16-bit output type, the type chosen once.
__device__ __forceinline__ void pack32(int dtype, const float (&x)[32], uint32_t (&w)[16]) {
  if (dtype == DT_BF16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack2<true>(x[2 * i], x[2 * i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack2<false>(x[2 * i], x[2 * i + 1]);
  }
}

// Write a warp's 32 x 32 output chunk (lane = row, x = its 32 columns) to global
// memory through the warp's shared-memory staging buffer, so that each store
// instruction writes whole row segments: 16-bit outputs 8 rows x 64 B, fp32
// 4 rows x 128 B (instead of 32 rows x 16 B).  The 16-byte pieces of a row are
// XOR-swizzled so that both the row-wise writes and the transposed reads are
// free of bank conflicts.  `out` points at (row 0, column 0) of the chunk;
// rows >= rows_valid and columns >= cols_valid are not written.  Warp-collective.
__device__ __forceinline__ void store_chunk_staged(uint32_t stg, const float (&x)[32], int dtype,
                                                   char* out, int64_t ld_bytes,
                                                   int32_t rows_valid, int32_t cols_valid,
                                                   bool direct) {
  const int lane = threadIdx.x & 31;
  if (direct) {
    // no staging buffer: each lane writes its own row (32 rows x 16 B per instruction)
    if (lane >= rows_valid) return;
    char* o = out + lane * ld_bytes;
    if (dtype == DT_F32) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (4 * q < cols_valid)
          *reinterpret_cast<uint4*>(o + 16 * q) =
              make_uint4(__float_as_uint(x[4 * q]), __float_as_uint(x[4 * q + 1]),
                         __float_as_uint(x[4 * q + 2]), __float_as_uint(x[4 * q + 3]));
    } else {
      uint32_t w[16];
      pack32(dtype, x, w);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (8 * q < cols_valid)
          *reinterpret_cast<uint4*>(o + 16 * q) =
              make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
    return;
  }
  if (dtype == DT_F32) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      ptx::st_shared_v4(stg + lane * 128 + ((q ^ (lane & 7)) << 4),
                        make_uint4(__float_as_uint(x[4 * q]), __float_as_uint(x[4 * q + 1]),
                                   __float_as_uint(x[4 * q + 2]), __float_as_uint(x[4 * q + 3])));
    __syncwarp();
    const int q = lane & 7;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = 4 * j + (lane >> 3);
      const uint4 v = ptx::ld_shared_v4(stg + r * 128 + ((q ^ (r & 7)) << 4));
      if (r < rows_valid && 4 * q < cols_valid)
        *reinterpret_cast<uint4*>(out + r * ld_bytes + 16 * q) = v;
    }
  } else {
    uint32_t w[16];
    pack32(dtype, x, w);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      ptx::st_shared_v4(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4),
                        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
    __syncwarp();
    const int q = lane & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 8 * j + (lane >> 2);
      const uint4 v = ptx::ld_shared_v4(stg + r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
      if (r < rows_valid && 8 * q < cols_valid)
        *reinterpret_cast<uint4*>(out + r * ld_bytes + 16 * q) = v;
    }
  }
  __syncwarp();  // the buffer is free again
}

// swap_ab: the caller's output holds the kernel's element (row, col) at
// [col][row], so a warp's chunk is 32 caller rows (the chunk's columns) of 32
// consecutive elements (its rows).  Each lane writes its 32 values down a
// column of the warp's staging buffer, then every store instruction writes
// whole 16-byte pieces of caller rows: 16-bit outputs 8 rows x 64 B, fp32 4 rows
// x 128 B, as in store_chunk_staged.  `out` points at the caller's [col0][row
// base]; rows_valid (a multiple of 8: the caller's N is) and cols_valid bound the
// chunk.  Warp-collective.
__device__ __forceinline__ void store_chunk_staged_t(uint32_t stg, const float (&x)[32], int dtype,
                                                     char* out, int64_t ld_bytes,
                                                     int32_t rows_valid, int32_t cols_valid,
                                                     bool direct) {
  const int lane = threadIdx.x & 31;
  if (direct) {
    // no staging buffer: each instruction writes one caller row's 32 elements
    if (lane >= rows_valid) return;
    if (dtype == DT_F32) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < cols_valid) *reinterpret_cast<float*>(out + j * ld_bytes + 4 * lane) = x[j];
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < cols_valid) {
          const uint32_t w = dtype == DT_BF16 ? pack2<true>(x[j], 0.f) : pack2<false>(x[j], 0.f);
          *reinterpret_cast<uint16_t*>(out + j * ld_bytes + 2 * lane) = static_cast<uint16_t>(w);
        }
    }
    return;
  }
  if (dtype == DT_F32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) ptx::st_shared_u32(stg + j * 128 + 4 * lane, __float_as_uint(x[j]));
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int pc = lane + 32 * it, j = pc >> 3, q = pc & 7;
      const uint4 v = ptx::ld_shared_v4(stg + j * 128 + 16 * q);
      if (j < cols_valid && 4 * q < rows_valid)
        *reinterpret_cast<uint4*>(out + j * ld_bytes + 16 * q) = v;
    }
  } else {
    if (dtype == DT_BF16) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        ptx::st_shared_u16(stg + j * 64 + 2 * lane, static_cast<uint16_t>(pack2<true>(x[j], 0.f)));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        ptx::st_shared_u16(stg + j * 64 + 2 * lane, static_cast<uint16_t>(pack2<false>(x[j], 0.f)));
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int pc = lane + 32 * it, j = pc >> 2, q = pc & 3;
      const uint4 v = ptx::ld_shared_v4(stg + j * 64 + 16 * q);
      if (j < cols_valid && 8 * q < rows_valid)
        *reinterpret_cast<uint4*>(out + j * ld_bytes + 16 * q) = v;
    }
  }
  __syncwarp();  // the buffer is free again
}

// Where a warp's chunk of an output starts: (row_base, col0) of batch `batch`
// (TR: the caller's [col0][row_base]).
template <bool TR = false>
__device__ __forceinline__ char* out_ptr(void* base, int64_t ld, int64_t sb, int dtype,
                                         int32_t row_base, int32_t col0, int32_t batch,
                                         const Params& p) {
  const int64_t out_batch = (p.num_groups > 0) ? 0 : batch;
  const int64_t off = TR ? static_cast<int64_t>(col0) * ld + row_base
                         : static_cast<int64_t>(row_base) * ld + col0;
  return static_cast<char*>(base) + (out_batch * sb + off) * dtype_bytes(dtype);
}

// One output chunk through the store of the layout (TR: swap_ab's transposed one).
template <bool TR>
__device__ __forceinline__ void store_out(const Params& p, uint32_t stg, const float (&x)[32],
                                          void* base, int64_t ld, int64_t sb, int dtype,
                                          int32_t row_base, int32_t rows_valid, int32_t col0,
                                          int32_t cols_valid, int32_t batch) {
  char* o = out_ptr<TR>(base, ld, sb, dtype, row_base, col0, batch, p);
  const int64_t ld_bytes = ld * dtype_bytes(dtype);
  if constexpr (TR)
    store_chunk_staged_t(stg, x, dtype, o, ld_bytes, rows_valid, cols_valid, p.out_stage_bytes == 0);
  else
    store_chunk_staged(stg, x, dtype, o, ld_bytes, rows_valid, cols_valid, p.out_stage_bytes == 0);
}

// Backward epilogue for one warp's 32 x 32 chunk: x (the pre-activation) comes
// from C, dout is the accumulator; D = act'(x) * dout, PostAct = act(x).
template <bool TR>
__device__ __forceinline__ void epilogue_chunk_dact(const Params& p, const uint32_t (&acc)[32],
                                                    int32_t row_base, int32_t rows_valid,
                                                    int32_t col0, int32_t batch,
                                                    const CRegs& creg, uint32_t stg) {
  const int32_t cols_valid = min(32, p.N - col0);
  const int lane = threadIdx.x & 31;
  const char* crow = (p.c_dtype == DT_F32 && lane < rows_valid)
                         ? c_ptr<TR>(p, row_base + lane, col0, batch) : nullptr;
  float x[32], y[32];
  c_values32<TR>(creg, p, crow, col0, x);
  dact_chunk(p.act, x, acc, y);
  store_out<TR>(p, stg, y, p.d, p.ldd, p.sbd, p.d_dtype, row_base, rows_valid, col0, cols_valid,
                batch);
  if (p.post != nullptr) {
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = x[j];
    act_chunk(p.act, y);
    store_out<TR>(p, stg, y, p.post, p.ldp, p.sbp, p.p_dtype, row_base, rows_valid, col0,
                  cols_valid, batch);
  }
}

// One warp's 32 x 32 chunk: rows row_base .. +31 (lane = row), columns col0 .. +31.
template <bool TR>
__device__ __forceinline__ void epilogue_chunk_t(const Params& p, const uint32_t (&acc)[32],
                                                 int32_t row_base, int32_t rows_valid,
                                                 int32_t col0, int32_t batch, float alpha,
                                                 float beta, const CRegs& creg, uint32_t stg) {
  if (p.dact) {
    epilogue_chunk_dact<TR>(p, acc, row_base, rows_valid, col0, batch, creg, stg);
    return;
  }
  const int32_t cols_valid = min(32, p.N - col0);
  float v[32];
  if (alpha == 1.f) {  // (x * 1 == x for every x, so skipping it changes no bit)
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(acc[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(acc[j]) * alpha;
  }
  if (p.c != nullptr) {
    const int lane = threadIdx.x & 31;
    const char* crow = (p.c_dtype == DT_F32 && lane < rows_valid)
                           ? c_ptr<TR>(p, row_base + lane, col0, batch) : nullptr;
    add_beta_c<TR>(creg, p, crow, col0, beta, v);
  }
  if (p.d != nullptr)
    store_out<TR>(p, stg, v, p.d, p.ldd, p.sbd, p.d_dtype, row_base, rows_valid, col0,
                  cols_valid, batch);
  if (p.post != nullptr) {
    act_chunk(p.act, v);
    store_out<TR>(p, stg, v, p.post, p.ldp, p.sbp, p.p_dtype, row_base, rows_valid, col0,
                  cols_valid, batch);
  }
}



// ------------------------------------------------------------------- roles
// `unit` / `units`: this CTA's (pair's) index and the number of CTAs (pairs).

// Split last wave, one epilogue warp's share of a tail tile (its 32 rows of the
// CTA's 128, its 32-column chunks): every slice's unit writes each raw fp32
// accumulator chunk to the workspace and then takes that chunk's ticket; the
// warp that takes a chunk's last ticket adds all slices' copies of it in slice
// order (so the sum does not depend on which unit came last) and runs its
// epilogue.  The slices walk their chunks in rotated orders, so different
// units come last for different chunks and share the final epilogue.  No warp
// waits for another unit, so the result does not depend on when (or in what
// order) the units run.  Partial chunk layout: float4 q of a lane's row in
// chunk c at [quad][c][q][lane], so each warp store / load moves 512
// contiguous bytes.
template <int BN, bool GATHER, int CG>
__device__ __forceinline__ float4* tail_chunk(const Params& p, int32_t tail_r, int32_t slice,
                                              uint32_t rank, int quad, int c, int lane) {
  constexpr int kChunks = BN / 32;
  const int64_t block = (static_cast<int64_t>(tail_r) * p.tail_splits + slice) * CG + rank;
  return reinterpret_cast<float4*>(p.partials + block * kBM * BN) + ((quad * kChunks + c) * 8) * 32 +
         lane;
}

// Writes this lane's 32 accumulator values of chunk c as the slice's partial.
__device__ __forceinline__ void tail_store(float4* dst, const uint32_t (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    dst[q * 32] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                              __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
}

// After the warp's partial chunk is written: count this slice in the chunk's
// ticket (per CTA, epilogue warp and chunk).  True (in every lane) for the warp
// whose slice came last, which then owns the chunk's outputs; it resets the
// ticket for the next launch.  The fence before the count publishes every lane's
// partial stores; the one after it orders the reads of the other slices'.
__device__ __forceinline__ bool tail_ticket(int32_t* ticket, int32_t splits) {
  __threadfence();
  __syncwarp();
  int32_t last = 0;
  if ((threadIdx.x & 31) == 0) {
    last = (atomicAdd(ticket, 1) == splits - 1) ? 1 : 0;
    if (last) atomicExch(ticket, 0);
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) __threadfence();
  return last != 0;
}

// The sum of every slice's partial of chunk c, in slice order (L2 reads: the
// other slices were written by other SMs during this launch).
template <int BN, bool GATHER, int CG>
__device__ __forceinline__ void tail_sum(const Params& p, int32_t tail_r, uint32_t rank, int quad,
                                         int c, int lane, uint32_t (&v)[32]) {
  float4 acc[8];
  const float4* src = tail_chunk<BN, GATHER, CG>(p, tail_r, 0, rank, quad, c, lane);
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = __ldcg(src + q * 32);
  for (int32_t sl = 1; sl < p.tail_splits; ++sl) {
    src = tail_chunk<BN, GATHER, CG>(p, tail_r, sl, rank, quad, c, lane);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 a = __ldcg(src + q * 32);
      acc[q].x += a.x;
      acc[q].y += a.y;
      acc[q].z += a.z;
      acc[q].w += a.w;
    }
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    v[4 * q] = __float_as_uint(acc[q].x);
    v[4 * q + 1] = __float_as_uint(acc[q].y);
    v[4 * q + 2] = __float_as_uint(acc[q].z);
    v[4 * q + 3] = __float_as_uint(acc[q].w);
  }
}

// Eight epilogue warps (four in the gather form), two per TMEM lane quadrant
// (warp w reads lanes 32*(w%4) .. +31); warp w takes the 32-column chunks c
// with c % 2 == w / 4, so two independent dependency chains per quadrant hide
// the TMEM-load and memory latencies.  C for the next chunk is loaded one chunk ahead (the
// first before the accumulator is ready).  TR: swap_ab's transposed output layout
// (a separate kernel instance, so that the usual one carries none of its code).
template <int BN, bool GATHER, int CG, bool TR>
__device__ __forceinline__ void epilogue_role(const Params& p, const Shared& sh,
                                              uint32_t tmem_base, int32_t num_tiles,
                                              uint32_t rank, const TileSched& ts,
                                              uint32_t stg) {
  using Cfg = KernelCfg<BN, GATHER, CG>;
  constexpr int kChunks = BN / 32;
  constexpr int kStride = Cfg::kEpiWarps / 4;  // warps per TMEM lane quadrant
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3, half = warp >> 2;
  const float alpha = p.alpha_dev ? *p.alpha_dev : p.alpha;
  const float beta = p.beta_dev ? *p.beta_dev : p.beta;
  uint32_t acc = 0, acc_phase = 0;
  for (int i = 0;; ++i) {
    const int32_t t = sched_next<CG>(ts, i, p, sh);
    if (t >= num_tiles) break;
    const TileCoord tc = tile_coord<BN, Cfg::kTileM>(t, p, sh);
    // a tile with no k-tiles (K == 0, or an empty varlen-K group) keeps a zero accumulator
    const bool has_acc = k_range(p, sh, tc.batch, t).tiles > 0;
    // split tail item (the gather forms never split: compiled out of their instances)
    const bool split = !GATHER && p.tail_tiles > 0 && t >= p.full_tiles;
    int32_t slice = 0, tail_r = 0;
    if (split) {
      tail_r = (t - p.full_tiles) / p.tail_splits;
      slice = t - p.full_tiles - tail_r * p.tail_splits;
    }
    const int32_t row_base = tc.m_row0 + static_cast<int32_t>(rank) * kBM + quad * 32;
    const int32_t rows_valid = min(32, tc.row_limit - row_base);  // warp-uniform, may be <= 0
    const int32_t row = row_base + lane;
    const bool has_c = p.c != nullptr && lane < rows_valid;
    // D only (no C, no PostAct, forward, 16-bit D, staged): each chunk goes straight
    // to the staging store, without the general epilogue's per-chunk decisions
    const bool lean = !TR && !p.dact && p.c == nullptr && p.post == nullptr &&
                      p.out_stage_bytes != 0 && p.d_dtype != DT_F32;
    CRegs cnext = {};
    if (!split && has_c && tc.n0 + half * 32 < p.N)
      load_c_chunk<TR>(p, row, tc.n0 + half * 32, tc.batch, cnext);
    // all lanes take the same branch: tcgen05.ld below is warp-collective
    const bool ok = wait_phase<CG == 2, true>(sh.tfull + 8 * acc, acc_phase, p, sh, 3, t);
    if (!__all_sync(0xffffffffu, ok)) break;
    ptx::tc_fence_after();
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
    // this warp's chunks are half, half + kStride, ...; a split item's slice s walks
    // them rotated by s * n / S, so that the S slices of a tile finish different
    // chunks last and share the tile's final epilogue between their units
    constexpr int kMine = (kChunks + kStride - 1) / kStride;
    const int shift = split ? static_cast<int>((slice * kMine) / p.tail_splits) : 0;
    // the last iteration that reads TMEM (a warp of a quadrant with one chunk fewer
    // skips one index, which is the last only without rotation)
    const int last_ci = (kMine - 1 + shift) % kMine;
    const int last_i = (half + last_ci * kStride >= kChunks) ? kMine - 2 : kMine - 1;
    bool finished = !split;
#pragma unroll 1
    for (int i = 0; i < kMine; ++i) {
      const int ci = (i + shift < kMine) ? i + shift : i + shift - kMine;
      const int c = half + ci * kStride;
      if (c >= kChunks) continue;  // (kChunks odd: the second warp of a quadrant has one fewer)
      const CRegs ccur = cnext;
      if (!split && has_c && c + kStride < kChunks && tc.n0 + (c + kStride) * 32 < p.N)
        load_c_chunk<TR>(p, row, tc.n0 + (c + kStride) * 32, tc.batch, cnext);
      uint32_t v[32];
      __syncwarp();  // tcgen05.ld / wait::ld are warp-collective
      if (has_acc) {
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, v);
        ptx::tmem_wait_ld(v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
      if (i == last_i) {
        // this warp's last TMEM read of the tile: hand its share of the buffer back
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CG == 1) ptx::mbar_arrive(sh.tempty + 8 * acc);
          else ptx::mbar_arrive_remote(ptx::mapa(sh.tempty + 8 * acc, 0));
        }
      }
      const int32_t col0 = tc.n0 + c * 32;
      if (split) {
        // the slice's raw accumulator chunk (this lane's 32 values), then its ticket;
        // the warp whose slice comes last for this chunk adds all slices and stores it
        tail_store(tail_chunk<BN, GATHER, CG>(p, tail_r, slice, rank, quad, c, lane), v);
        int32_t* ticket = p.tail_tickets +
                          ((static_cast<int64_t>(tail_r) * CG + rank) * Cfg::kEpiWarps + warp) *
                              kTicketsPerWarp + ci;
        if (tail_ticket(ticket, p.tail_splits)) {
          if (ci == 0) finished = true;
          // (a split item prefetches no C: cnext is free for this chunk's C)
          if (has_c && col0 < p.N) load_c_chunk<TR>(p, row, col0, tc.batch, cnext);
          tail_sum<BN, GATHER, CG>(p, tail_r, rank, quad, c, lane, v);
          if (rows_valid > 0 && col0 < p.N)
            epilogue_chunk_t<TR>(p, v, row_base, rows_valid, col0, tc.batch, alpha, beta, cnext,
                                 stg);
        }
        continue;
      }
      if (rows_valid > 0 && col0 < p.N) {
        if (lean) {
          float x[32];
          if (alpha == 1.f) {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]) * alpha;
          }
          store_chunk_staged(stg, x, p.d_dtype,
                             out_ptr(p.d, p.ldd, p.sbd, p.d_dtype, row_base, col0, tc.batch, p),
                             2 * p.ldd, rows_valid, min(32, p.N - col0), false);
        } else {
          epilogue_chunk_t<TR>(p, v, row_base, rows_valid, col0, tc.batch, alpha, beta, ccur,
                               stg);
        }
      }
    }
    if ((p.flags & FLAG_TILE_COUNTS) && p.tile_counts != nullptr && rank == 0 && warp == 0 &&
        lane == 0 && finished)
      atomicAdd(p.tile_counts + (split ? p.full_tiles + tail_r : t), 1);
    acc ^= 1u;
    if (acc == 0) acc_phase ^= 1u;
  }
}

// The whole MMA warp walks the loop (so descriptors stay warp-uniform); one
// elected lane issues the MMAs and commits.  The operand kind (f16 / f8) is a
// template parameter, fixed before the loop: chosen inside it, both MMA forms
// stayed in the issue stream (one predicated off), which doubled the tensor-pipe
// instructions per MMA and measured 11 % slower on an 8192^3 bf16 problem.
template <int BN, bool GATHER, int CG, bool F8>
__device__ __forceinline__ void mma_loop(const Params& p, const Shared& sh, uint32_t a0,
                                         uint32_t b0, uint32_t tmem_base, int32_t num_tiles,
                                         const TileSched& ts) {
  using Cfg = KernelCfg<BN, GATHER, CG>;
  int stage = 0;
  uint32_t phase = 0, acc = 0, acc_phase = 0;
  // Descriptor strides: K-major rows are 128 B apart, 8-row swizzle atoms 1 KiB apart;
  // M- / N-major: 64-element chunks are (bk rows * 128 B) apart, 8-row K groups 1 KiB
  // apart, and one MMA's 16 K rows span 2 KiB.
  const uint32_t a_lbo = p.a_mn_major ? static_cast<uint32_t>(p.bk) * kRowBytes : 16u;
  const uint32_t a_kstep = p.a_mn_major ? 16u * kRowBytes : 32u;
  const uint32_t b_lbo = p.b_mn_major ? static_cast<uint32_t>(p.bk) * kRowBytes : 16u;
  const uint32_t b_kstep = p.b_mn_major ? 16u * kRowBytes : 32u;
  for (int i = 0;; ++i) {
    const int32_t t = sched_next<CG>(ts, i, p, sh);
    if (t >= num_tiles) break;
    bool ok = wait_phase<CG == 2>(sh.tempty + 8 * acc, acc_phase ^ 1u, p, sh, 2, t);
    if (!__all_sync(0xffffffffu, ok)) return;
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * BN;
    const KRange kr = (p.k_groups > 0 || p.tail_tiles > 0)
                          ? k_range(p, sh, tile_coord<BN, Cfg::kTileM>(t, p, sh).batch, t)
                          : KRange{0, p.K, p.k_tiles, false};
    const bool rev = !GATHER && k_reversed(p, t, ts.units);
    for (int kt = 0; kt < kr.tiles; ++kt) {
      const int32_t kte = rev ? kr.tiles - 1 - kt : kt;  // the k-tile this stage holds
      ok = wait_phase<CG == 2>(sh.full + 8 * stage, phase, p, sh, 1, t);
      if (!__all_sync(0xffffffffu, ok)) return;
      ptx::tc_fence_after();
      if (GATHER) ptx::fence_proxy_async_smem();  // cp.async (generic proxy) writes -> MMA reads
      const uint32_t a_addr = a0 + stage * Cfg::kABytes;
      const uint32_t b_addr = b0 + stage * Cfg::kBBytes;
      const int32_t nk = (kte == kr.tiles - 1) ? ksteps_of(p, kr, kte) : 4;
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // up to 4 MMAs of 32 bytes of K each
          if (kk >= nk) break;
          const uint64_t adesc = smem_desc(a_addr + kk * a_kstep, a_lbo, 1024u);
          const uint64_t bdesc = smem_desc(b_addr + kk * b_kstep, b_lbo, 1024u);
          const uint32_t accumulate = (kt > 0 || kk > 0) ? 1u : 0u;
          if constexpr (CG == 1) {
            if constexpr (F8) ptx::mma_f8(d_tmem, adesc, bdesc, p.idesc, accumulate);
            else ptx::mma_f16(d_tmem, adesc, bdesc, p.idesc, accumulate);
          } else {
            if constexpr (F8) ptx::mma_f8_pair(d_tmem, adesc, bdesc, p.idesc, accumulate);
            else ptx::mma_f16_pair(d_tmem, adesc, bdesc, p.idesc, accumulate);
          }
        }
        // frees the stage (in both CTAs of a pair) once these MMAs finish
        if (CG == 1) ptx::mma_commit(sh.empty + 8 * stage);
        else ptx::mma_commit_pair(sh.empty + 8 * stage, 0x3);
      }
      __syncwarp();
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
    if (!(p.flags & FLAG_TEST_DROP_ACC_FULL) && ptx::elect_one()) {
      if (CG == 1) ptx::mma_commit(sh.tfull + 8 * acc);
      else ptx::mma_commit_pair(sh.tfull + 8 * acc, 0x3);
    }
    __syncwarp();
    acc ^= 1u;
    if (acc == 0) acc_phase ^= 1u;
  }
}

template <int BN, bool GATHER, int CG>
__device__ __forceinline__ void mma_role(const Params& p, const Shared& sh, uint32_t a0,
                                         uint32_t b0, uint32_t tmem_base, int32_t num_tiles,
                                         const TileSched& ts) {
  if (p.f8) mma_loop<BN, GATHER, CG, true>(p, sh, a0, b0, tmem_base, num_tiles, ts);
  else mma_loop<BN, GATHER, CG, false>(p, sh, a0, b0, tmem_base, num_tiles, ts);
}

// One TMA box into this CTA's shared memory; a pair's copies signal the leader's barrier.
template <int CG>
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                         int32_t x, int32_t y, int32_t z) {
  if (CG == 1) ptx::tma_load_3d(dst, m, bar, x, y, z);
  else ptx::tma_load_3d_pair(dst, m, bar, x, y, z);
}

// This CTA's tensor-map slot `slot` in the workspace.
__device__ __forceinline__ uint8_t* kmap_slot(const Params& p, int slot) {
  return p.kmaps + (static_cast<int64_t>(blockIdx.x) * kMapSlots + slot) * kMapSlotBytes;
}

// Varlen-K: write a copy of the A and B tensor maps whose K extent ends at the
// group's last column into this CTA's map slot `slot` (the pages'
// update_tensormap_shape), so that the group's last k-tile reads zeros past
// its end instead of the next group's columns.  Warp-collective.
__device__ __forceinline__ const uint8_t* publish_kmaps(const Params& p, const CUtensorMap* tmA,
                                                        const CUtensorMap* tmB, uint32_t scratch,
                                                        int slot, int32_t k_end) {
  const int lane = threadIdx.x & 31;
  uint8_t* dst = kmap_slot(p, slot);
  ptx::st_shared_u32(scratch + 4 * lane, reinterpret_cast<const uint32_t*>(tmA)[lane]);
  ptx::st_shared_u32(scratch + 128 + 4 * lane, reinterpret_cast<const uint32_t*>(tmB)[lane]);
  __syncwarp();
  if (lane == 0) {
    // K is dimension 0 of a K-major map and dimension 1 of an M- / N-major one
    if (p.a_mn_major) ptx::tmap_set_global_dim<1>(scratch, k_end);
    else ptx::tmap_set_global_dim<0>(scratch, k_end);
    if (p.b_mn_major) ptx::tmap_set_global_dim<1>(scratch + 128, k_end);
    else ptx::tmap_set_global_dim<0>(scratch + 128, k_end);
  }
  __syncwarp();
  ptx::tmap_publish(dst, scratch);
  ptx::tmap_publish(dst + 128, scratch + 128);
  ptx::tmap_acquire(dst);
  ptx::tmap_acquire(dst + 128);
  return dst;
}

// The whole producer warp walks the loop; one elected lane issues the copies.
template <int BN, bool GATHER, int CG>
__device__ __forceinline__ void tma_producer_role(const Params& p, const Shared& sh,
                                                  const CUtensorMap* tmA, const CUtensorMap* tmB,
                                                  uint32_t a0, uint32_t b0, uint32_t map_scratch,
                                                  int32_t num_tiles, uint32_t rank,
                                                  const TileSched& ts) {
  using Cfg = KernelCfg<BN, GATHER, CG>;
  int stage = 0;
  uint32_t phase = 0;
  // varlen-K: the group whose maps are in use, and the slot they occupy
  int32_t map_group = -1;
  uint32_t maps_used = 0;
  const uint8_t* map_cur = nullptr;
  const bool map_helper = !ts.dyn;  // the map warp walks the static schedule only
  const CUtensorMap* mA = tmA;
  const CUtensorMap* mB = tmB;
  for (int i = 0;; ++i) {
    // the producer fetches the tile stream (the peer CTA of a pair reads it)
    const int32_t t =
        (rank == 0) ? sched_fetch<CG>(ts, i, p, sh, num_tiles) : sched_next<CG>(ts, i, p, sh);
    if (t >= num_tiles) break;
    const TileCoord tc = tile_coord<BN, Cfg::kTileM>(t, p, sh);
    const KRange kr = k_range(p, sh, tc.batch, t);
    const int32_t row0 = tc.m_row0 + static_cast<int32_t>(rank) * kBM;
    const int32_t bn0 = tc.n0 + static_cast<int32_t>(rank) * Cfg::kBRows;
    const bool rev = k_reversed(p, t, ts.units);
    for (int kt = 0; kt < kr.tiles; ++kt) {
      const bool ok = wait_phase<CG == 2>(sh.empty + 8 * stage, phase ^ 1u, p, sh, 0, t);
      if (!__all_sync(0xffffffffu, ok)) return;
      if (kt == 0) {
        if (kr.ragged && tc.batch != map_group) {
          // The w-th ragged group reads slot w % kMapSlots.  A slot is rewritten only
          // after the group `stages` later has passed the wait above: every ragged
          // group issues at least one k-tile, and that wait has seen the k-tile
          // `stages` back consumed, so no copy still reads the old maps.
          const int slot = static_cast<int>(maps_used % kMapSlots);
          if (map_helper) {
            // the map warp wrote this slot ahead of time
            const uint32_t par = (maps_used / kMapSlots) & 1u;
            if (!__all_sync(0xffffffffu, wait_phase(sh.map_full + 8 * slot, par, p, sh, 10, t)))
              return;
            map_cur = kmap_slot(p, slot);
            ptx::tmap_acquire(map_cur);
            ptx::tmap_acquire(map_cur + 128);
            if (maps_used >= static_cast<uint32_t>(p.stages) && ptx::elect_one())
              ptx::mbar_arrive(sh.map_empty + 8 * ((maps_used - p.stages) % kMapSlots));
            __syncwarp();
          } else {
            map_cur = publish_kmaps(p, tmA, tmB, map_scratch, slot, kr.k_end);
          }
          ++maps_used;
          map_group = tc.batch;
        }
        // a ragged group reads through its clipped maps; any other range is cut by
        // the MMA K-step count, so the launch's maps serve it
        mA = kr.ragged ? reinterpret_cast<const CUtensorMap*>(map_cur) : tmA;
        mB = kr.ragged ? reinterpret_cast<const CUtensorMap*>(map_cur + 128) : tmB;
      }
      const uint32_t full = sh.full + 8 * stage;
      const int32_t k0 = kr.k0 + (rev ? kr.tiles - 1 - kt : kt) * p.bk;
      const uint32_t adst = a0 + stage * Cfg::kABytes;
      const uint32_t bdst = b0 + stage * Cfg::kBBytes;
      if (ptx::elect_one()) {
        // both CTAs' bytes of a pair complete on the leader's barrier, which the leader arms
        if (CG == 1) ptx::mbar_arrive_expect_tx(full, Cfg::kStageBytes);
        else if (rank == 0) ptx::mbar_arrive_expect_tx(full, 2 * Cfg::kStageBytes);
        const uint32_t bar = (CG == 1) ? full : ptx::mapa(full, 0);
        // K-major operands: one box of (bk columns, rows); M- / N-major: 64-wide boxes of bk rows
        if (!p.a_mn_major) {
          tma_load<CG>(adst, mA, bar, k0, row0, tc.a_batch);
        } else {
#pragma unroll
          for (int j = 0; j < kBM / 64; ++j)
            tma_load<CG>(adst + j * (64 * kRowBytes), mA, bar, row0 + 64 * j, k0, tc.a_batch);
        }
        if (!p.b_mn_major) {
          tma_load<CG>(bdst, mB, bar, k0, bn0, tc.b_batch);
        } else {
#pragma unroll
          for (int j = 0; j < Cfg::kBRows / 64; ++j)
            tma_load<CG>(bdst + j * (64 * kRowBytes), mB, bar, bn0 + 64 * j, k0, tc.b_batch);
        }
      }
      __syncwarp();
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
}

// Varlen-K with the static schedule: walk this CTA's tiles ahead of the
// producer and write the clipped tensor maps of each ragged group into the
// next slot, so that the fences of the rewrite stay off the producer's path.
// It may run kMapSlots - stages groups ahead; the producer hands each slot back.
template <int BN, int CG>
__device__ __forceinline__ void map_warp_role(const Params& p, const Shared& sh,
                                              const CUtensorMap* tmA, const CUtensorMap* tmB,
                                              uint32_t scratch, int32_t num_tiles,
                                              const TileSched& ts) {
  using Cfg = KernelCfg<BN, false, CG>;
  if (p.k_groups == 0 || ts.dyn) return;
  int32_t last = -1;
  uint32_t n = 0;
  for (int i = 0;; ++i) {
    const int32_t t = ts.unit + i * ts.units;
    if (t >= num_tiles) break;
    const TileCoord tc = tile_coord<BN, Cfg::kTileM>(t, p, sh);
    const KRange kr = k_range(p, sh, tc.batch, t);
    if (!kr.ragged || tc.batch == last) continue;
    const int slot = static_cast<int>(n % kMapSlots);
    if (n >= static_cast<uint32_t>(kMapSlots)) {
      const uint32_t par = ((n / kMapSlots) - 1u) & 1u;
      if (!__all_sync(0xffffffffu, wait_phase(sh.map_empty + 8 * slot, par, p, sh, 9, t))) return;
    }
    publish_kmaps(p, tmA, tmB, scratch, slot, kr.k_end);
    __syncwarp();
    if (ptx::elect_one()) ptx::mbar_arrive(sh.map_full + 8 * slot);
    __syncwarp();
    last = tc.batch;
    ++n;
  }
}

// B of a one-CTA tile by TMA: one box (K-major) or BN/64 boxes of 64 columns (N-major).
template <int BN>
__device__ __forceinline__ void load_b_1cta(const Params& p, const CUtensorMap* tmB, uint32_t dst,
                                            uint32_t bar, int32_t k0, int32_t n0, int32_t batch) {
  if (!p.b_mn_major) {
    ptx::tma_load_3d(dst, tmB, bar, k0, n0, batch);
  } else {
#pragma unroll
    for (int j = 0; j < BN / 64; ++j)
      ptx::tma_load_3d(dst + j * (64 * kRowBytes), tmB, bar, n0 + 64 * j, k0, batch);
  }
}

// B of a one-CTA tile by 16-byte cp.async that reads nothing at or past column
// k_end (the rest of each copy is zero-filled): a ragged varlen-K group's last
// k-tile without a clipped tensor map.  Same swizzled layouts as the TMA boxes.
// kGatherThreads threads; gt = this thread's index among them.
template <int BN>
__device__ __forceinline__ void copy_b_clipped(const Params& p, uint32_t dst, int32_t kbase,
                                               int32_t k_end, int32_t n0, int gt) {
  constexpr int kStep = kGatherThreads / 8;  // rows between a thread's copies
  const int q = gt & 7;  // 16-byte piece of a 128-byte row
  const int sub = gt >> 3;
  if (!p.b_mn_major) {
    // rows n hold 64 K elements; piece q holds K elements kbase + 8q .. +7
    const int32_t kel = kbase + 8 * q;
    const int32_t kbytes = max(0, min(16, 2 * (k_end - kel)));
#pragma unroll
    for (int i = 0; i < BN / kStep; ++i) {
      const int n = sub + kStep * i;
      const uint32_t bytes = (n0 + n < p.N) ? static_cast<uint32_t>(kbytes) : 0u;
      const uint8_t* src =
          bytes ? p.b_src + static_cast<int64_t>(n0 + n) * p.b_ld + 2 * static_cast<int64_t>(kel)
                : p.b_src;
      ptx::cp_async_16(dst + n * kRowBytes + ((q ^ (n & 7)) << 4), src, bytes);
    }
  } else {
    // 64-column chunks of bk K rows; piece q holds columns 8q .. 8q+7 of the chunk
#pragma unroll
    for (int j = 0; j < BN / 64; ++j) {
#pragma unroll
      for (int i = 0; i < 64 / kStep; ++i) {
        const int k = sub + kStep * i;
        const int32_t nel = n0 + 64 * j + 8 * q;
        const uint32_t bytes = (kbase + k < k_end && nel < p.N) ? 16u : 0u;
        const uint8_t* src =
            bytes ? p.b_src + static_cast<int64_t>(kbase + k) * p.b_ld + 2 * static_cast<int64_t>(nel)
                  : p.b_src;
        ptx::cp_async_16(dst + j * (64 * kRowBytes) + k * kRowBytes + ((q ^ (k & 7)) << 4), src,
                         bytes);
      }
    }
  }
}

static_assert(kGatherThreads == 128, "gather-K: 16 threads per K row, 8 rows per thread");
static_assert(kIdxChunk % kGatherThreads == 0 && (kIdxChunk / 64 & (kIdxChunk / 64 - 1)) == 0,
              "gather-K index chunks: whole passes of the gather threads, a power of two of k-tiles");

// Stages into this warp's index buffer the source rows of the K rows it copies
// (rows 2w + r + 8j, r < 2, j < 8, of each k-tile; w = this gather warp) for the
// kIdxChunk / 64 k-tiles from K row kbase0 on, at entry 16 * k-tile + 8 r + j.
// Rows at or past k_end get -1 (zeros); an index out of range (or negative) too,
// and it is recorded.  Loading the indices per k-tile instead left every k-tile
// waiting for loads queued behind the gather copies (half the producer's time).
__device__ __forceinline__ void stage_k_indices(const Params& p, int32_t* idxw, int32_t kbase0,
                                                int32_t k_end, int w, int lane, int32_t tile) {
  constexpr int kPer = kIdxChunk / kGatherThreads;  // entries per lane
  int32_t v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    const int32_t kg = kbase0 + (e >> 4) * 64 + 2 * w + ((e >> 3) & 1) + 8 * (e & 7);
    v[i] = (kg < k_end) ? __ldg(p.a_idx + kg) : -1;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    const int32_t kg = kbase0 + (e >> 4) * 64 + 2 * w + ((e >> 3) & 1) + 8 * (e & 7);
    if (kg < k_end && (v[i] < 0 || v[i] >= p.a_src_rows)) {
      record_status(p, DEV_INDEX_RANGE, 4, tile);
      v[i] = -1;
    }
    idxw[e] = v[i];
  }
}

// Gather-K (varlen-K with A gathered along K, the pages' gather_k copy): row k
// of the k-tile's effective A^T is row a_idx[k] of the source X (M contiguous
// 16-bit elements), staged M-major: 64-element chunks of bk K rows, 128-byte
// swizzle.  Thread gt copies 16-byte piece gt % 16 of the tile's 256-byte M
// segment for K rows gt / 16 + 8 i; the indices come from shared memory,
// staged kIdxChunk at a time.
// B comes by TMA, except the last k-tile of a ragged group, copied only up to
// the group's end.  A K row past the group's end, an M element past M, or an
// index out of range reads zeros (the last is reported).
template <int BN>
__device__ __forceinline__ void gather_k_producer_role(const Params& p, const Shared& sh,
                                                       const CUtensorMap* tmB, uint32_t a0,
                                                       uint32_t b0, int32_t num_tiles,
                                                       const TileSched& ts) {
  using Cfg = KernelCfg<BN, true, 1>;
  const int gt = threadIdx.x - Cfg::kLoadWarp * 32;  // 0..127
  const int q = gt & 15;
  const int ksub = gt >> 4;
  const uint32_t a_off = static_cast<uint32_t>(q >> 3) * (64 * kRowBytes);  // M chunk
  const int gw = gt >> 5, lane = gt & 31;
  int32_t* idxw = sh.idx + gw * (kIdxChunk / kGatherWarps);  // this warp's index buffer
  // this thread's eight rows of a k-tile: 32 contiguous bytes, 64 bytes per k-tile
  const uint32_t my_idx = ptx::smem_addr(idxw + (lane >> 4) * 8);
  int stage = 0;
  uint32_t phase = 0;
  for (int i = 0;; ++i) {
    const int32_t t = (gt < 32) ? sched_fetch<1>(ts, i, p, sh, num_tiles) : sched_next<1>(ts, i, p, sh);
    if (t >= num_tiles) break;
    const TileCoord tc = tile_coord<BN, kBM>(t, p, sh);
    const KRange kr = k_range(p, sh, tc.batch, t);
    const int32_t m_el = tc.m_row0 + 8 * q;
    const bool m_ok = m_el < p.M;  // M is a multiple of 8: whole pieces
    constexpr int kChunkTiles = kIdxChunk / 64;
    for (int kt = 0; kt < kr.tiles; ++kt) {
      if ((kt & (kChunkTiles - 1)) == 0) {
        __syncwarp();  // the warp is done with the previous chunk
        stage_k_indices(p, idxw, kr.k0 + kt * 64, kr.k_end, gw, lane, t);
        __syncwarp();
      }
      const bool ok = wait_phase(sh.empty + 8 * stage, phase ^ 1u, p, sh, 0, t);
      if (!__all_sync(0xffffffffu, ok)) return;
      const uint32_t full = sh.full + 8 * stage;
      const int32_t kbase = kr.k0 + kt * p.bk;
      const uint32_t abase = a0 + stage * Cfg::kABytes;
      const uint32_t bbase = b0 + stage * Cfg::kBBytes;
      // B by TMA, except the last k-tile of a ragged group: there by copies that stop
      // at the group's end (the K-step count cuts every other range exactly)
      if (!(kr.ragged && kt == kr.tiles - 1)) {
        if (gt < 32 && ptx::elect_one()) {
          ptx::mbar_arrive_expect_tx(full, Cfg::kBBytes);
          load_b_1cta<BN>(p, tmB, bbase, full, kbase, tc.n0, 0);
        }
      } else {
        if (gt < 32 && ptx::elect_one()) ptx::mbar_arrive(full);
        copy_b_clipped<BN>(p, bbase, kbase, kr.k_end, tc.n0, gt);
      }
      // the k-tile's eight source rows in two vector loads, all read before the first
      // copy (read one by one between the copies, their latencies added up: ~1,200
      // cycles per k-tile)
      const uint32_t ia = my_idx + static_cast<uint32_t>(kt & (kChunkTiles - 1)) * 64u;
      const uint4 lo = ptx::ld_shared_v4(ia), hi = ptx::ld_shared_v4(ia + 16);
      const int32_t rows[8] = {static_cast<int32_t>(lo.x), static_cast<int32_t>(lo.y),
                               static_cast<int32_t>(lo.z), static_cast<int32_t>(lo.w),
                               static_cast<int32_t>(hi.x), static_cast<int32_t>(hi.y),
                               static_cast<int32_t>(hi.z), static_cast<int32_t>(hi.w)};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = ksub + 8 * j;
        // K rows past the group's end (and M pieces past M) read zeros
        const int32_t src = m_ok ? rows[j] : -1;
        const uint8_t* sp =
            src >= 0 ? p.a_src + static_cast<int64_t>(src) * p.a_src_ld + 2 * static_cast<int64_t>(m_el)
                     : p.a_src;
        ptx::cp_async_16(abase + a_off + k * kRowBytes + (((q & 7) ^ (k & 7)) << 4), sp,
                         src >= 0 ? 16u : 0u);
      }
      ptx::cp_async_mbar_arrive_noinc(full);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
}

// This CTA's rows of B for one k-tile by TMA, completing on the stage's barrier
// (the leader's, for a CTA pair: the leader arms it for both halves).  One lane.
template <int BN, int CG>
__device__ __forceinline__ void load_b_stage(const Params& p, const CUtensorMap* tmB, uint32_t dst,
                                             uint32_t full, uint32_t rank, int32_t k0, int32_t n0,
                                             int32_t batch) {
  using Cfg = KernelCfg<BN, true, CG>;
  if (CG == 1) {
    ptx::mbar_arrive_expect_tx(full, Cfg::kBBytes);
    load_b_1cta<BN>(p, tmB, dst, full, k0, n0, batch);
    return;
  }
  // both halves of B, and the 4 bytes the peer's relay stores when its rows are in
  if (rank == 0) ptx::mbar_arrive_expect_tx(full, 2 * Cfg::kBBytes + 4);
  const uint32_t bar = ptx::mapa(full, 0);
  const int32_t bn0 = n0 + static_cast<int32_t>(rank) * Cfg::kBRows;
  if (!p.b_mn_major) {
    ptx::tma_load_3d_pair(dst, tmB, bar, k0, bn0, batch);
  } else {
#pragma unroll
    for (int j = 0; j < Cfg::kBRows / 64; ++j)
      ptx::tma_load_3d_pair(dst + j * (64 * kRowBytes), tmB, bar, bn0 + 64 * j, k0, batch);
  }
}

// Four warps: 8 threads per 128-byte A row, 16 rows per pass, 8 passes.  On a
// CTA pair each CTA gathers its own 128 rows of the 256-row tile and loads its
// half of B; the copies land in this CTA's shared memory and arrive on its own
// stage barrier (the peer's are relayed to the leader by relay_role).
template <int BN, int CG>
__device__ __forceinline__ void gather_producer_role(const Params& p, const Shared& sh,
                                                     const CUtensorMap* tmB, uint32_t a0,
                                                     uint32_t b0, int32_t num_tiles,
                                                     uint32_t rank, const TileSched& ts) {
  using Cfg = KernelCfg<BN, true, CG>;
  if constexpr (CG == 1) {
    if (p.k_groups > 0) {
      gather_k_producer_role<BN>(p, sh, tmB, a0, b0, num_tiles, ts);
      return;
    }
  }
  constexpr int kRows = kBM * 8 / kGatherThreads;  // rows per thread (8 threads a row)
  const int gt = threadIdx.x - Cfg::kLoadWarp * 32;  // 0 .. kGatherThreads-1
  const int chunk = gt & 7;
  const int rsub = gt >> 3;
  constexpr int kRowStep = kGatherThreads / 8;
  int stage = 0;
  uint32_t phase = 0;
  for (int i = 0;; ++i) {
    // the first gather warp (of the leader) fetches the tile stream, the others read it
    const int32_t t = (gt < 32 && rank == 0) ? sched_fetch<CG>(ts, i, p, sh, num_tiles)
                                             : sched_next<CG>(ts, i, p, sh);
    if (t >= num_tiles) break;
    const TileCoord tc = tile_coord<BN, Cfg::kTileM>(t, p, sh);
    // index rows: plain gather reads a_idx[batch][row], varlen reads a_idx[global row]
    const int64_t idx_base = (p.num_groups > 0) ? 0 : static_cast<int64_t>(tc.batch) * p.M;
    const int32_t row0 = tc.m_row0 + static_cast<int32_t>(rank) * kBM;
    int32_t src[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int32_t r = row0 + rsub + kRowStep * i;
      int32_t s = -1;
      if (r < tc.row_limit) {
        s = __ldg(p.a_idx + idx_base + r);
        if (s < 0 || s >= p.a_src_rows) {
          record_status(p, DEV_INDEX_RANGE, 4, t);
          s = -1;  // the row is zero-filled instead of read
        }
      }
      src[i] = s;
    }
    for (int kt = 0; kt < p.k_tiles; ++kt) {
      if (!wait_phase<CG == 2>(sh.empty + 8 * stage, phase ^ 1u, p, sh, 0, t)) return;
      const uint32_t full = sh.full + 8 * stage;
      if (gt < 32 && ptx::elect_one())  // one lane of the first gather warp: B by TMA
        load_b_stage<BN, CG>(p, tmB, b0 + stage * Cfg::kBBytes, full, rank, kt * p.bk, tc.n0,
                             tc.b_batch);
      const int32_t kbyte = kt * kRowBytes + chunk * 16;
      const uint32_t kvalid = (kbyte < p.k_bytes) ? 16u : 0u;
      const uint32_t abase = a0 + stage * Cfg::kABytes;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const int r = rsub + kRowStep * i;
        const uint32_t dst = abase + r * kRowBytes + ((chunk ^ (r & 7)) << 4);
        // a zero-byte copy still gets an in-bounds source address
        const bool live = src[i] >= 0 && kvalid != 0u;
        const uint8_t* s =
            live ? p.a_src + static_cast<int64_t>(src[i]) * p.a_src_ld + kbyte : p.a_src;
        ptx::cp_async_16(dst, s, live ? 16u : 0u);
      }
      ptx::cp_async_mbar_arrive_noinc(full);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
}

// CTA pair with gathered A, the peer CTA's idle MMA warp: once the peer's own
// gather copies of a stage have landed (its local barrier), make them visible
// to the tensor core's proxy and signal the leader's barrier of that stage,
// whose MMAs read both CTAs' shared memory.  Walks the producers' k-tiles.
// The signal is a 4-byte st.async that completes 4 transaction bytes of the
// leader's barrier: measured, a remote mbarrier arrive with cluster-scope
// release kept the relay waiting ~1,800 cycles per stage, which throttled the
// pair to a third of the one-CTA speed.
template <int BN>
__device__ __forceinline__ void relay_role(const Params& p, const Shared& sh, int32_t num_tiles,
                                           const TileSched& ts) {
  int stage = 0;
  uint32_t phase = 0;
  for (int i = 0;; ++i) {
    const int32_t t = sched_next<2>(ts, i, p, sh);
    if (t >= num_tiles) break;
    for (int kt = 0; kt < p.k_tiles; ++kt) {
      const bool ok = wait_phase(sh.full + 8 * stage, phase, p, sh, 12, t);
      if (!__all_sync(0xffffffffu, ok)) return;
      ptx::fence_proxy_async_smem();
      if (ptx::elect_one())
        ptx::st_async_complete_tx(ptx::mapa(sh.map_full + (kRelayWord - kMapBars), 0), 0u,
                                  ptx::mapa(sh.full + 8 * stage, 0));
      __syncwarp();
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
}

// ------------------------------------------------------------------ kernel

template <int BN, bool GATHER, int CG, bool TR = false>
__global__ void __launch_bounds__(KernelCfg<BN, GATHER, CG>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ Params p) {
  using Cfg = KernelCfg<BN, GATHER, CG>;
  extern __shared__ uint8_t smem_raw[];
  // the next launch may start its own setup on SMs this grid leaves (it waits
  // for this grid's completion before touching memory)
  ptx::griddep_launch_dependents();
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1 KiB alignment
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int S = p.stages;
  const uint32_t a0 = base;
  const uint32_t b0 = base + S * Cfg::kABytes;
  const uint32_t out_stage = base + S * Cfg::kStageBytes;  // epilogue staging, per warp
  uint8_t* ctrl = base_ptr + S * Cfg::kStageBytes + Cfg::kEpiWarps * p.out_stage_bytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (2 * S + 5 + 2 * kSchedDepth));
  int32_t* abort_flag = reinterpret_cast<int32_t*>(tmem_slot + 1);
  int32_t* prefix = reinterpret_cast<int32_t*>(ctrl + kCtrlBytes);
  int32_t* cu_s = prefix + (kMaxGroups + 1);
  // gather-K only (the host sizes it); 16-byte aligned for vector reads (prefix
  // is 1 KiB aligned)
  int32_t* idx_s = prefix + ((2 * (kMaxGroups + 1) + 3) & ~3);

  Shared sh;
  sh.full = ptx::smem_addr(ctrl);
  sh.empty = sh.full + 8 * S;
  sh.tfull = sh.empty + 8 * S;
  sh.tempty = sh.tfull + 16;
  sh.map_full = ptx::smem_addr(ctrl + kMapBars);
  sh.map_empty = sh.map_full + 8 * kMapSlots;
  const uint32_t drain_bar = sh.tempty + 16;  // MMAs in flight have finished
  TileSched ts;
  // a unit is a CTA or a CTA pair
  ts.unit = static_cast<int32_t>(blockIdx.x) / CG;
  ts.units = static_cast<int32_t>(gridDim.x) / CG;
  const bool clc = (p.flags & FLAG_CLC_SCHED) != 0;
  ts.dyn = clc || ((p.flags & FLAG_DYNAMIC_SCHED) != 0 && p.status != nullptr);
  ts.counter = p.status + 4;
  ts.full = drain_bar + 8;
  ts.empty = ts.full + 8 * kSchedDepth;
  ts.ring = ptx::smem_addr(tmem_slot + 2);
  sh.abort = abort_flag;
  sh.prefix = prefix;
  sh.cu = cu_s;
  sh.idx = idx_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rank within the pair (rank 0 leads: it issues the MMAs of the pair)
  const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // gather forms: the copy threads' arrivals, plus the B bytes' arrival (one CTA
      // or the pair's leader, which also counts the peer's relayed bytes)
      ptx::mbar_init(sh.full + 8 * s,
                     !GATHER ? 1 : ((CG == 1 || rank == 0) ? 1 + kGatherThreads : kGatherThreads));
      ptx::mbar_init(sh.empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(sh.tfull + 8 * b, 1);
      ptx::mbar_init(sh.tempty + 8 * b, Cfg::kEpiWarps * CG);
    }
    ptx::mbar_init(drain_bar, 1);
    for (int i = 0; i < kMapSlots; ++i) {
      ptx::mbar_init(sh.map_full + 8 * i, 1);
      ptx::mbar_init(sh.map_empty + 8 * i, 1);
    }
    // ring slot consumers: the MMA warp, every epilogue warp (both CTAs of a pair),
    // the producer warps but the fetching one (both CTAs of a pair) and, for a
    // gathering pair, the peer's relay warp
    const uint32_t producers = GATHER ? kGatherWarps : 1;
    const uint32_t consumers =
        (CG == 2) ? 2 * Cfg::kEpiWarps + 1 + (2 * producers - 1) + (GATHER ? 1 : 0)
                  : Cfg::kEpiWarps + 1 + (producers - 1);
    for (int i = 0; i < kSchedDepth; ++i) {
      ptx::mbar_init(ts.full + 8 * i, 1);
      ptx::mbar_init(ts.empty + 8 * i, consumers);
    }
    ptx::mbar_init(clc_bar_addr(sh), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == Cfg::kLoadWarp && lane == 0 && p.k_tiles > 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == Cfg::kMmaWarp) {
    if (CG == 1) {
      ptx::tmem_alloc(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
      ptx::tmem_relinquish();
    } else {
      ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
      ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
  }
  // Everything above touched only this CTA's shared memory and TMEM; from here
  // on global memory that an earlier kernel in the stream may write is read.
  ptx::griddep_wait();
  // varlen-M: copy cu_seqlens and build the per-group tile prefix (warp 0)
  if (p.num_groups > 0 && warp == 0) {
    const int G = p.num_groups;
    const int per = (G + 31) / 32;
    const int g0 = min(lane * per, G), g1 = min(g0 + per, G);
    int32_t mine = 0;
    for (int g = g0; g < g1; ++g) {
      const int32_t lo = __ldg(p.cu_seqlens + g), hi = __ldg(p.cu_seqlens + g + 1);
      if (lo < 0 || hi > p.M || hi < lo) record_status(p, DEV_INDEX_RANGE, 5, g);
      const int32_t len = max(0, min(hi, p.M) - max(lo, 0));
      mine += ((len + Cfg::kTileM - 1) / Cfg::kTileM) * p.tiles_n;
    }
    int32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int32_t run = incl - mine;
    for (int g = g0; g < g1; ++g) {
      const int32_t lo = __ldg(p.cu_seqlens + g), hi = __ldg(p.cu_seqlens + g + 1);
      const int32_t clo = max(lo, 0);
      const int32_t len = max(0, min(hi, p.M) - clo);
      prefix[g] = run;
      cu_s[g] = clo;
      run += ((len + Cfg::kTileM - 1) / Cfg::kTileM) * p.tiles_n;
    }
    if (lane == 31) {
      prefix[G] = incl;
      cu_s[G] = min(max(__ldg(p.cu_seqlens + G), 0), p.M);
    }
  }
  // varlen-K: each group's K columns [start, end).  A group that breaks the
  // rules (out of [0, total_K], decreasing, or a start that is not a whole
  // 16 bytes into a K-major row) is recorded and contracts nothing.
  if (p.k_groups > 0 && warp == 0) {
    for (int g = lane; g < p.k_groups; g += 32) {
      int32_t lo = __ldg(p.cu_seqlens_k + g), hi = __ldg(p.cu_seqlens_k + g + 1);
      const bool bad = lo < 0 || hi < lo || hi > p.K || (hi > lo && lo % p.k_align != 0);
      if (bad) {
        record_status(p, DEV_INDEX_RANGE, 8, g);
        lo = hi = 0;
      }
      cu_s[g] = lo;
      prefix[g] = hi;
    }
  }
  // batch_idx_permute (plain): copy it and check that it lists each batch once.
  // Every CTA reaches the same verdict, so on a bad table all of them skip the
  // work together (no tile is computed, no role waits for another).
  if (p.batch_perm != nullptr && warp == 0) {
    const int32_t L = p.L;  // <= kMaxGroups (the host checks)
    uint32_t* seen = reinterpret_cast<uint32_t*>(cu_s);  // 1024 bits, then the verdict
    seen[lane] = 0u;
    __syncwarp();
    constexpr int32_t kNone = 0x7fffffff;
    int32_t bad_pos = kNone;  // this lane's first entry outside [0, L)
    for (int32_t l = lane; l < L; l += 32) {
      const int32_t b = __ldg(p.batch_perm + l);
      if (b < 0 || b >= L) {
        if (bad_pos == kNone) bad_pos = l;
        continue;
      }
      prefix[l] = b;
      atomicOr(seen + (b >> 5), 1u << (b & 31));
    }
    __syncwarp();
    const int32_t first_pos = __reduce_min_sync(0xffffffffu, bad_pos);
    // L entries in range name every batch iff no batch is named twice
    int32_t missing_batch = kNone;
    if (first_pos == kNone && lane < (L + 31) / 32) {
      const int32_t rem = L - 32 * lane;
      const uint32_t want = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
      const uint32_t missing = want & ~seen[lane];
      if (missing != 0u) missing_batch = 32 * lane + __ffs(static_cast<int>(missing)) - 1;
    }
    const int32_t first_missing = __reduce_min_sync(0xffffffffu, missing_batch);
    const int32_t detail = first_pos != kNone ? first_pos : first_missing;
    __syncwarp();
    if (lane == 0) {
      if (detail != kNone) record_status(p, DEV_INDEX_RANGE, 14, detail);
      seen[32] = detail != kNone ? 1u : 0u;
    }
  }
  __syncthreads();
  if (CG == 2) ptx::cluster_sync();  // the peer's barriers exist before anyone signals them
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool perm_bad = p.batch_perm != nullptr && cu_s[32] != 0;
  const int32_t num_tiles =
      (p.num_groups > 0) ? prefix[p.num_groups] : (perm_bad ? 0 : p.num_tiles);

  if (warp < Cfg::kEpiWarps) {
    epilogue_role<BN, GATHER, CG, TR>(p, sh, tmem_base, num_tiles, rank, ts,
                                  out_stage + warp * p.out_stage_bytes);
  } else if (warp == Cfg::kMmaWarp) {
    if (rank == 0) mma_role<BN, GATHER, CG>(p, sh, a0, b0, tmem_base, num_tiles, ts);
    else if constexpr (GATHER) relay_role<BN>(p, sh, num_tiles, ts);
  } else if (GATHER) {
    gather_producer_role<BN, CG>(p, sh, &tmB, a0, b0, num_tiles, rank, ts);
  } else if (warp == Cfg::kLoadWarp) {
    tma_producer_role<BN, GATHER, CG>(p, sh, &tmA, &tmB, a0, b0,
                                      ptx::smem_addr(ctrl + kMapScratch), num_tiles, rank, ts);
  } else {
    map_warp_role<BN, CG>(p, sh, &tmA, &tmB, ptx::smem_addr(ctrl + kMapScratch), num_tiles, ts);
  }

  __syncthreads();
  // Every MMA this CTA issued has finished before TMEM is freed (after an abort
  // nobody else has waited for them); the wait is bounded like all others.
  if (warp == Cfg::kMmaWarp && rank == 0) {
    if (ptx::elect_one()) {
      if (CG == 1) ptx::mma_commit(drain_bar);
      else ptx::mma_commit_pair(drain_bar, 0x1);
    }
    __syncwarp();
    wait_phase<CG == 2>(drain_bar, 0, p, sh, 6, -1);
  }
  __syncthreads();
  // no CTA of a pair leaves (or frees TMEM) while its peer may still signal it
  if (CG == 2) ptx::cluster_sync();
  if (*abort_flag) {
    // let copies and MMAs that were in flight land before the memory goes away
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 200000ull) __nanosleep(1000);
  }
  // the last CTA (pair) to finish clears the claim counter for the next call
  if (ts.dyn && !clc && rank == 0 && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.status + 5, 1) == ts.units - 1) {
      atomicExch(p.status + 4, 0);
      atomicExch(p.status + 5, 0);
    }
  }
  // split last wave: every ticket is reset by the warp that takes its last count.
  // After an abort some may be left counting, so the last unit to finish clears
  // them whenever a device error is on record (every unit has taken its tickets
  // before it counts itself finished).
  if (p.tail_tiles > 0 && rank == 0 && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.status + 7, 1) == ts.units - 1) {
      atomicExch(p.status + 7, 0);
      if (atomicAdd(p.status, 0) != 0) {
        const int32_t n = p.tail_tiles * CG * Cfg::kEpiWarps * kTicketsPerWarp;
        for (int32_t i = 0; i < n; ++i) atomicExch(p.tail_tickets + i, 0);
      }
    }
  }
  if (warp == Cfg::kMmaWarp) {
    __syncwarp();  // dealloc is warp-collective
    ptx::tc_fence_after();
    if (CG == 1) ptx::tmem_dealloc(tmem_base, Cfg::kTmemCols);
    else ptx::tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace gge
