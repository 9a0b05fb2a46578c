// Kernel parameter block shared by the host launcher and the device kernel.
#pragma once

#include <cstdint>

#include "gge_sched.cuh"

namespace gge {

enum : int32_t { DT_BF16 = 0, DT_F16 = 1, DT_E4M3 = 2, DT_E5M2 = 3, DT_F32 = 4 };
enum : int32_t { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU_TANH = 2, ACT_SILU = 3, ACT_RELU_SQ = 4 };

// Device status words (the first bytes of the caller's workspace).
enum : int32_t {
  DEV_OK = 0,
  DEV_TIMEOUT = 6,      // an mbarrier wait ran past its time limit
  DEV_INDEX_RANGE = 7,  // a gather index or a group offset was out of range
};

// Flags (debug / test switches carried in Params::flags).
enum : int32_t {
  FLAG_TILE_COUNTS = 1,        // epilogue counts visits per tile into tile_counts
  FLAG_TEST_DROP_ACC_FULL = 2, // the MMA warp never signals "accumulator full" (timeout test)
  FLAG_DYNAMIC_SCHED = 4,      // tiles claimed from an atomic counter instead of a fixed stride
  FLAG_DIRECT_STORES = 8,      // epilogue stores straight from registers (no staging buffers)
  FLAG_NO_SPLIT = 32,          // never split the last wave along K
  FLAG_RASTER_N = 128,         // raster bands of n-tiles (n varies fastest in a band)
  FLAG_CLC_SCHED = 256,        // one cluster per tile; running clusters take over the tiles
                               // of clusters not yet launched (cluster launch control)
  FLAG_SWAP_AB = 512,          // compute D^T = B A^T (the kernel's rows are the caller's N)
  FLAG_K_SERPENTINE = 1024,    // odd waves walk K backwards (L2 reuse across waves)
  FLAG_RESERVED = 16 | 64,     // reserved bits: a call that sets one is rejected
};

struct Params {
  // problem
  int32_t M;        // rows per batch (plain) or total output rows (varlen)
  int32_t N;
  int32_t K;
  int32_t L;        // batches (plain)
  int32_t k_tiles;  // ceil(K / bk)
  int32_t bk;       // K elements per stage row (128 bytes)
  int32_t stages;
  int32_t num_tiles;  // plain only: work items (tiles, plus the split tail's extra slices)
  PlainSchedule sched;
  // split last wave (plain problems; see plan_tail_split): items >= full_tiles
  // are slices; tail_tiles == 0 disables it
  int32_t full_tiles, tail_tiles, tail_splits;
  int32_t* tail_tickets;  // workspace: per tail tile, CTA, epilogue warp and chunk, the number
                          // of slices whose partial chunk that warp has written (0 between launches)
  float* partials;        // workspace: per tail tile, slice and CTA, 128 x BN fp32 accumulators
  FastDivmod tiles_n_div;  // varlen: local tile -> (m-tile, n-tile)
  int32_t tiles_n;
  // plain: the schedule's batch b computes batch batch_perm[b] (the pages'
  // batch_idx_permute; copied to shared memory and checked at kernel start)
  const int32_t* batch_perm;

  // varlen-M
  int32_t num_groups;  // 0: plain batched problem
  const int32_t* cu_seqlens;

  // varlen-K: batch l of the schedule is group l, which contracts the K
  // columns cu_seqlens_k[l] .. cu_seqlens_k[l+1]-1 of A [M, total_K] and B [N, total_K]
  int32_t k_groups;            // 0: every batch contracts all K columns
  const int32_t* cu_seqlens_k;
  int32_t k_align;             // group starts must be multiples of this (K-major operands)
  uint8_t* kmaps;              // workspace: per CTA, kMapSlots pairs of 128-byte A / B tensor maps
  const uint8_t* b_src;        // B's storage (gather-K copies a ragged group's B rows)
  int64_t b_ld;                // bytes between B's storage rows

  // gather-A (rows along M) and gather-K (rows of X along K)
  const int32_t* a_idx;   // [L][M] (plain), [total_M] (varlen-M) or [total_K] (gather-K)
  const uint8_t* a_src;   // source matrix base
  int64_t a_src_ld;       // bytes between source rows
  int32_t a_src_rows;     // valid index range
  int32_t k_bytes;        // K * element size (gather K-tail predicate)

  // epilogue
  void* d;
  int64_t ldd, sbd;       // elements
  void* post;
  int64_t ldp, sbp;
  const void* c;
  int64_t ldc, sbc;
  int32_t d_dtype, p_dtype, c_dtype;
  int32_t act;
  int32_t dact;  // backward epilogue: C is the pre-activation x, D = act'(x) * acc, PostAct = act(x)
  int32_t out_trans;  // swap_ab: C / D / PostAct hold the kernel's element (row, col) at [col][row]
  int32_t out_stage_bytes;  // shared-memory staging per epilogue warp: 32 x 32 outputs (2 or
                            // 4 KiB); 0: each lane stores its own row directly
  float alpha, beta;
  const float* alpha_dev;
  const float* beta_dev;

  // MMA
  uint32_t idesc;
  int32_t f8;          // operands are 8-bit (kind::f8f6f4)
  int32_t a_mn_major;  // A staged M-major (16-bit operands only)
  int32_t b_mn_major;  // B staged N-major (16-bit operands only)

  // control
  int32_t* status;       // workspace: [0] code, [1] where, [2] tile, [3] detail,
                         //            [4] tile claim counter, [5] finished CTAs (pairs),
                         //            [7] finished units of a split launch
  int32_t* tile_counts;  // debug visit counters
  int32_t flags;
  uint64_t timeout_ns;
};

}  // namespace gge
