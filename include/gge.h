/*
 * gge.h -- C ABI of libgge.so: fused persistent GEMM epilogues on one GB300
 * (sm_103a).
 *
 * The operation is the one the QuACK pages implement for Hopper
 * (quack-kernels 0.2.0: quack/dense_gemm_sm90.py ``GemmSm90``,
 * quack/gemm_act_sm90.py ``GemmActSm90`` / ``gemm_act_sm90``):
 *
 *   D[m,n,l]       = alpha * sum_k A[m,k,l] * B[n,k,l] + beta * C[m,n,l]
 *   PostAct[m,n,l] = act( same value, before rounding )
 *
 * with fp32 accumulation; each output is rounded once (round to nearest even)
 * to its own dtype.  Without C there is no beta term (the pages' epilogue
 * visit adds ``beta * C`` only when C is given).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  Nothing is
 *     allocated, freed or synchronised by the library (except
 *     gge_read_device_status and gge_read_static_scratch_status, which
 *     synchronise the given stream).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *     Kernels are launched with programmatic stream serialization: a launch may
 *     begin its setup (shared memory, TMEM) while the previous kernel in the
 *     stream is finishing, but reads and writes no global memory before that
 *     kernel has completed, so stream order holds as for any launch.
 *   - Validation happens on the host before any launch; a rejected call
 *     launches nothing and returns GGE_ERR_INVALID_ARG / GGE_ERR_UNSUPPORTED /
 *     GGE_ERR_ALIGNMENT / GGE_ERR_WORKSPACE.  A failed launch returns
 *     GGE_ERR_CUDA.  Faults found on the device (a wait that ran out of time,
 *     a gather index or group offset out of range) are written to the
 *     workspace and read back with gge_read_device_status.
 *   - Strides are in ELEMENTS.  The contiguous dimension of every tensor must
 *     have stride 1, every other stride and every base pointer must be 16-byte
 *     aligned (the pages' rule: the contiguous dimension 16-byte aligned).
 *   - Sizes are int64 in the structs but every extent must be < 2^31.
 */
#ifndef GGE_H_
#define GGE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gge_stream_t; /* same type as cudaStream_t */

typedef enum gge_status {
  GGE_OK = 0,
  GGE_ERR_INVALID_ARG = 1, /* NULL where a pointer is required, inconsistent shapes */
  GGE_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement      */
  GGE_ERR_ALIGNMENT = 3,   /* base pointer or stride not 16-byte aligned             */
  GGE_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than gge_workspace_size      */
  GGE_ERR_CUDA = 5,        /* a CUDA runtime / driver call failed                    */
  GGE_ERR_TIMEOUT = 6,     /* device: a pipeline wait ran past its time limit        */
  GGE_ERR_INDEX_RANGE = 7  /* device: gather index / group offset out of range       */
} gge_status;

typedef enum gge_dtype {
  GGE_BF16 = 0,
  GGE_F16 = 1,
  GGE_E4M3 = 2, /* float8_e4m3fn */
  GGE_E5M2 = 3, /* float8_e5m2   */
  GGE_F32 = 4
} gge_dtype;

/* Activations of the fused epilogue.  The pages list relu and
 * gelu_tanh_approx (quack/gemm_act_sm90.py ``act_fn_map``); SiLU is the
 * textbook x / (1 + exp(-x)). */
typedef enum gge_act {
  GGE_ACT_NONE = 0,
  GGE_ACT_RELU = 1,      /* x > 0 ? x : 0                                        */
  GGE_ACT_GELU_TANH = 2, /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))      */
  GGE_ACT_SILU = 3,      /* x / (1 + exp(-x))                                    */
  GGE_ACT_RELU_SQ = 4    /* relu(x)^2 (act_fn_map's relu_sq)                     */
} gge_act;

/* A strided 3-D view [rows, cols, batch]. */
typedef struct gge_tensor {
  void* ptr;            /* device pointer to element [0,0,0]                    */
  int32_t dtype;        /* gge_dtype                                            */
  int32_t reserved;     /* must be 0                                            */
  int64_t rows, cols, batch;
  int64_t stride_row, stride_col, stride_batch; /* in elements                  */
} gge_tensor;

/* Optional tuning / debug knobs; pass NULL for the defaults. */
typedef struct gge_config {
  int32_t tile_n;         /* 0 = auto; else output columns per tile: 64 (TMA forms),
                             128 or 256 on one CTA, 256, 224, 192 or 160 on a
                             CTA pair (the narrower pair tiles need a K-major B) */
  int32_t num_ctas;       /* 0 = one persistent CTA per SM                         */
  int32_t raster_band;    /* 0 = auto; tiles per raster band (plain problems): auto
                             takes the width that keeps a wave's A and B rows
                             fewest, sqrt(units * tile_n / tile_m) m-tiles     */
  int32_t stages;         /* 0 = as many as shared memory holds                    */
  int32_t flags;          /* bit 0: count tile visits into tile_counts;
                             bit 1: test hook -- the MMA warp never signals a
                             finished accumulator, so the epilogue's bounded wait
                             runs out and the call reports GGE_ERR_TIMEOUT;
                             bit 2: dynamic tile scheduler -- after its first
                             tile each CTA (pair) claims the next one from a
                             counter in the workspace (needs a workspace);
                             bit 3: direct epilogue stores -- each lane stores its
                             own output row instead of staging 32 x 32 chunks in
                             shared memory (frees 16-32 KiB: one more pipeline
                             stage on a CTA pair; best when K is long);
                             bit 4: reserved (a call that sets it returns
                             GGE_ERR_UNSUPPORTED);
                             bit 5: never split the last wave.  By default a
                             plain problem whose last wave of tiles is at most
                             half full cuts those tiles into 2-8 K-slices that
                             otherwise idle CTAs compute.  Each slice leaves its
                             fp32 partial sums in the workspace; whichever unit
                             finishes a tile's slices last adds them, in slice
                             order, and runs the epilogue.  No CTA waits for
                             another, so the result does not depend on when the
                             CTAs run.  Not with the dynamic scheduler or the
                             gather and varlen forms; needs gge_workspace_size
                             bytes;
                             bit 6: reserved (a call that sets it returns
                             GGE_ERR_UNSUPPORTED);
                             bit 7: raster along N -- plain problems walk bands
                             of raster_band n-tiles, the n-tile varying fastest
                             (default: bands of m-tiles, the m-tile fastest);
                             bit 8: cluster launch control -- the grid has one
                             CTA (pair) per tile, and a running one takes over
                             the tiles of those not launched yet
                             (clusterlaunchcontrol.try_cancel) instead of a
                             fixed stride; no workspace needed; not with bit 2;
                             the last wave is not split;
                             bit 9: swap_ab -- compute D^T = B A^T: the kernel's
                             tiles run over the caller's N (rows) and M
                             (columns) and the epilogue stores C / D / PostAct
                             transposed into the caller's N-major [M, N]
                             layout (plain problems: gge_gemm, gge_gemm_act,
                             gge_gemm_dact).  For small M, so that M becomes the
                             tile width (64-wide one-CTA tiles exist for this);
                             bit 10: serpentine K -- work items of odd waves
                             (item index / resident units) walk K backwards, so
                             each wave starts on the k-slices the previous one
                             read last, still in L2 (plain and varlen-M forms
                             with TMA-loaded A; reproducible, the direction is
                             fixed by the plan).                               */
  int32_t cta_group;      /* 0 = auto; 1 = one CTA per 128-row tile; 2 = a CTA pair
                             per 256-row tile (tcgen05 cta_group::2; with gather-A
                             256-column tiles only; not with gather-K)           */
  int32_t* tile_counts;   /* device int32 per tile (debug coverage), or NULL       */
  uint64_t timeout_ns;    /* 0 = default (2 s) limit for each pipeline wait        */
  const int32_t* batch_idx_permute;
                          /* NULL, or device int32[L], a permutation of 0..L-1
                             (the pages' batch_idx_permute; plain problems with
                             L <= 1024 only, else GGE_ERR_UNSUPPORTED): the
                             scheduler visits batch batch_idx_permute[b] where it
                             would visit batch b, so it fixes the order in which
                             batches run, never the results.  Every CTA checks
                             it on the device before any work: an entry outside
                             [0, L) or a batch listed twice records
                             GGE_ERR_INDEX_RANGE (where 14, tile = the first bad
                             position, or the first batch not listed) and the
                             launch computes and writes nothing.               */
} gge_config;

/*
 * Arguments of one GEMM.
 *   A : [M, K, L]  rows = M, cols = K.  K-major (stride_col == 1) or, for
 *       16-bit operands loaded by TMA (every form but the gathers), M-major
 *       (stride_row == 1).  In gather-A, A is the SOURCE matrix
 *       [rows_src, K, 1], K-major; in gather-K, the M-major source [M, K_src, 1].
 *   B : [N, K, L]  rows = N, cols = K.  K-major (stride_col == 1) or, for
 *       16-bit operands, N-major (stride_row == 1).  8-bit operands must be
 *       K-major (as on the pages).
 *   C : optional [M, N, L] input, N-major.  NULL: no beta term.
 *   D : optional [M, N, L] output, N-major.
 *   PostAct : optional [M, N, L] output of act(...), N-major.  Required when
 *       act != GGE_ACT_NONE.
 *   Dtypes: A and B both 16-bit and equal (bf16 or f16), or both 8-bit
 *       (e4m3 / e5m2 in any combination).  C, D, PostAct: bf16, f16 or f32.
 *   N must be a multiple of 8.
 *   alpha_dev / beta_dev: optional device float scalars that override alpha /
 *       beta (read once per CTA).
 */
typedef struct gge_gemm_args {
  gge_tensor A;
  gge_tensor B;
  const gge_tensor* C;
  const gge_tensor* D;
  const gge_tensor* PostAct;
  float alpha;
  float beta;
  const float* alpha_dev;
  const float* beta_dev;
  int32_t act;               /* gge_act */
  int32_t reserved;
  const gge_config* config;  /* NULL = defaults */
} gge_gemm_args;

/* Bytes of device workspace that let a call run at full speed, for every
 * entry point except gge_gemm_varlen_k and gge_gemm_gather_k (see
 * gge_workspace_size_varlen_k): 256 bytes of status words and scheduler
 * counters, plus, for plain problems, room to split the last, partly filled
 * wave of tiles along K (16 KiB of tickets, then one 128 x 256 fp32 partial
 * block per SM: about 20 MiB on a 152-SM GPU; the split needs a 256-byte
 * aligned workspace).  Any workspace of at least 256 bytes works: with less
 * room the last wave runs unsplit.  Layout: bytes 0-255 status words, then
 * the tickets, then the partial blocks (or, for varlen-K, the tensor-map
 * slots), so one workspace serves every entry point in turn.  The workspace is caller-owned, at least 16-byte
 * aligned, must be zeroed once before first use, and is reusable across calls
 * on the same stream (not by calls running concurrently on other streams).
 * The arguments are not inspected (they may be NULL); the size depends on the
 * current device. */
size_t gge_workspace_size(const gge_gemm_args* args, int32_t num_groups);

/* Workspace bytes gge_gemm_varlen_k and gge_gemm_gather_k need on the current
 * device: the status words and the ticket region plus 4 KiB of tensor-map copies for each CTA a
 * launch can have (one per SM: about 0.6 MiB on a 152-SM GPU).  The arguments
 * are not inspected (they may be NULL); returns 0 if the device cannot be
 * queried.  (The slots start after the 16 KiB ticket region, which these
 * calls leave untouched.) */
size_t gge_workspace_size_varlen_k(const gge_gemm_args* args, int32_t num_groups);

/* D = alpha A B^T + beta C (PostAct must be NULL and act NONE).
 * Page: quack/dense_gemm_sm90.py, gemm_sm90 / GemmSm90.epi_visit_acc_subtile. */
gge_status gge_gemm(const gge_gemm_args* args, void* workspace, size_t workspace_bytes,
                    gge_stream_t stream);

/* D (optional) and PostAct = act(alpha A B^T + beta C), act applied to the
 * unrounded fp32 value.  Page: quack/gemm_act_sm90.py, gemm_act_sm90 /
 * GemmActSm90.epi_visit_acc_subtile. */
gge_status gge_gemm_act(const gge_gemm_args* args, void* workspace, size_t workspace_bytes,
                        gge_stream_t stream);

/* Backward activation epilogue: the accumulator S = A B^T is the incoming
 * gradient dout, C (required) holds the pre-activation x, and
 *   D = act'(x) * S      (required)        PostAct = act(x)   (optional)
 * with act in {relu, relu_sq, gelu_tanh, silu}; alpha and beta are not used.
 * Page: quack-kernels 0.2.0 diff, quack/gemm_dact_sm90.py, gemm_dact_sm90 /
 * GemmDActSm90.epi_visit_acc_subtile (act_bwd(x, dout) -> (dx, out)). */
gge_status gge_gemm_dact(const gge_gemm_args* args, void* workspace, size_t workspace_bytes,
                         gge_stream_t stream);

/* Varlen-M grouped GEMM: A is [total_M, K, 1], B is [N, K, G] (batch = G
 * groups), C / D / PostAct are [total_M, N, 1].  Group g owns rows
 * cu_seqlens_m[g] .. cu_seqlens_m[g+1]-1 and multiplies them by B[:,:,g];
 * rows outside every group are not written.  cu_seqlens_m: DEVICE int32
 * [G+1], non-decreasing, cu[0] >= 0, cu[G] <= total_M (violations are
 * clamped and reported as GGE_ERR_INDEX_RANGE by gge_read_device_status).
 * 1 <= G <= 1024.  act as in gge_gemm_act.
 * Page: quack/dense_gemm_sm90.py, GemmSm90 with VarlenArguments(mCuSeqlensM). */
gge_status gge_gemm_varlen_m(const gge_gemm_args* args, const int32_t* cu_seqlens_m,
                             int32_t num_groups, void* workspace, size_t workspace_bytes,
                             gge_stream_t stream);

/* Varlen-K grouped GEMM (the weight-gradient shape of grouped experts):
 * A is [M, total_K, 1], B is [N, total_K, 1], C / D / PostAct are [M, N, G]
 * (batch = G groups).  Group g contracts the K columns
 * cu_seqlens_k[g] .. cu_seqlens_k[g+1]-1:
 *   D[:,:,g] = alpha * A[:, K_g] B[:, K_g]^T + beta * C[:,:,g]
 * and an empty group gives alpha * 0 + beta * C.  Columns outside every group
 * take part in no product.  cu_seqlens_k: DEVICE int32 [G+1], non-decreasing,
 * cu[0] >= 0, cu[G] <= total_K.  When A or B is K-major, every non-empty
 * group must start on a 16-byte boundary of the K-major rows (a multiple of 8
 * for 16-bit, 16 for 8-bit operands); with A M-major and B N-major any
 * offsets are allowed.  A group that breaks these rules contracts nothing and
 * is reported as GGE_ERR_INDEX_RANGE by gge_read_device_status.
 * 1 <= G <= 1024.  act as in gge_gemm_act.  The workspace (256-byte aligned,
 * zeroed once) must hold gge_workspace_size_varlen_k bytes: the kernel keeps
 * per-CTA copies of the A / B tensor maps there, rewritten with each group's
 * K extent.  Page: quack/dense_gemm_sm90.py, GemmSm90 with
 * VarlenArguments(mCuSeqlensK) (update_tensormap_shape per group; a group
 * with k_tile_cnt == 0 keeps a zero accumulator). */
gge_status gge_gemm_varlen_k(const gge_gemm_args* args, const int32_t* cu_seqlens_k,
                             int32_t num_groups, void* workspace, size_t workspace_bytes,
                             gge_stream_t stream);

/* Gather-K: the varlen-K GEMM above whose A is gathered along K.  args->A is
 * the SOURCE [M, K_src, 1], M-major (stride_row == 1; the usual storage of
 * X [K_src, M] row-major), 16-bit, M a multiple of 8; a_idx is DEVICE int32
 * [total_K] with total_K = columns of B.  Column k of the effective A is
 * column a_idx[k] of the source; B [N, total_K] is read at column k itself.
 * Group rules as in gge_gemm_varlen_k (with a K-major B, non-empty groups
 * start on multiples of 8); an index outside [0, K_src) reads zeros and is
 * reported as GGE_ERR_INDEX_RANGE.  One CTA per 128 x BN tile; the rows are
 * copied by four gather warps with 16-byte cp.async (a TMA row gather issues
 * too slowly for four rows of 128 bytes at a time).  The workspace (256-byte
 * aligned) must hold gge_workspace_size_varlen_k bytes.  Page: quack/dense_gemm_sm90.py,
 * GemmSm90 with gather_A and VarlenArguments(mCuSeqlensK)
 * (copy_utils.gather_k_get_copy_fn). */
gge_status gge_gemm_gather_k(const gge_gemm_args* args, const int32_t* a_idx,
                             const int32_t* cu_seqlens_k, int32_t num_groups, void* workspace,
                             size_t workspace_bytes, gge_stream_t stream);

/* Gather-A GEMM: row r of the effective A is row a_idx[r] of the source
 * matrix args->A ([rows_src, K, 1], K-major, 16-bit).  With cu_seqlens_m
 * (DEVICE int32 [G+1]) it is the varlen-M problem above, a_idx being
 * [total_M] with total_M = rows of D / PostAct; with cu_seqlens_m == NULL it
 * is a plain batched problem of M = rows of D per batch and a_idx [L][M].
 * An index outside [0, rows_src) reads zeros and is reported as
 * GGE_ERR_INDEX_RANGE.  Page: quack/dense_gemm_sm90.py,
 * GemmSm90.load_AB_gather_A (mAIdx). */
gge_status gge_gemm_gather_a(const gge_gemm_args* args, const int32_t* a_idx,
                             const int32_t* cu_seqlens_m, int32_t num_groups, void* workspace,
                             size_t workspace_bytes, gge_stream_t stream);

/* gge_gemm_act without a caller workspace, for callers that cannot allocate
 * device memory where they run the GEMM (a host framework that owns all device
 * memory through its own arena or caching allocator, or a latency-critical path
 * that must not call the allocator).  The pages have no counterpart: it is an
 * addition of this library.
 *   - The scratch (the 256 bytes of status words) lives in a fixed 1024-byte
 *     __device__ area inside the library, held on every GPU that loads it until
 *     process exit.  It has no room for partial sums, so the last wave of tiles
 *     is never split along K on this path (see gge_workspace_size).
 *   - The first call on a device looks up that area's device address (on the
 *     current device); make that first call before any stream capture.  A
 *     failed lookup returns GGE_ERR_CUDA and is tried again by the next call.
 *   - Each call clears the area's scheduler counters (an async memset on
 *     `stream`), then launches the same kernel as gge_gemm_act.  Nothing is
 *     allocated.
 *   - Device errors (a wait past its limit, GGE_ERR_TIMEOUT) are recorded in
 *     the area and kept until gge_read_static_scratch_status reads them.
 *   - All calls on a device share the one area: calls that overlap on the GPU
 *     (different streams without ordering) race on it. */
gge_status gge_gemm_act_static_scratch(const gge_gemm_args* args, gge_stream_t stream);

/* gge_read_device_status for the library's own scratch area: synchronises
 * `stream`, returns the device status that gge_gemm_act_static_scratch calls
 * on the current device recorded since it was last read (GGE_OK or
 * GGE_ERR_TIMEOUT), and clears it.  `detail` (may be NULL) receives
 * [where, tile].  No counterpart on the pages. */
gge_status gge_read_static_scratch_status(gge_stream_t stream, int32_t* detail);

/* Synchronises `stream`, returns the device status recorded in `workspace`
 * since it was last cleared (GGE_OK, GGE_ERR_TIMEOUT or GGE_ERR_INDEX_RANGE)
 * and clears it.  `detail` (may be NULL) receives [where, tile]. */
gge_status gge_read_device_status(void* workspace, gge_stream_t stream, int32_t* detail);

const char* gge_status_string(gge_status status);

/* ---- host-side helpers (no GPU needed) -------------------------------- */

/* FastDivmod parameters as quack/fast_math.py FastDivmod.create builds them:
 * p = 31 + ceil(log2 d), multiplier = ceil(2^p / d), shift = p - 32. */
void gge_fastdivmod_params(int32_t divisor, uint32_t* multiplier, uint32_t* shift);

/* q = n / d by the FastDivmod formula (host build of the device code),
 * for 0 <= n < 2^31. */
int32_t gge_fastdivmod_div(int32_t divisor, int32_t n);

/* The plain persistent schedule: tile index t -> (batch, m-tile, n-tile) for a
 * grid of tiles_m x tiles_n tiles per batch and `batches` batches, with
 * `band` m-tiles per raster band (n-tiles when along_n != 0, config flag
 * bit 7).  Writes `count` triples into out[3*count] for t = 0 .. count-1.
 * Returns the number of tiles of the problem.  Page: quack/dense_gemm_sm90.py,
 * the tile scheduler's raster_order and max_swizzle_size. */
int32_t gge_schedule_map(int32_t tiles_m, int32_t tiles_n, int32_t batches, int32_t band,
                         int32_t along_n, int32_t count, int32_t* out);

/* The launch plan the library would use for `args` (tile and pipeline
 * shape).  form: GGE_FORM_DEFAULT (plain, or varlen-M when num_groups > 0),
 * GGE_FORM_GATHER_A, GGE_FORM_VARLEN_K or GGE_FORM_GATHER_K.  Returns GGE_OK or the validation
 * error of the call. */
enum { GGE_FORM_DEFAULT = 0, GGE_FORM_GATHER_A = 1, GGE_FORM_VARLEN_K = 2, GGE_FORM_GATHER_K = 3 };
typedef struct gge_plan_info {
  int32_t tile_m, tile_n, tile_k, stages;  /* tile_m: rows per (pair) tile */
  int32_t num_tiles;  /* plain and varlen-K problems; -1 for varlen-M (known on
                         the device only) */
  int32_t grid;
  int32_t threads;
  int32_t smem_bytes;
  int32_t raster_band;
  int32_t cta_group;  /* 1 or 2 CTAs per tile */
  int32_t raster_along_n; /* 1: bands of n-tiles (config flag bit 7) */
  int32_t tail_tiles; /* tiles of the last, partly filled wave that are split along K
                         (plain problems; 0: none).  Reported only when the unit
                         count is known here, i.e. config->num_ctas is set. */
  int32_t tail_splits; /* K-slices per split tile (1: none) */
} gge_plan_info;
gge_status gge_plan(const gge_gemm_args* args, int32_t num_groups, int32_t form,
                    gge_plan_info* out);

/* ---- autotuning ---------------------------------------------------------
 * Page: quack-kernels 0.2.0 diff, quack/gemm_config.py (GemmConfig and
 * get_all_configs: a space of tile shapes, cooperative / ping-pong
 * warpgroups, 1x2 / 2x1 clusters and swap_ab to search by timing).  Here the space is the launch shapes this library
 * has: one CTA per 128 x 128 or 128 x 256 tile, or a CTA pair per 256 x 256,
 * 224, 192 or 160 tile (not with the gather forms), times the raster of
 * plain problems (bands of m-tiles of the automatic width or 8, or bands of
 * n-tiles: flag bit 7), times staged or direct epilogue stores.  The pages' swap_ab is not in the space: it needs M-major
 * output stores, which the epilogue does not have. */

/* Which entry point a tuning call times. */
enum {
  GGE_OP_GEMM = 0,      /* gge_gemm (PostAct NULL) or gge_gemm_act          */
  GGE_OP_DACT = 1,      /* gge_gemm_dact                                      */
  GGE_OP_VARLEN_M = 2,  /* gge_gemm_varlen_m (cu = cu_seqlens_m)              */
  GGE_OP_GATHER_A = 3,  /* gge_gemm_gather_a (idx = a_idx, cu may be NULL)    */
  GGE_OP_VARLEN_K = 4,  /* gge_gemm_varlen_k (cu = cu_seqlens_k)              */
  GGE_OP_GATHER_K = 5   /* gge_gemm_gather_k (idx = a_idx, cu = cu_seqlens_k) */
};

/* Writes up to `max` candidate configurations for (args, op) into `out`
 * (host only, no GPU needed: shapes the planner rejects are left out) and
 * returns how many there are (which may exceed `max`).  Each candidate is
 * args->config (or the defaults) with tile_n, cta_group and raster_band set. */
int32_t gge_tune_candidates(const gge_gemm_args* args, int32_t op, int32_t num_groups,
                            gge_config* out, int32_t max);

/* Times every candidate of (args, op) on `stream` -- `reps` launches each
 * after one warm-up launch, CUDA events around them -- and writes the fastest
 * configuration to *best (and its mean time in ms to *best_ms, if not NULL).
 * Every launch computes the real outputs, so they hold the result on return.
 * Synchronises `stream`.  The result is also stored in an in-process cache
 * keyed by the problem's shapes, dtypes, strides pattern, activation and op,
 * which gge_tuned_config reads.  Errors of a launch are returned as they are;
 * a candidate rejected by the planner is skipped. */
gge_status gge_autotune(const gge_gemm_args* args, int32_t op, const int32_t* idx,
                        const int32_t* cu, int32_t num_groups, void* workspace,
                        size_t workspace_bytes, gge_stream_t stream, int32_t reps,
                        gge_config* best, float* best_ms);

/* The configuration gge_autotune found for a problem of the same key, or
 * GGE_ERR_INVALID_ARG if there is none (no GPU work).  The launch-shape
 * fields are the search's; tile_counts, timeout_ns and batch_idx_permute are
 * taken from args->config (NULL / 0 without one). */
gge_status gge_tuned_config(const gge_gemm_args* args, int32_t op, int32_t num_groups,
                            gge_config* out);

/* Library version string. */
const char* gge_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GGE_H_ */
