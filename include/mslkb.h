/*
 * mslkb.h -- C ABI of libmslkb.so: the FP8 rowwise-scaled grouped GEMM
 * f8f8bf16_rowwise_grouped for NVIDIA GB300 (sm_103a), stacked and dynamic layouts.
 *
 * The operation (MSLK #471 "Back the FP8 rowwise grouped GEMM ops with FlyDSL on ROCm":
 * commit introducing the rowwise scaling scheme; PR Summary table) is, for each group g
 * and every row r that group owns,
 *
 *     out[r, n] = bf16_rne( scale_a[r] * scale_b[g, n] * sum_k A[r, k] * B[g, n, k] )
 *
 * with A and B in OCP FP8 E4M3 ("e4m3fn"), scale_a and scale_b in fp32, the sum held in
 * fp32 and never rounded before the scales are applied (once, after the K loop), and
 * the result rounded to bf16 with round-to-nearest-even.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - Pointers named as device pointers must point to memory the current CUDA device
 *   can access (device or managed memory).  They are owned by the caller, are only
 *   read/written by work enqueued on `stream`, and are not retained after the call
 *   returns.  Every buffer is dense and row-major with the sizes given; strided views
 *   are not supported (the kernel addresses the output as one flat row-major buffer:
 *   MSLK #471, commit rejecting a strided output).
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy default stream.
 *   Calls are asynchronous: they enqueue work and return without synchronising.
 *   The first call on a device performs one-time set-up (device query, kernel attributes,
 *   driver entry point).  The first call on each stream (outside stream capture) also
 *   allocates that stream's workspace (2 x #SMs x 128 KB of fp32 partial sums for split
 *   tiles, plus counters, among them the tile claim counter of the CTA-pair plans; about
 *   40 MB on GB300), which lasts until mslkb_release_workspace or the end of the process;
 *   later calls on the stream allocate nothing and may be captured in a CUDA graph.  A
 *   call captured on a stream that has no workspace yet runs without splitting tiles and,
 *   on CTA pairs, takes its tiles in a fixed stride (same results within tolerance,
 *   possibly slower).
 *   Calls on one stream share its workspace in stream order; a captured graph keeps the
 *   workspace of the stream it was captured on, so two launches of such graphs, or one
 *   and a call on that stream, must not run at the same time.
 * - Sizes are int64_t.  Errors are reported by the return value; nothing is enqueued
 *   when a call returns anything but MSLKB_OK.  Argument checks happen before any CUDA
 *   call, so a bad argument is reported even where no GPU is present.
 * - The library is compiled for sm_103a only; any other device gives MSLKB_ERR_DEVICE.
 * - Errors found on the device (a wait that timed out, m_sizes that overran total_M)
 *   cannot be returned by an asynchronous call; they are OR-ed into a per-device status
 *   word read by mslkb_get_device_status().
 * - Host threads may call at the same time, on one stream or on several; the library's
 *   tables (device set-up, stream workspaces) are guarded by a lock.
 * - Every kernel launch is enqueued inside an NVTX push/pop range of the domain "mslkb"
 *   whose message is the kernel variant's name (mslkb_variant_name) and whose int64
 *   payload is the rows of A, so a profiler can select this library's launches (ncu:
 *   --nvtx --nvtx-include "mslkb@<variant name>/").  With no tool attached the range
 *   calls return at once; a launch captured in a CUDA graph replays without them.
 */
#ifndef MSLKB_H_
#define MSLKB_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSLKB_API __attribute__((visibility("default")))
#else
#define MSLKB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mslkb_status {
  MSLKB_OK = 0,
  MSLKB_ERR_NULL = 1,   /* a pointer needed for the given sizes is NULL */
  MSLKB_ERR_SHAPE = 2,  /* a size is negative, too large, or N is not a multiple of 8 */
  MSLKB_ERR_ALIGN = 3,  /* out is not 16-byte aligned (ragged layouts: or A / B not
                           16-byte aligned, or their row length not a multiple of 16) */
  MSLKB_ERR_DEVICE = 4, /* the current device is not sm_103 (GB300 / B300) */
  MSLKB_ERR_CUDA = 5,   /* a CUDA runtime or driver call failed; see mslkb_last_cuda_error */
  MSLKB_ERR_TOO_LARGE = 6 /* needs more scratch than the allocation-free entry point holds */
} mslkb_status;

/* Bits of the device status word (mslkb_get_device_status). */
#define MSLKB_DEV_TIMEOUT 0x1u        /* a pipeline wait in the kernel gave up (~1 s)  */
#define MSLKB_DEV_MSIZES_CLAMPED 0x2u /* m_sizes had a negative entry or summed past total_M */
#define MSLKB_DEV_BAD_SLICE 0x4u      /* ragged K: a slice bound not a multiple of 16 */
#define MSLKB_DEV_BOUNDS 0x8u         /* checked build (libmslkb_checked.so) only: a kernel
                                         index fell outside the buffers of the call; that
                                         access was not made as asked.  Bits 16..23 then name
                                         the kinds of access: 16 group metadata, 17 TMA load
                                         K coordinate, 18 TMA load row / column / group
                                         coordinate, 19 TMA K coordinate not 16-byte aligned,
                                         20 scales, 21 direct output store, 22 TMA output
                                         store, 23 split-tile workspace */

/* Limits. */
#define MSLKB_MAX_GROUPS 1024         /* G (kernel keeps per-group tables in shared memory) */
#define MSLKB_MAX_DIM 2147483647LL    /* every size, and total_M * K, N * K, rows * N ... */

/*
 * Stacked layout (op f8f8bf16_rowwise_grouped_stacked; MSLK #471, PR Summary table:
 * "[G] int64 row counts", and the commits on the packed "sizes" layout and its tile
 * retire guard).
 *
 *   A        device, e4m3 codes [total_M, K]      rows of all groups packed along M
 *   B        device, e4m3 codes [G, N, K]         one [N, K] weight matrix per group
 *   scale_a  device, fp32 [total_M]               one scale per row of A
 *   scale_b  device, fp32 [G, N]                  one scale per (group, column)
 *   m_sizes  device, int64 [G]                    rows per group, in group order
 *   out      device, bf16 [total_M, N]            16-byte aligned
 *
 * Group g owns rows [off_g, off_g + m_g) with off_0 = 0, off_{g+1} = off_g + m_g.
 * Empty groups own no rows and cost no work.  Each m_g is clamped into
 * [0, total_M - off_g]; if any entry needed clamping, MSLKB_DEV_MSIZES_CLAMPED is set in
 * the device status word.  Rows of out past the last group are left untouched.
 * K = 0 writes +0.0 to every owned row (MSLK #471, commit zeroing an empty reduction).
 * Any K >= 0 is accepted: when K is a multiple of 16 and A and B are 16-byte aligned
 * the tiles are fetched by TMA; otherwise a narrower asynchronous copy path is used,
 * with zero fill past K (MSLK #471, commit on the K tail).
 * N must be a multiple of 8, the width of one 16-byte bf16 store (MSLK #471, commits on
 * the N tail and on predicating a store on its last column).
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_rowwise_grouped_stacked(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int64_t *m_sizes, void *out, int64_t total_M, int64_t G, int64_t N, int64_t K,
    void *stream);

/*
 * Dynamic (padded) layout (op f8f8bf16_rowwise_grouped_dynamic; MSLK #471, PR Summary
 * table: "[G, M, K] slabs, runtime valid-row count", commit adding the padded layout and
 * commit adding its test: padding rows asserted zero).
 *
 *   A                   device, e4m3 codes [G * expected_m, K]   one slab per group
 *   B                   device, e4m3 codes [G, N, K]
 *   scale_a             device, fp32 [G * expected_m]
 *   scale_b             device, fp32 [G, N]
 *   zero_start_index_M  device, int64 [G]      valid rows at the top of each slab
 *   out                 device, bf16 [G * expected_m, N], 16-byte aligned
 *
 * Group g owns slab rows [g*E, (g+1)*E) with E = expected_m; the first
 * v_g = min(max(zero_start_index_M[g], 0), E) rows are computed and every other row of
 * the slab is written +0.0, whatever A and scale_a hold there (the zeroed-output
 * contract, folded into the kernel so that every output byte is written once).
 * K and N rules as for the stacked layout.
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_rowwise_grouped_dynamic(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int64_t *zero_start_index_M, void *out, int64_t G, int64_t expected_m,
    int64_t N, int64_t K, void *stream);

/*
 * Offsets layout (2D-3D, the torch-native grouped-mm addressing; MSLK #471, commits
 * decoding group boundaries from an int32 inclusive prefix sum and binding the `_mm` op's
 * 2D-3D rank combination).  As the stacked call, but the groups are given as
 *
 *   offsets  device, int32 [G]   inclusive prefix: group g owns rows
 *                                [offsets[g-1], offsets[g]) with offsets[-1] = 0
 *
 * A row count is the step between successive offsets; a negative step owns no rows and
 * steps past total_M are clamped (both set MSLKB_DEV_MSIZES_CLAMPED), as for m_sizes.
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_rowwise_grouped_offsets(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int32_t *offsets, void *out, int64_t total_M, int64_t G, int64_t N, int64_t K,
    void *stream);

/*
 * Batched layout (3D-3D; MSLK #471, commit adding the layout whose groups all carry their
 * full complement of rows, and the one eliding its retire guard).  Every group owns a full
 * slab of M rows and no metadata is read:
 *
 *   A        device, e4m3 codes [G, M, K]
 *   B        device, e4m3 codes [G, N, K]
 *   scale_a  device, fp32 [G, M]
 *   scale_b  device, fp32 [G, N]
 *   out      device, bf16 [G, M, N], 16-byte aligned
 *
 * M need not divide the tile height: rows past a slab are never written (the next slab's
 * rows belong to the next group).  K and N rules as for the stacked layout.
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_rowwise_grouped_batched(
    const void *A, const void *B, const float *scale_a, const float *scale_b, void *out,
    int64_t G, int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Ragged-N layout (3D-2D; MSLK #471, commit adding the form whose weights are one
 * [total_N, K] matrix that the groups partition by row, results packed side by side).
 * Group g owns the output columns [offsets[g-1], offsets[g]) (offsets[-1] = 0):
 *
 *   out[m, n] = bf16_rne((acc * scale_a[g, m]) * scale_b[n]),
 *   acc = sum_k A[g, m, k] * B[n, k]                       for every n of group g
 *
 *   A        device, e4m3 codes [G, M, K] (one slab of M rows per group), 16-byte aligned
 *   B        device, e4m3 codes [total_N, K], 16-byte aligned
 *   scale_a  device, fp32 [G, M]
 *   scale_b  device, fp32 [total_N]
 *   offsets  device, int32 [G]   inclusive prefix over the columns
 *   out      device, bf16 [M, total_N], 16-byte aligned; columns past offsets[G-1] are
 *            not written
 *
 * K must be a multiple of 16 (TMA rows) and total_N of 8; a group's column count may be
 * anything (its last columns are stored one by one).  Column counts follow the offsets
 * rules of mslkb_f8f8bf16_rowwise_grouped_offsets (clamped at total_N, status bit set).
 * M = 0, G = 0 or total_N = 0: nothing to do.  K = 0: the owned columns are +0.0.
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_rowwise_grouped_n_offsets(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int32_t *offsets, void *out, int64_t G, int64_t M, int64_t total_N, int64_t K,
    void *stream);

/*
 * Ragged-K layout (2D-2D; MSLK #471, commit adding the layout whose groups slice K).
 * Group g contracts over k in [offsets[g-1], offsets[g]) (offsets[-1] = 0) and writes a
 * whole [M, N] slab:
 *
 *   out[g, m, n] = bf16_rne((acc * scale_a[g, m]) * scale_b[g, n]),
 *   acc = sum over the slice of A[m, k] * B[n, k]
 *
 *   A        device, e4m3 codes [M, total_K], 16-byte aligned
 *   B        device, e4m3 codes [N, total_K], 16-byte aligned
 *   scale_a  device, fp32 [G, M]
 *   scale_b  device, fp32 [G, N]
 *   offsets  device, int32 [G]   inclusive prefix over K
 *   out      device, bf16 [G, M, N], 16-byte aligned; every element is written
 *
 * total_K must be a multiple of 16, N of 8, and every slice must start and end on a
 * multiple of 16: a group whose slice does not is not computed -- its slab is written
 * +0.0 and MSLKB_DEV_BAD_SLICE is set.  An empty slice gives +0.0 (the empty sum).
 * Slice bounds are clamped into [0, total_K] as row counts are for the offsets layout.
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_rowwise_grouped_k_offsets(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int32_t *offsets, void *out, int64_t G, int64_t M, int64_t N, int64_t total_K,
    void *stream);

/*
 * Block-scaled (groupwise) stacked layout (MSLK #471, commit introducing the rowwise
 * scheme beside the block scheme the grouped kernel already had: a scale per scale block,
 * applied to each block's partial sum inside the K loop; K and N must cover whole scale
 * blocks).  Scale blocks of 128 along K and N:
 *
 *   out[r, n] = bf16_rne( sum_kb scale_a[r, kb] * scale_b[g, n / 128, kb] * S_kb ),
 *   S_kb = sum over k in [128 kb, 128 kb + 128) of A[r, k] * B[g, n, k]
 *
 *   A, B, m_sizes, out  as for mslkb_f8f8bf16_rowwise_grouped_stacked
 *   scale_a  device, fp32 [total_M, K / 128]
 *   scale_b  device, fp32 [G, N / 128, K / 128]
 *
 * K and N must be multiples of 128 (MSLKB_ERR_SHAPE otherwise); A and B 16-byte aligned
 * (MSLKB_ERR_ALIGN).  Each K block's partial sum is scaled in fp32 on its way from the
 * tensor core into the fp32 accumulator.
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_groupwise_grouped_stacked(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int64_t *m_sizes, void *out, int64_t total_M, int64_t G, int64_t N, int64_t K,
    void *stream);

/*
 * Block-scaled (groupwise) dynamic layout (MSLK #471: the block scheme of the commit
 * introducing the rowwise scheme -- "a compile-time blockscale flag" over the grouped
 * kernel's layouts -- on the padded layout of the PR Summary table and its commit; the
 * padded layout's per-group slab addressing is what a [G, scale_k, M] scale tensor needs).
 * Scale blocks of 128 along K and N:
 *
 *   A                   device, e4m3 codes [G * expected_m, K]   one slab per group
 *   B                   device, e4m3 codes [G, N, K]
 *   scale_a             device, fp32 [G * expected_m, K / 128]   per slab row and K block
 *   scale_b             device, fp32 [G, N / 128, K / 128]
 *   zero_start_index_M  device, int64 [G]      valid rows at the top of each slab
 *   out                 device, bf16 [G * expected_m, N], 16-byte aligned
 *
 *   out[r, n] = bf16_rne( sum_kb scale_a[r, kb] * scale_b[g, n / 128, kb] * S_kb )
 *
 * for the first v_g = min(max(zero_start_index_M[g], 0), E) rows of slab g, +0.0 for the
 * rest of the slab whatever A and scale_a hold there.  K and N must be multiples of 128
 * (MSLKB_ERR_SHAPE otherwise); A and B 16-byte aligned (MSLKB_ERR_ALIGN).
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_groupwise_grouped_dynamic(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int64_t *zero_start_index_M, void *out, int64_t G, int64_t expected_m,
    int64_t N, int64_t K, void *stream);

/*
 * Block-scaled (groupwise) batched layout: the block scaling above on the batched layout
 * (MSLK #471, commit adding the layout whose groups all carry their full complement of
 * rows): every group owns a full slab of M rows and no metadata is read.
 *
 *   A        device, e4m3 codes [G, M, K]
 *   B        device, e4m3 codes [G, N, K]
 *   scale_a  device, fp32 [G, M, K / 128]
 *   scale_b  device, fp32 [G, N / 128, K / 128]
 *   out      device, bf16 [G, M, N], 16-byte aligned
 */
MSLKB_API mslkb_status mslkb_f8f8bf16_groupwise_grouped_batched(
    const void *A, const void *B, const float *scale_a, const float *scale_b, void *out,
    int64_t G, int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Allocation-free stacked call (no counterpart on the pages: an addition of this library).
 *
 * For callers that cannot allocate device memory when they call: plug-ins whose host
 * framework owns every device allocation (and gives a library none of its own), and
 * serving loops that cannot take the device-wide synchronisation a cudaMalloc can cause.
 * Same arguments, layout, results and errors as mslkb_f8f8bf16_rowwise_grouped_stacked;
 * the caller still provides inputs and output.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Its split-tile scratch (fp32 partial sums and arrival counters) is a static device
 * array of MSLKB_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading the library holds
 * until the process exits.  The plans that split tiles by default (swap-AB tiles, up to
 * 32 rows per group on average, e.g. MoE decode) need at most 2 x #SMs x 16 KB of it; a
 * plan that needs more -- 128-row activation tiles split under mslkb_set_split_k(2), or a
 * device with very many SMs -- returns MSLKB_ERR_TOO_LARGE and launches nothing.  CTA-pair
 * plans take their tiles in a fixed stride here (no claim counter).
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 * once per device, with that device current).  Each call clears the counters it uses on
 * `stream` (cudaMemsetAsync) before its kernel.  All calls share the one array, which
 * keeps the last call's contents: calls that overlap on the GPU (different streams, say)
 * race and must be serialised by the caller.
 */
#define MSLKB_NOALLOC_SCRATCH_BYTES (8u << 20)
MSLKB_API mslkb_status mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc(
    const void *A, const void *B, const float *scale_a, const float *scale_b,
    const int64_t *m_sizes, void *out, int64_t total_M, int64_t G, int64_t N, int64_t K,
    void *stream);

/* Static description of a status code.  Never NULL. */
MSLKB_API const char *mslkb_status_string(mslkb_status status);

/* The cudaError_t (or, for a failed tensor-map encode, the CUresult) behind the last
 * MSLKB_ERR_CUDA returned on this thread. */
MSLKB_API int mslkb_last_cuda_error(void);

/*
 * Reads the device status word of the current device and clears it.  Enqueued on
 * `stream` and then waits for that stream, so it orders after earlier calls on it.
 * flags: host pointer receiving the MSLKB_DEV_* bits.  When the word reports a timeout,
 * the split-tile arrival counters of every stream workspace on the device are cleared as
 * well (a kernel that gave up may have left them short), on `stream`: call it while no
 * other stream runs this library's kernels on the device.
 */
MSLKB_API mslkb_status mslkb_get_device_status(void *stream, uint32_t *flags);

/*
 * Kernel variants and the plan the host would choose.  Pure host code: no CUDA call.
 * layout: 0 = stacked (rows = total_M), 1 = dynamic (rows = expected_m per group),
 *         2 = ragged N (rows = M, N = total_N), 3 = ragged K (rows = M, K = total_K),
 *         4 = block-scaled stacked (rows = total_M), 5 = block-scaled dynamic or batched
 *         (rows = expected_m per group).
 * num_sms: streaming multiprocessors of the target device.
 * a_align / b_align: the byte alignment of the A and B base addresses (e.g. 256).
 */
typedef struct mslkb_plan_info {
  int32_t variant;      /* index into the variant table, see mslkb_variant_name */
  int32_t swap_ab;      /* 1: weights take the MMA M side and tokens the N side */
  int32_t tile_m;       /* activation rows per tile */
  int32_t tile_n;       /* weight rows (output columns) per tile */
  int32_t stages;       /* shared-memory pipeline depth */
  int32_t tma;          /* 1: TMA loads; 0: cp.async loader */
  int32_t copy_width;   /* bytes per asynchronous copy of the cp.async loader */
  int32_t grid;         /* persistent CTAs launched */
  int32_t threads;      /* threads per CTA */
  int32_t smem_bytes;   /* dynamic shared memory per CTA */
  int64_t tiles_bound;  /* host upper bound on output tiles */
  int32_t split_k;      /* 1: the last waves' tiles are split along K over all CTAs */
  int32_t reserved;
} mslkb_plan_info;

MSLKB_API mslkb_status mslkb_plan(int32_t layout, int64_t rows, int64_t G, int64_t N, int64_t K,
                        int32_t num_sms, int64_t a_align, int64_t b_align,
                        mslkb_plan_info *info);

/* Number of kernel variants and the name of one (NULL past the end). */
MSLKB_API int32_t mslkb_num_variants(void);
MSLKB_API const char *mslkb_variant_name(int32_t variant);

/*
 * Resources of one kernel variant on the current device: CTAs that fit on one SM (the
 * library needs 1) and registers per thread.  Makes CUDA calls (device query, kernel
 * attributes); the library runs the same check before a variant's first launch.
 */
MSLKB_API mslkb_status mslkb_variant_resources(int32_t variant, int32_t *blocks_per_sm,
                                               int32_t *regs_per_thread);

/*
 * Failure detection (an addition of this library; the pages have no counterpart).  Every
 * wait of the kernels' pipelines is bounded: a wait that runs past the limit (default
 * ~1 s) makes the kernel give up, record MSLKB_DEV_TIMEOUT in the device status word, let
 * its copies in flight land, free its tensor memory and return, so the context stays
 * usable.  mslkb_set_wait_timeout_us sets the limit for the following launches (0: the
 * default; otherwise at least 1000 us, else MSLKB_ERR_SHAPE).
 */
MSLKB_API mslkb_status mslkb_set_wait_timeout_us(int64_t us);

/*
 * Frees the split-tile workspace of `stream` on the current device (see the conventions
 * above), after waiting for the work already enqueued on `stream`.  The next call on that
 * stream allocates a new one.  A CUDA graph captured on the stream keeps the address of
 * the workspace it was captured with: destroy such graphs first.  A stream with no
 * workspace: nothing to do.  Other streams' workspaces are not touched.
 */
MSLKB_API mslkb_status mslkb_release_workspace(void *stream);

/* Number of stream workspaces the library holds on the current device. */
MSLKB_API int32_t mslkb_workspace_count(void);

/* Library version, as major * 10000 + minor * 100 + patch. */
MSLKB_API int32_t mslkb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSLKB_H_ */
