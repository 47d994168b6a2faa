/*
 * mslkb_tuning.h -- tuning and test hooks of libmslkb.so (declared apart from the entry
 * points in mslkb.h; the pages have no counterpart).
 *
 * Every setting here is PROCESS-GLOBAL: it applies to every following call on every
 * thread and device until it is changed back.  None of them changes what a call computes
 * beyond the tolerance the library keeps (the accumulation chunk is limited to lengths
 * that keep it), except mslkb_test_stall_next_launch, which spoils one launch on purpose.
 * They exist for the library's own tests, for benchmarks and for tuning studies; a
 * production caller needs none of them, and one that flips them changes the performance
 * of every other thread's calls.
 */
#ifndef MSLKB_TUNING_H_
#define MSLKB_TUNING_H_

#include "mslkb.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Test hook: force every following call on any thread to use one variant (index from
 * mslkb_variant_name; -1 restores the heuristic).  A variant that cannot serve a call
 * (a TMA variant with K % 16 != 0, say) makes that call return MSLKB_ERR_SHAPE.
 * Used to check that different variants give bit-identical results.
 */
MSLKB_API mslkb_status mslkb_force_variant(int32_t variant);

/*
 * Split policy (stream-K).  With T output tiles and P CTAs, tiles of all full waves but
 * the last run whole; the remaining tiles are cut into K blocks and every CTA takes an
 * equal contiguous share, so no SM idles in the last wave.  A split tile is finished by
 * the CTA that completes its last piece, which adds the fp32 partial sums of all pieces
 * in a fixed order (results do not depend on timing).  0 runs whole tiles only; 1 (the
 * default) splits plans with swap-AB tiles (few rows per group: each piece's partial sums
 * are small, and more SMs stream the weights); 2 splits every plan.  Applies to every
 * following call from any thread; a tuning and test hook.  Other values give
 * MSLKB_ERR_SHAPE.
 */
MSLKB_API mslkb_status mslkb_set_split_k(int32_t enable);

/*
 * Accumulation chunk.  The tensor core's own fp32 accumulation adds with round-toward-
 * zero; over a long K with cancelling partial sums that bias exceeds the tolerance of
 * 1e-6 * sum|terms|.  So the kernel lets the tensor core sum at most `kblocks` blocks of
 * 128 K elements into one TMEM buffer, and its epilogue adds each such partial sum into
 * fp32 registers with round-to-nearest (the accumulator is still fp32 and is never
 * rounded to a narrower type before the scales are applied).  Default 8 (1024 K
 * elements): partial sums built to cancel inside every chunk then stay within half the
 * tolerance on GB300 (4 K-blocks: a quarter; 16 K-blocks, or the whole K in the tensor
 * core, exceed it).  So only 1 to 8 are accepted; other values give MSLKB_ERR_SHAPE and
 * leave the setting unchanged.  Shorter chunks cost time (more hand-overs to the
 * epilogue).  Applies to every following call from any thread.
 */
MSLKB_API mslkb_status mslkb_set_accumulation_chunk(int32_t kblocks);
MSLKB_API int32_t mslkb_accumulation_chunk(void);

/*
 * Weight prefetch of the swap-AB (few rows per group) plans.  With programmatic dependent
 * launch a CTA can be resident while the kernel before it on the stream finishes; in that
 * time it reads the group metadata speculatively, works out its first `kblocks` K blocks
 * of weights and asks L2 to prefetch them.  A hint only: the schedule is rebuilt from the
 * metadata after the dependency wait, and every load reads L2, which is coherent with
 * what the earlier kernel writes.  -1: the default, 14 K blocks (224 KB of weights per
 * CTA); 0: off.
 * Applies to every following call from any thread; a tuning and test hook.  Values
 * below -1 give MSLKB_ERR_SHAPE.
 */
MSLKB_API mslkb_status mslkb_set_weight_prefetch(int32_t kblocks);

/*
 * Test hook for the weight prefetch: the next launch builds its speculative schedule from
 * `meta` (a device buffer laid out like that call's own metadata, G entries) instead of
 * the call's metadata, so that the prefetch goes to other tiles than the call computes.
 * The results must not change.  A launch through the ragged entry points, which prefetch
 * nothing, uses the hook up.
 */
MSLKB_API mslkb_status mslkb_test_speculate_from_next_launch(const void* meta);

/*
 * Test hook for failure detection: the next launch, through any entry point, has its
 * first CTA (both CTAs of its first pair, on CTA-pair kernels) withhold one pipeline stage,
 * so that a wait of that CTA runs out after the limit set by mslkb_set_wait_timeout_us and
 * the kernel's abort path runs.  That launch's output is incomplete and the status word
 * reports MSLKB_DEV_TIMEOUT; a following call computes normally.  Only kernels fed by TMA
 * take part: a launch of the cp.async kernels uses the hook up and computes normally.
 */
MSLKB_API mslkb_status mslkb_test_stall_next_launch(void);

#ifdef __cplusplus
}
#endif

#endif /* MSLKB_TUNING_H_ */
