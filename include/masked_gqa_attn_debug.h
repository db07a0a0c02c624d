/*
 * masked_gqa_attn_debug.h -- extra entry points of the debug library,
 * libmgqa_debug.so: the same sources as libmgqa.so built with MGQA_DEBUG.
 * The engine pages have no counterpart; this is test equipment.
 *
 * The debug library exports everything masked_gqa_attn.h declares, with
 * three differences on the device:
 *   - bounds and alignment checks on the global, TMA and mask accesses: a
 *     failed check writes MGQA_ERR_DEVICE_CHECK to *dev_error and skips the
 *     access (no trap);
 *   - event counters (read with mgqa_debug_counters);
 *   - an injectable stall of the tensor-core prefill's load pipeline with a
 *     shortened wait limit, so that a test can watch a bounded wait give up
 *     (MGQA_ERR_TIMEOUT) without hanging the GPU.
 * The debug state is one copy per device, in device memory; the functions
 * below act on the current device and synchronise with it.
 */
#ifndef MASKED_GQA_ATTN_DEBUG_H
#define MASKED_GQA_ATTN_DEBUG_H

#include "masked_gqa_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Number of event counters. */
#define MGQA_DEBUG_NUM_COUNTERS 4
/* counter 0: softmax warps of the tensor-core prefill that rescaled their
 *            running output (the row max grew by more than 2^8 within a row);
 * counter 1: key tiles the tensor-core prefill's softmax warps processed;
 * counters 2, 3: unused (0). */

/* Copies the first n (<= MGQA_DEBUG_NUM_COUNTERS) counters to host memory
 * `out`. Synchronous. */
MGQA_API mgqa_status mgqa_debug_counters(uint64_t *out, int32_t n);

/* Zeroes the counters, removes any injected stall and restores the normal
 * wait limit (2 s). Synchronous. */
MGQA_API mgqa_status mgqa_debug_reset(void);

/* From the next tensor-core prefill launch on, the TMA producer issues no
 * load for non-empty key tile `tile` (its position in the row's list of
 * non-empty tiles, >= 1) or any later one, and every pipeline wait gives up
 * after `wait_limit_ns` (> 0). Every load issued before the stall lands
 * before the CTA exits, and every MMA issued completes before the tensor
 * memory is freed. tile < 0 removes the stall. Synchronous. */
MGQA_API mgqa_status mgqa_debug_inject_prefill_stall(int32_t tile, uint64_t wait_limit_ns);

/* Per-CTA timeline of the decode launches since the previous read, for the
 * first n_ctas (<= 512) CTAs in launch order (x fastest), as written by the
 * most recent launch that reached each stamp: 16 values per CTA -- the SM
 * clock at the kernel's phase boundaries 0..8 (entry; after the grid-
 * dependency wait; the allowed-slot words formed; the first batch's copies
 * issued; the first batch landed; every batch computed; the in-CTA merge; the
 * partials sent to their owners in the cluster; this CTA's slice of the
 * output merged and written), then at four points around the first batch of
 * the 16-bit path: 9 (masked rows fixed up), 10 (the shared maximum
 * exchanged), 11 (this warp's scores and maximum formed), 12 (the batch's
 * bytes armed); the global timer (ns) at entry and at stamp 7, and the SM id.
 * A stamp a CTA did not reach reads 0. Reading clears the record for all
 * CTAs. Synchronous. */
MGQA_API mgqa_status mgqa_debug_decode_timeline(uint64_t *out, int32_t n_ctas);

/* Per-CTA timeline of the tensor-core prefill launches since the previous
 * read, for the first n_ctas (<= 1024) CTAs in launch order (x fastest), as
 * written by the most recent launch that reached each stamp: 16 values per
 * CTA -- the SM clock at 0 (entry), 1 (after the grid-dependency wait), 9
 * (the first copies issued and the segment range formed), 11 (the packed-bit
 * mask folded into per-tile bits), 12 (every key tile classified), 2 (the
 * non-empty tiles counted), 3 (the first score MMAs issued), 10 (head 0's
 * first scores complete), 4 (head 0's first P handed over), 8 (the last P.V
 * MMAs issued), 5 (head 0's output complete), 6 (head 0's output tile
 * stored), 7 (head 0's epilogue done); the global timer (ns) at entry and at
 * stamp 7, and the SM id. A stamp a CTA did not reach reads 0.
 * Reading clears the record. Synchronous. */
MGQA_API mgqa_status mgqa_debug_prefill_timeline(uint64_t *out, int32_t n_ctas);

/* Per-key-tile event trace of the first n_ctas (<= 4) CTAs of the
 * tensor-core prefill launches since the previous read, in launch order (x
 * fastest), as written by the most recent launch: 64 tiles x 18 values per
 * CTA (the SM clock), for the CTA's n-th non-empty key tile n < 64. Events
 * 2t and 2t+1: the MMA warp begins issuing / has committed S_t(n) = Q_t K^T
 * (head t); 4+2t and 5+2t: the same for O_t += P_t(n) V(n); 8+4t: softmax
 * warpgroup t sees S_t(n) complete (its first warp); 9+4t: every warp of it
 * has read the scores; 10+4t: the first warp's exponentials are done; 11+4t:
 * every warp has handed P_t(n) over; 16 / 17: the producer has issued the
 * loads of K(n) / V(n). An event not reached reads 0. Reading clears the
 * record. Synchronous. */
MGQA_API mgqa_status mgqa_debug_prefill_trace(uint64_t *out, int32_t n_ctas);

#ifdef __cplusplus
}
#endif

#endif /* MASKED_GQA_ATTN_DEBUG_H */
