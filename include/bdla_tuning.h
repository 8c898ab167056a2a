/*
 * bdla_tuning.h — process-wide settings of libbdla.so that are not part of
 * the operation itself: the sequence-segment policy, a measurement hook and
 * two test hooks for the bounded waits.  None of them changes a result
 * beyond floating-point rounding order; the defaults are what a user wants.
 *
 * Each setting is one value held by the library for the whole process and
 * read by every later call, on any thread (the values are atomics, so
 * setting one while another thread makes calls is not a data race, but the
 * other thread's calls see the change).
 */
#ifndef BDLA_TUNING_H
#define BDLA_TUNING_H

#include "bdla.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Sequence parallelism inside one GPU.  The state passes from chunk to
 * chunk ("Engineering Long-Context Training for Trillion-Parameter MoE
 * Models: Three Key Breakthroughs", sec. 3.1), so a (document, head) pair is
 * a chain of 128-token blocks.  When those pairs are too few to occupy the
 * GPU, the library cuts each document into segments of `blocks` 128-token
 * blocks, first computes the state (forward) or adjoint state (backward)
 * entering every segment (kernel id BDLA_KERNEL_SEG: one summary GEMM pass
 * and one scan over the segments), then runs one CTA per segment.  The
 * result is the same up to floating-point rounding order.
 *   blocks == 0 (default): automatic; documents are cut, into about four
 *                          segments per SM, only when (documents x heads x
 *                          dv/128 slices) is below the GPU's SM count.
 *   blocks <  0: never cut.
 *   blocks >  0: always cut into segments of `blocks` blocks (at least as
 *                long as needed to keep the segment count within 65535).
 * The workspace size depends on it (bdla_workspace_bytes reads it), so size
 * the workspace after changing it.  Always BDLA_OK.
 */
bdla_status bdla_set_seq_split(int blocks);

/*
 * Measurement hook.  Until called again with NULL events, every later call
 * that launches kernel `kernel` (BDLA_KERNEL_*) records `start_event` just
 * before and `stop_event` just after that launch, on the call's stream, so
 * the caller can time the kernel alone (cudaEventElapsedTime).  Both events
 * are cudaEvent_t created by the caller.  Returns BDLA_ERR_SHAPE for an
 * unknown kernel id.
 */
enum { BDLA_KERNEL_DECAY = 0, BDLA_KERNEL_FWD = 1, BDLA_KERNEL_BWD = 2, BDLA_KERNEL_STATES = 3,
       BDLA_KERNEL_SEG = 4, BDLA_KERNEL_COUNT = 5 };
bdla_status bdla_set_kernel_events(int kernel, void *start_event, void *stop_event);

#ifdef __cplusplus
}
#endif

#endif /* BDLA_TUNING_H */
