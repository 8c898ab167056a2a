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

/*
 * Test hooks for the bounded waits.  Every wait of a kernel's pipeline
 * (a TMA copy landing, an MMA completing, a hand-off between warps) gives up
 * after a time limit instead of spinning forever; the CTA then records
 * BDLA_ERR_TIMEOUT in the call's status word, lets the copies and MMAs it
 * started finish, frees its tensor memory and returns, so the CUDA context
 * stays usable.  These two settings let a test exercise that path.
 *
 * bdla_set_wait_limit_ns: limit of the pipeline waits in nanoseconds for
 * later launches (default 2 s; 0 restores the default).  The waits that
 * drain a CTA's own copies and MMAs before it exits keep the default.
 *
 * bdla_set_test_stall: until called again with role 0, every later launch
 * of kernel `kernel` (BDLA_KERNEL_FWD, _BWD, _STATES or _SEG) makes the
 * warp(s) of one role wait, at their second block (their first if there is
 * one block), on a barrier that nothing arrives at; the wait runs out after
 * the limit above.  Returns BDLA_ERR_SHAPE for an unknown kernel or role.
 * Off by default; not for production use.
 */
enum { BDLA_STALL_NONE = 0, BDLA_STALL_PRODUCER = 1, BDLA_STALL_MMA = 2, BDLA_STALL_EPILOGUE = 3 };
bdla_status bdla_set_wait_limit_ns(uint64_t ns);
bdla_status bdla_set_test_stall(int kernel, int role);

#ifdef __cplusplus
}
#endif

#endif /* BDLA_TUNING_H */
