// Host-side launcher interface between the C ABI (bdla_api.cu) and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bdla_common.cuh"

namespace bdla {

struct Problem {
    const int32_t *cu;   // device cu_seqlens or nullptr (fixed-length)
    int n_docs;          // documents (B for fixed-length calls)
    int T;               // per-document length (fixed) or total tokens (varlen)
    int64_t tokens;      // total tokens in the tensors
    int H, dk, dv;
    float b;
    int mode;            // bdla_decay
    DeviceStatus *st;
    cudaStream_t stream;
};

// Slots of a checkpoint array with the given stride.
inline int64_t ckpt_slots(const Problem &p, int stride)
{
    return (p.tokens + stride - 1) / stride + p.n_docs;
}

// Events recorded around a kernel's launches (measurement hook, see
// bdla_set_kernel_events); null when unset.
struct KernelEvents {
    cudaEvent_t start = nullptr, stop = nullptr;
};
extern KernelEvents g_kernel_events[BDLA_KERNEL_COUNT];

inline void mark_start(int kernel, cudaStream_t s)
{
    if (g_kernel_events[kernel].start)
        cudaEventRecord(g_kernel_events[kernel].start, s);
}
inline void mark_stop(int kernel, cudaStream_t s)
{
    if (g_kernel_events[kernel].stop)
        cudaEventRecord(g_kernel_events[kernel].stop, s);
}

// gamma and dfac (d lambda / d a, may be nullptr) are head-major [H][tokens].
cudaError_t launch_decay(const Problem &p, const float *a, float *gamma, float *dfac);

// Tile-serial forward on CUDA cores.  Used with o == nullptr to write fp32
// checkpoints whose stride is below the 128-token block.
cudaError_t launch_fwd_tile(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                            const __nv_bfloat16 *v, const float *gamma, const float *h0, void *o,
                            int o_f32, float *hT, float *ckpt, int ckpt_stride);

// Tensor-core forward (tcgen05 / TMEM / TMA): o, hT and checkpoints whose
// stride is a multiple of 128 tokens.
// o == nullptr runs the state chain only (checkpoints for the backward).
cudaError_t launch_fwd_sm100(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const float *gamma, const float *h0, void *o,
                             int o_f32, float *hT, void *ckpt, int ck_bf16, int ckpt_stride);

// Tensor-core backward.  `states` holds the state before every 128-token
// block: checkpoints whose stride divides 128, fp32 or bf16.  For dv = 256
// the value columns are split in two slices; `part` (bwd_partial_floats
// floats of workspace) receives the second slice's partial dq, dk, da.
size_t bwd_partial_floats(const Problem &p);
cudaError_t launch_bwd_sm100(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const __nv_bfloat16 *dO, const float *gamma,
                             const float *dfac, const void *states, int st_bf16, int st_stride,
                             const float *dhT, float *dq, float *dk, float *dv, float *da, float *dh0,
                             float *part);



}  // namespace bdla
