// Device-side helpers shared by the bdla kernels (not by the oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bdla.h"

namespace bdla {

constexpr int kChunk = 16;  // decay tile: the unit of the bound (16 tokens)

// Status word at the start of the workspace.  Kernels record the first error
// with atomicCAS and never trap.
struct DeviceStatus {
    unsigned int code;
    unsigned int where;  // kernel-specific detail (e.g. document index)
    unsigned int pad[62];
};
constexpr size_t kStatusBytes = 256;

__device__ __forceinline__ void set_status(DeviceStatus *st, unsigned int code, unsigned int where)
{
    if (st != nullptr && atomicCAS(&st->code, 0u, code) == 0u)
        st->where = where;
}

// Log-decay parameterisations ("Engineering Long-Context Training for
// Trillion-Parameter MoE Models", sec. 3.2): bounded b * sigmoid(a), or the
// unbounded -softplus(a).  sigmoid and softplus are written from their
// definitions 1 / (1 + e^-a) and max(a, 0) + log1p(e^-|a|).
__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }

__device__ __forceinline__ float log_decay(float a, float b, int mode)
{
    if (mode == BDLA_DECAY_BOUNDED_SIGMOID)
        return b * sigmoidf_(a);
    return -(fmaxf(a, 0.0f) + log1pf(expf(-fabsf(a))));
}

// d lambda / d a
__device__ __forceinline__ float log_decay_deriv(float a, float b, int mode)
{
    float s = sigmoidf_(a);
    if (mode == BDLA_DECAY_BOUNDED_SIGMOID)
        return b * s * (1.0f - s);
    return -s;
}

// Document [start, end) of document n: packed offsets or fixed length T.
struct DocSpan {
    int64_t start;
    int64_t len;
};

__device__ __forceinline__ DocSpan doc_span(const int32_t *cu, int n, int T)
{
    DocSpan d;
    if (cu != nullptr) {
        d.start = cu[n];
        d.len = (int64_t)cu[n + 1] - (int64_t)cu[n];
    } else {
        d.start = (int64_t)n * T;
        d.len = T;
    }
    return d;
}

// A document span must lie inside the tensors; kernels skip (and the decay
// kernel reports) spans that do not, so malformed cu_seqlens never cause an
// out-of-bounds access.
__device__ __forceinline__ bool doc_valid(const DocSpan &d, int64_t tokens)
{
    return d.start >= 0 && d.len >= 0 && d.start + d.len <= tokens;
}

// Checkpoint slot of (document n, doc-local block c) for a given stride.
__device__ __forceinline__ int64_t ckpt_slot(int64_t doc_start, int n, int64_t c, int stride)
{
    return doc_start / stride + n + c;
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

}  // namespace bdla
