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

// d lambda / d a.  sigma'(a) = sigma(a) (1 - sigma(a)) is taken as
// sigma(a) sigma(-a): equal in exact arithmetic, and it keeps its relative
// accuracy for saturated logits, where 1 - sigma(a) in fp32 rounds to 0.
__device__ __forceinline__ float log_decay_deriv(float a, float b, int mode)
{
    if (mode == BDLA_DECAY_BOUNDED_SIGMOID)
        return b * sigmoidf_(a) * sigmoidf_(-a);
    return -sigmoidf_(a);
}

// Gamma of one token: the inclusive sum of the log-decays up to it inside its
// 16-token tile.  Lane l of a full warp holds position (l & 15) of a tile
// (lanes 0-15 one tile, 16-31 the next) and passes its lambda (0 past the
// end of the document: positions past the end never enter an earlier
// position's sum).  Every kernel takes Gamma from this four-step shuffle
// scan, so all of them see bitwise the same Gamma for the same logits.
__device__ __forceinline__ float tile_gamma(float lam, int lane)
{
#pragma unroll
    for (int off = 1; off < kChunk; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, lam, off, kChunk);
        if ((lane & (kChunk - 1)) >= off)
            lam += y;
    }
    return lam;
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

// Sequence segments (sequence parallelism inside one GPU).  When the
// (document, head) units are too few to fill the GPU, each document is cut
// into segments of seg_blk 128-token blocks (a document without tokens still
// has one, empty, segment) and one CTA takes one segment.  Segment s of
// document n owns slot floor(cu[n] / L) + n + s, L = 128 seg_blk tokens;
// slots are distinct across documents and fewer than ceil(tokens / L) +
// n_docs.  Slots that no segment owns are gaps.  seg_blk == 0: no cut, the
// slot is the document index.
struct SegSpan {
    int n;               // document
    int s;               // segment inside the document
    int64_t doc_start;   // first token of the document
    int64_t start;       // first token of the segment
    int64_t len;         // tokens in the segment
    int blk_base;        // doc-local index of the segment's first 128-token block
    bool last;           // the document's last segment
    bool valid;          // false: a gap or a malformed document
};

__device__ __forceinline__ SegSpan seg_span(const int32_t *cu, int T, int64_t tokens, int n_docs,
                                            int slot, int seg_blk)
{
    SegSpan g;
    g.valid = false;
    g.s = 0;
    g.blk_base = 0;
    g.last = true;
    if (seg_blk <= 0) {
        g.n = slot;
        const DocSpan d = doc_span(cu, slot, T);
        g.doc_start = g.start = d.start;
        g.len = d.len;
        g.valid = doc_valid(d, tokens);
        return g;
    }
    const int64_t L = (int64_t)seg_blk * 128;
    // largest n with floor(start(n) / L) + n <= slot (increasing in n for valid offsets)
    int lo = 0, hi = n_docs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int64_t sm = cu != nullptr ? (int64_t)cu[mid] : (int64_t)mid * T;
        if (sm / L + mid <= slot)
            lo = mid;
        else
            hi = mid - 1;
    }
    const DocSpan d = doc_span(cu, lo, T);
    if (!doc_valid(d, tokens))
        return g;
    const int64_t s = (int64_t)slot - (d.start / L + lo);
    const int64_t nseg = d.len > 0 ? (d.len + L - 1) / L : 1;
    if (s < 0 || s >= nseg)
        return g;
    g.n = lo;
    g.s = (int)s;
    g.doc_start = d.start;
    g.start = d.start + s * L;
    g.len = d.len - s * L < L ? d.len - s * L : L;
    g.blk_base = (int)(s * seg_blk);
    g.last = s == nseg - 1;
    g.valid = true;
    return g;
}

// Checkpoint slot of (document n, doc-local block c) for a given stride.
__device__ __forceinline__ int64_t ckpt_slot(int64_t doc_start, int n, int64_t c, int stride)
{
    return doc_start / stride + n + c;
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

}  // namespace bdla
