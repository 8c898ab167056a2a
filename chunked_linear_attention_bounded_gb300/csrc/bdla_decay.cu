// Decay kernel: per-token log-decay and its tile-local inclusive cumsum.
//
// "Engineering Long-Context Training for Trillion-Parameter MoE Models",
// sec. 3.1: each chunk carries a per-position cumulative decay Gamma whose
// reciprocal normalises the in-chunk products; sec. 3.2: the log-decay is
// b * sigmoid(a) (bounded) instead of -softplus(a).  Gamma restarts at every
// doc-local 16-token tile, so with the bound it stays in [16 b, 0].
//
// One CTA handles 128 consecutive tokens of one document for 32 heads at a
// time: the [128 x heads] slab of logits is read coalesced (a is token-major)
// into shared memory, each thread sums one (tile, head) column, and Gamma is
// written head-major ([H][tokens]) so the attention kernels read one head's
// 128 values as a single coalesced line.  Optionally also writes
// d lambda / d a in the same layout (used by the backward).
#include "bdla_internal.h"

namespace bdla {

namespace {
constexpr int kTok = 128;   // tokens per slab (8 tiles)
constexpr int kHeads = 32;  // heads per pass
}

__global__ void __launch_bounds__(256)
decay_kernel(const float *__restrict__ a, float b, int mode, const int32_t *__restrict__ cu,
             int n_docs, int T, int64_t tokens, int H, float *__restrict__ gamma,
             float *__restrict__ dfac, DeviceStatus *st)
{
    __shared__ float sa[kTok][kHeads + 1];
    const int n = blockIdx.y;
    const DocSpan d = doc_span(cu, n, T);
    if (cu != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        bool bad = cu[n + 1] < cu[n];
        if (n == 0 && cu[0] != 0)
            bad = true;
        if (n == n_docs - 1 && (int64_t)cu[n_docs] != tokens)
            bad = true;
        if (bad)
            set_status(st, BDLA_ERR_DEVICE, (unsigned)n);
    }
    if (!doc_valid(d, tokens))
        return;
    const int64_t nslab = (d.len + kTok - 1) / kTok;
    for (int64_t sl = blockIdx.x; sl < nslab; sl += gridDim.x) {
        const int64_t t0 = d.start + sl * kTok;
        const int len = (int)(d.len - sl * kTok < kTok ? d.len - sl * kTok : kTok);
        for (int h0 = 0; h0 < H; h0 += kHeads) {
            const int nh = H - h0 < kHeads ? H - h0 : kHeads;
            __syncthreads();
            for (int e = threadIdx.x; e < kTok * nh; e += blockDim.x) {
                const int t = e / nh, hh = e % nh;
                sa[t][hh] = t < len ? a[(t0 + t) * H + h0 + hh] : 0.0f;
            }
            __syncthreads();
            if (dfac != nullptr) {
                for (int e = threadIdx.x; e < kTok * nh; e += blockDim.x) {
                    const int hh = e / kTok, t = e % kTok;
                    if (t < len)
                        dfac[(int64_t)(h0 + hh) * tokens + t0 + t] = log_decay_deriv(sa[t][hh], b, mode);
                }
                __syncthreads();
            }
            for (int e = threadIdx.x; e < (kTok / kChunk) * nh; e += blockDim.x) {
                const int hh = e / (kTok / kChunk), c = e % (kTok / kChunk);
                float acc = 0.0f;
                for (int i = 0; i < kChunk; ++i) {
                    const int t = c * kChunk + i;
                    if (t < len) {
                        acc += log_decay(sa[t][hh], b, mode);
                        sa[t][hh] = acc;
                    }
                }
            }
            __syncthreads();
            for (int e = threadIdx.x; e < kTok * nh; e += blockDim.x) {
                const int hh = e / kTok, t = e % kTok;
                if (t < len)
                    gamma[(int64_t)(h0 + hh) * tokens + t0 + t] = sa[t][hh];
            }
        }
    }
}

// Documents by decreasing length (ties: lower index first).  The kernels
// that give one CTA to a whole document take documents in this order, so
// the longest chains start first.  One CTA; each thread ranks its documents
// against all others.
__global__ void __launch_bounds__(1024)
doc_order_kernel(const int32_t *__restrict__ cu, int n_docs, int32_t *__restrict__ order)
{
    for (int n = threadIdx.x; n < n_docs; n += blockDim.x) {
        const int64_t ln = (int64_t)cu[n + 1] - cu[n];
        int rank = 0;
        for (int m = 0; m < n_docs; ++m) {
            const int64_t lm = (int64_t)cu[m + 1] - cu[m];
            rank += (lm > ln || (lm == ln && m < n)) ? 1 : 0;
        }
        order[rank] = n;
    }
}

cudaError_t launch_doc_order(const Problem &p, int32_t *order)
{
    if (p.cu == nullptr || p.n_docs <= 1)
        return cudaSuccess;
    doc_order_kernel<<<1, 1024, 0, p.stream>>>(p.cu, p.n_docs, order);
    return cudaGetLastError();
}

cudaError_t launch_decay(const Problem &p, const float *a, float *gamma, float *dfac)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    // slabs per document: exact for fixed-length inputs; packed documents
    // spread over a grid sized for the average length (grid-stride inside).
    int64_t per_doc = p.cu ? (p.tokens / p.n_docs + kTok - 1) / kTok + 1 : (p.T + kTok - 1) / kTok;
    per_doc = per_doc < 1 ? 1 : (per_doc > 65535 ? 65535 : per_doc);
    dim3 grid((unsigned)per_doc, (unsigned)p.n_docs);
    decay_kernel<<<grid, 256, 0, p.stream>>>(a, p.b, p.mode, p.cu, p.n_docs, p.T, p.tokens, p.H,
                                             gamma, dfac, p.st);
    return cudaGetLastError();
}

}  // namespace bdla
