// Decay kernel: per-token log-decay and its tile-local inclusive cumsum.
//
// "Engineering Long-Context Training for Trillion-Parameter MoE Models",
// sec. 3.1: each chunk carries a per-position cumulative decay Gamma whose
// reciprocal normalises the in-chunk products; sec. 3.2: the log-decay is
// b * sigmoid(a) (bounded) instead of -softplus(a).  Gamma restarts at every
// doc-local 16-token tile, so with the bound it stays in [16 b, 0].
//
// The tensor-core forward forms Gamma from the logits itself; this kernel
// serves the kernels that read it from memory (the backward, which also
// reads d lambda / d a, the segment summaries, the tile-serial state pass,
// the checkpoint expansion) and the bdla_decay entry point.  It takes the
// same shuffle scan (tile_gamma) with the same lane of each token, so every
// kernel sees bitwise the same Gamma.
//
// One CTA handles 128 consecutive tokens of one document for 32 heads at a
// time: the [128 x heads] slab of logits is read coalesced (a is token-major)
// into shared memory, each warp scans 32 tokens (two tiles) of one head, and
// Gamma (and optionally d lambda / d a) is written head-major ([H][tokens])
// straight from the scan's registers, so a kernel reads one head's 128
// values as a single coalesced line.
#include "bdla_internal.h"

namespace bdla {

namespace {
constexpr int kTok = 128;   // tokens per slab (8 tiles)
constexpr int kHeads = 32;  // heads per pass
}

// One CTA per 128-token slab of a document (slab s of document n is slot
// floor(cu[n] / 128) + n + s, as the segment slots with one block per
// segment; other slots are gaps and return at once).
__global__ void __launch_bounds__(256)
decay_kernel(const float *__restrict__ a, float b, int mode, const int32_t *__restrict__ cu,
             int n_docs, int T, int64_t tokens, int H, float *__restrict__ gamma,
             float *__restrict__ dfac)
{
    __shared__ float sa[kTok][kHeads + 1];
    const SegSpan sl = seg_span(cu, T, tokens, n_docs, (int)blockIdx.x, 1);
    if (!sl.valid || sl.len <= 0)
        return;
    const int64_t t0 = sl.start;
    const int len = (int)sl.len;   // at most kTok
    for (int h0 = 0; h0 < H; h0 += kHeads) {
        const int nh = H - h0 < kHeads ? H - h0 : kHeads;
        if (h0 > 0)
            __syncthreads();   // the previous head group is done with sa
        for (int e = threadIdx.x; e < kTok * nh; e += blockDim.x) {
            const int t = e / nh, hh = e % nh;
            sa[t][hh] = t < len ? a[(t0 + t) * H + h0 + hh] : 0.0f;
        }
        __syncthreads();
        // thread <-> (head, token) with the token fastest: the head-major
        // stores are coalesced, and the 16 tokens of a tile sit in 16
        // consecutive lanes.  kTok * nh is a multiple of 32, so every warp
        // runs whole iterations (the scan needs all 32 lanes).
        for (int e = threadIdx.x; e < kTok * nh; e += blockDim.x) {
            const int hh = e / kTok, t = e % kTok;
            const float x = sa[t][hh];
            const float g = tile_gamma(t < len ? log_decay(x, b, mode) : 0.0f, (int)(threadIdx.x & 31));
            if (t < len) {
                const int64_t o = (int64_t)(h0 + hh) * tokens + t0 + t;
                gamma[o] = g;
                if (dfac != nullptr)
                    dfac[o] = log_decay_deriv(x, b, mode);
            }
        }
    }
}

// Checks the packed offsets (cu[0] = 0, non-decreasing, cu[n_docs] = tokens;
// the first bad document is reported as BDLA_ERR_DEVICE) and, when `order`
// is given, lists the documents by decreasing length (ties: lower index
// first).  The kernels that give one CTA to a whole document take documents
// in this order, so the longest chains start first.  One CTA; each thread
// ranks its documents against all others.
__global__ void __launch_bounds__(1024)
doc_check_kernel(const int32_t *__restrict__ cu, int n_docs, int64_t tokens, int32_t *__restrict__ order,
                 DeviceStatus *st)
{
    for (int n = threadIdx.x; n < n_docs; n += blockDim.x) {
        bool bad = cu[n + 1] < cu[n];
        if (n == 0 && cu[0] != 0)
            bad = true;
        if (n == n_docs - 1 && (int64_t)cu[n_docs] != tokens)
            bad = true;
        if (bad)
            set_status(st, BDLA_ERR_DEVICE, (unsigned)n);
    }
    if (order == nullptr)
        return;
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

cudaError_t launch_doc_check(const Problem &p, int32_t *order)
{
    if (p.cu == nullptr || p.n_docs <= 0)
        return cudaSuccess;
    doc_check_kernel<<<1, 1024, 0, p.stream>>>(p.cu, p.n_docs, p.tokens, p.n_docs > 1 ? order : nullptr, p.st);
    return cudaGetLastError();
}

cudaError_t launch_decay(const Problem &p, const float *a, float *gamma, float *dfac)
{
    if (p.n_docs <= 0 || p.tokens <= 0)
        return cudaSuccess;
    const int64_t slots = (p.tokens + kTok - 1) / kTok + p.n_docs;
    decay_kernel<<<(unsigned)slots, 256, 0, p.stream>>>(a, p.b, p.mode, p.cu, p.n_docs, p.T, p.tokens, p.H,
                                                        gamma, dfac);
    return cudaGetLastError();
}

}  // namespace bdla
