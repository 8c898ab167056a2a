// Decay kernel: per-token log-decay and its tile-local inclusive cumsum.
//
// "Engineering Long-Context Training for Trillion-Parameter MoE Models",
// sec. 3.1: each chunk carries a per-position cumulative decay Gamma whose
// reciprocal normalises the in-chunk products; sec. 3.2: the log-decay is
// b * sigmoid(a) (bounded) instead of -softplus(a).  Gamma restarts at every
// doc-local 16-token tile, so with the bound it stays in [16 b, 0].
#include "bdla_internal.h"

namespace bdla {

__global__ void __launch_bounds__(256)
decay_kernel(const float *__restrict__ a, float b, int mode, const int32_t *__restrict__ cu,
             int n_docs, int T, int64_t tokens, int H, float *__restrict__ gamma,
             DeviceStatus *st)
{
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
    const int64_t ntiles = (d.len + kChunk - 1) / kChunk;
    const int64_t work = ntiles * H;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < work;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int h = (int)(idx % H);
        const int64_t c = idx / H;
        const int64_t t0 = d.start + c * kChunk;
        const int m = (int)(d.len - c * kChunk < kChunk ? d.len - c * kChunk : kChunk);
        float acc = 0.0f;
        for (int i = 0; i < m; ++i) {
            acc += log_decay(a[(t0 + i) * H + h], b, mode);
            gamma[(t0 + i) * H + h] = acc;
        }
    }
}

cudaError_t launch_decay(const Problem &p, const float *a, float *gamma)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    const int64_t max_tiles = p.cu ? (p.tokens + kChunk - 1) / kChunk + 1 : (p.T + kChunk - 1) / kChunk;
    int64_t gx = (max_tiles * p.H + 255) / 256;
    if (p.cu)  // document lengths are on the device: spread each document over a fixed grid
        gx = (gx + p.n_docs - 1) / p.n_docs + 1;
    gx = gx < 1 ? 1 : (gx > 4096 ? 4096 : gx);
    dim3 grid((unsigned)gx, (unsigned)p.n_docs);
    decay_kernel<<<grid, 256, 0, p.stream>>>(a, p.b, p.mode, p.cu, p.n_docs, p.T, p.tokens, p.H,
                                             gamma, p.st);
    return cudaGetLastError();
}

}  // namespace bdla
