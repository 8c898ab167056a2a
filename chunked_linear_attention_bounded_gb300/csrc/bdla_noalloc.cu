// Forward entry point that allocates nothing and needs no workspace.
//
// Some callers cannot hand the library device memory for scratch: code that
// runs where cudaMalloc is forbidden or unavailable (inside a custom
// allocator's own callbacks, a runtime that hands out only fixed, pre-planned
// buffers for inputs and outputs, or a framework layer that must not touch
// the allocator on this path).  bdla_fwd_noalloc serves them: the per-token
// decay scratch (Gamma) and the device status word live in file-scope
// __device__ arrays of this library, so the caller passes only inputs and
// outputs.  The price is a fixed maximum problem size and a shared scratch.
//
// The arrays are part of the library's device image: every GPU that loads
// the library holds them (8 MiB + 256 B) until the process exits.
#include <mutex>

#include "bdla_internal.h"

namespace bdla {

namespace {

// Gamma for at most this many (token, head) pairs: 8 MiB of fp32.
constexpr size_t kNoAllocMaxTokenHeads = (size_t)1 << 21;

__device__ __align__(256) float g_noalloc_gamma[kNoAllocMaxTokenHeads];
__device__ __align__(256) DeviceStatus g_noalloc_status;

constexpr int kMaxDevices = 64;
struct NoAllocPtrs {
    float *gamma = nullptr;
    DeviceStatus *status = nullptr;
};
NoAllocPtrs g_noalloc_ptrs[kMaxDevices];
std::mutex g_noalloc_mu;

// Device addresses of the two arrays on the current device, looked up once
// per device (the host-side names are stand-ins, not device addresses).
bdla_status noalloc_setup(NoAllocPtrs &out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return BDLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocPtrs &p = g_noalloc_ptrs[dev];
    if (p.gamma == nullptr) {
        void *g = nullptr, *s = nullptr;
        if (cudaGetSymbolAddress(&g, g_noalloc_gamma) != cudaSuccess)
            return BDLA_ERR_CUDA;
        if (cudaGetSymbolAddress(&s, g_noalloc_status) != cudaSuccess)
            return BDLA_ERR_CUDA;
        p.gamma = static_cast<float *>(g);
        p.status = static_cast<DeviceStatus *>(s);
    }
    out = p;
    return BDLA_OK;
}

}  // namespace

}  // namespace bdla

using namespace bdla;

extern "C" bdla_status bdla_fwd_noalloc(const void *q, const void *k, const void *v, const float *a,
                                        float b, int chunk, const float *h0, void *o,
                                        bdla_dtype o_dtype, float *hT, bdla_dims d,
                                        bdla_decay_mode mode, void *stream)
{
    if (d.T < 0 || d.H < 1 || d.B < 1)
        return BDLA_ERR_SHAPE;
    if (d.dk != 64 && d.dk != 128)
        return BDLA_ERR_UNSUPPORTED;
    if (d.dv != 64 && d.dv != 128 && d.dv != 256)
        return BDLA_ERR_UNSUPPORTED;
    if (chunk != kChunk || (mode != BDLA_DECAY_BOUNDED_SIGMOID && mode != BDLA_DECAY_NEG_SOFTPLUS))
        return BDLA_ERR_UNSUPPORTED;
    if (mode == BDLA_DECAY_BOUNDED_SIGMOID &&
        (!isfinite(b) || b > 0.0f || (double)chunk * fabs((double)b) > 80.0))
        return BDLA_ERR_RANGE;
    const int64_t tokens = (int64_t)d.B * d.T;
    if ((size_t)tokens * (size_t)d.H > kNoAllocMaxTokenHeads)
        return BDLA_ERR_TOO_LARGE;
    if (tokens > 0 && (!q || !k || !v || !a || !o))
        return BDLA_ERR_NULL;
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(o) || !a16(a) || !a16(h0) || !a16(hT))
        return BDLA_ERR_ALIGN;
    if (o_dtype != BDLA_BF16 && o_dtype != BDLA_F32)
        return BDLA_ERR_UNSUPPORTED;

    NoAllocPtrs ptrs;
    const bdla_status s = noalloc_setup(ptrs);
    if (s != BDLA_OK)
        return s;

    Problem p;
    p.cu = nullptr;
    p.n_docs = d.B;
    p.T = d.T;
    p.tokens = tokens;
    p.H = d.H;
    p.dk = d.dk;
    p.dv = d.dv;
    p.b = b;
    p.mode = mode;
    p.st = ptrs.status;
    p.stream = reinterpret_cast<cudaStream_t>(stream);
    // the status word is shared by every call: start each call from zero
    if (cudaMemsetAsync(ptrs.status, 0, sizeof(DeviceStatus), p.stream) != cudaSuccess)
        return BDLA_ERR_CUDA;
    if (launch_decay(p, a, ptrs.gamma, nullptr) != cudaSuccess)
        return BDLA_ERR_CUDA;
    if (launch_fwd_sm100(p, static_cast<const __nv_bfloat16 *>(q),
                         static_cast<const __nv_bfloat16 *>(k),
                         static_cast<const __nv_bfloat16 *>(v), ptrs.gamma, h0, o,
                         o_dtype == BDLA_F32, hT, nullptr, 0, 0, SegPlan{}) != cudaSuccess)
        return BDLA_ERR_CUDA;
    return BDLA_OK;
}
