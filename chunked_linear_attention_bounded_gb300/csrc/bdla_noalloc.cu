// Forward entry point that allocates nothing and needs no workspace.
//
// Some callers cannot hand the library device memory for scratch: code that
// runs where cudaMalloc is forbidden or unavailable (inside a custom
// allocator's own callbacks, a runtime that hands out only fixed, pre-planned
// buffers for inputs and outputs, or a framework layer that must not touch
// the allocator on this path).  bdla_fwd_noalloc serves them: the forward
// kernel forms the decay cumsum from the logits itself, and the device status
// word lives in a file-scope __device__ variable of this library, so the
// caller passes only inputs and outputs.
//
// The status word is part of the library's device image: every GPU that
// loads the library holds it (256 B) until the process exits.  It keeps the
// first device-side error of any call (it starts at zero with the image)
// until bdla_noalloc_read_status reads and clears it.
#include <mutex>

#include "bdla_internal.h"

namespace bdla {

namespace {

__device__ __align__(256) DeviceStatus g_noalloc_status;

constexpr int kMaxDevices = 64;
struct NoAllocPtrs {
    DeviceStatus *status = nullptr;
};
NoAllocPtrs g_noalloc_ptrs[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the status word on the current device, looked up once
// per device (the host-side name is a stand-in, not a device address).
bdla_status noalloc_setup(NoAllocPtrs &out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return BDLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocPtrs &p = g_noalloc_ptrs[dev];
    if (p.status == nullptr) {
        void *s = nullptr;
        if (cudaGetSymbolAddress(&s, g_noalloc_status) != cudaSuccess)
            return BDLA_ERR_CUDA;
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
    bdla_status s = check_dims(d, false, 0);
    if (s != BDLA_OK)
        return s;
    if ((s = check_decay(b, chunk, mode)) != BDLA_OK)
        return s;
    // token coordinates of the kernels' tensor copies are 32-bit
    const int64_t tokens = (int64_t)d.B * d.T;
    if (tokens > (int64_t)INT32_MAX)
        return BDLA_ERR_TOO_LARGE;
    if (tokens > 0 && (!q || !k || !v || !a || !o))
        return BDLA_ERR_NULL;
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(o) || !a16(a) || !a16(h0) || !a16(hT))
        return BDLA_ERR_ALIGN;
    if (o_dtype != BDLA_BF16 && o_dtype != BDLA_F32)
        return BDLA_ERR_DTYPE;

    NoAllocPtrs ptrs;
    if ((s = noalloc_setup(ptrs)) != BDLA_OK)
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
    // the first device-side error of any call stays in the status word until
    // bdla_noalloc_read_status reads and clears it
    p.st = ptrs.status;
    p.stream = reinterpret_cast<cudaStream_t>(stream);
    if (launch_fwd_sm100(p, static_cast<const __nv_bfloat16 *>(q),
                         static_cast<const __nv_bfloat16 *>(k),
                         static_cast<const __nv_bfloat16 *>(v), a, h0, o,
                         o_dtype == BDLA_F32, hT, nullptr, 0, 0, SegPlan{}) != cudaSuccess)
        return BDLA_ERR_CUDA;
    return BDLA_OK;
}

extern "C" bdla_status bdla_noalloc_read_status(void *stream)
{
    NoAllocPtrs ptrs;
    const bdla_status s = noalloc_setup(ptrs);
    if (s != BDLA_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return BDLA_ERR_CUDA;
    // a plain copy out of the library's own array: no allocation, and the
    // stream is idle, so no call is writing the word meanwhile
    unsigned int code = 0;
    if (cudaMemcpy(&code, &ptrs.status->code, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
        return BDLA_ERR_CUDA;
    if (code != 0 && cudaMemset(ptrs.status, 0, sizeof(DeviceStatus)) != cudaSuccess)
        return BDLA_ERR_CUDA;
    return static_cast<bdla_status>(code);
}
