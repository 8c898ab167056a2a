// Recurrent decode step: one new token per sequence against its resident
// state, the inference side of the long-context stages the pages describe
// ("Engineering Long-Context Training for Trillion-Parameter MoE Models",
// sec. 2 and 3.3):
//     S <- e^{lambda} S + k v^T,   o = S^T q          (S updated in place)
// with lambda = b * sigmoid(a) (or -softplus(a)), the same recurrence the
// chunked forward evaluates tile by tile, so a chunked prefill's hT hands
// over to decode steps and back.
//
// The step reads and writes the fp32 state once (8 dk dv bytes per
// sequence-head) and touches a few hundred bytes of q, k, v, o: it is bound
// by HBM bandwidth, so it runs on CUDA cores with 16-byte coalesced state
// accesses.  One CTA per (sequence, head, 64-column state slice): 16 column
// groups of 4 floats x 16 row groups; o's column sums are reduced in shared
// memory.
#include "bdla_internal.h"

namespace bdla {

namespace {

constexpr int kDecThreads = 256;
constexpr int kCols = 64;           // state columns per CTA
constexpr int kColGroups = kCols / 4;
constexpr int kRowGroups = kDecThreads / kColGroups;   // 16

template <int DK>
__global__ void __launch_bounds__(kDecThreads)
decode_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
              const __nv_bfloat16 *__restrict__ v, const float *__restrict__ a, float b, int mode,
              float *__restrict__ state, void *__restrict__ o, int o_f32, int H, int dv)
{
    __shared__ float qs[DK], ks[DK];
    __shared__ float4 part[kRowGroups][kColGroups];
    const int tid = threadIdx.x;
    const int j0 = blockIdx.x * kCols, h = blockIdx.y, n = blockIdx.z;
    const int64_t unit = (int64_t)n * H + h;
    for (int i = tid; i < DK; i += kDecThreads) {
        qs[i] = bf2f(q[unit * DK + i]);
        ks[i] = bf2f(k[unit * DK + i]);
    }
    const float g = expf(log_decay(a[unit], b, mode));
    const int cg = tid % kColGroups, rg = tid / kColGroups;
    const int j = j0 + 4 * cg;
    const float4 vv = make_float4(bf2f(v[unit * dv + j]), bf2f(v[unit * dv + j + 1]),
                                  bf2f(v[unit * dv + j + 2]), bf2f(v[unit * dv + j + 3]));
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 *S = reinterpret_cast<float4 *>(state + unit * (int64_t)DK * dv + j);
    const int stride4 = dv / 4;   // one state row in float4
#pragma unroll
    for (int ii = 0; ii < DK / kRowGroups; ++ii) {
        const int i = rg + kRowGroups * ii;
        float4 s = S[(int64_t)i * stride4];
        const float ki = ks[i], qi = qs[i];
        s.x = fmaf(g, s.x, ki * vv.x);
        s.y = fmaf(g, s.y, ki * vv.y);
        s.z = fmaf(g, s.z, ki * vv.z);
        s.w = fmaf(g, s.w, ki * vv.w);
        S[(int64_t)i * stride4] = s;
        acc.x = fmaf(qi, s.x, acc.x);
        acc.y = fmaf(qi, s.y, acc.y);
        acc.z = fmaf(qi, s.z, acc.z);
        acc.w = fmaf(qi, s.w, acc.w);
    }
    part[rg][cg] = acc;
    __syncthreads();
    if (tid < kCols) {
        // column j0 + tid: sum over the row groups
        const int c4 = tid / 4, e = tid % 4;
        float sum = 0.0f;
#pragma unroll
        for (int r = 0; r < kRowGroups; ++r) {
            const float4 p = part[r][c4];
            sum += e == 0 ? p.x : (e == 1 ? p.y : (e == 2 ? p.z : p.w));
        }
        const int64_t off = unit * dv + j0 + tid;
        if (o_f32)
            reinterpret_cast<float *>(o)[off] = sum;
        else
            reinterpret_cast<__nv_bfloat16 *>(o)[off] = __float2bfloat16_rn(sum);
    }
}

}  // namespace

cudaError_t launch_decode(int B, int H, int dk, int dv, const __nv_bfloat16 *q,
                          const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *a, float b,
                          int mode, float *state, void *o, int o_f32, cudaStream_t stream)
{
    if (B <= 0)
        return cudaSuccess;
    dim3 grid(dv / kCols, H, B);
    if (dk == 64)
        decode_kernel<64><<<grid, kDecThreads, 0, stream>>>(q, k, v, a, b, mode, state, o, o_f32, H, dv);
    else
        decode_kernel<128><<<grid, kDecThreads, 0, stream>>>(q, k, v, a, b, mode, state, o, o_f32, H, dv);
    return cudaGetLastError();
}

}  // namespace bdla
