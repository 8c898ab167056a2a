// Tile-serial forward and backward on CUDA cores (fp32 arithmetic).
//
// One CTA walks one (document, head[, dv slice]) through its 16-token tiles
// ("Engineering Long-Context Training for Trillion-Parameter MoE Models",
// sec. 3.1: products inside a tile, recurrent state between tiles):
//   Gamma_t   tile-local inclusive cumsum of log-decay (decay kernel output,
//             head-major [H][tokens])
//   A_ts      = (q_t . k_s) e^{Gamma_t - Gamma_s},  s <= t in the tile
//   o_t       = e^{Gamma_t} S_in^T q_t + sum_s A_ts v_s
//   S_out     = e^{gamma} S_in + sum_s e^{gamma - Gamma_s} k_s v_s^T,
// gamma = Gamma at the tile's last token.  The backward walks the tiles in
// reverse with the state adjoint E (gradient w.r.t. the state at the end of
// the tile from all later tokens):
//   dq_t = e^{Gamma_t} S_in dO_t + sum_{s<=t} dP_ts k_s
//   dk_s = e^{gamma - Gamma_s} E v_s + sum_{t>=s} dP_ts q_t
//   dv_s = e^{gamma - Gamma_s} E^T k_s + sum_{t>=s} A_ts dO_t
//   E   <- e^{gamma} E + sum_t e^{Gamma_t} q_t dO_t^T
// with dP_ts = (dO_t . v_s) e^{Gamma_t - Gamma_s}.  The decay gradient uses
// pair sums W_ts = A_ts (dO_t . v_s) instead of the global reverse cumsum of
// q.dq - k.dk (which cancels catastrophically over long documents):
//   dlambda_r = sum_{u<r} X_u + sum_{t>=r} Y_t + e^{gamma} <S_in, E>
//   X_u = sum_{t>u} W_tu - sum_{s<u} W_us + k_u . dk_inter_u
//   Y_t = q_t . dq_inter_t
// (pairs across r inside the tile, pairs from this tile to earlier / later
// tiles, and pairs spanning the whole tile).
#include "bdla_internal.h"

namespace bdla {

namespace {

constexpr int kThreads = 256;
constexpr int kDvSlice = 64;  // forward dv slice per CTA

template <int DK>
struct FwdSmem {
    float S[DK][kDvSlice];
    float q[kChunk][DK + 1];
    float k[kChunk][DK + 1];
    float v[kChunk][kDvSlice];
    float A[kChunk][kChunk + 1];
    float g[kChunk];   // Gamma_t (padded rows repeat the last value)
    float wk[kChunk];  // e^{gamma - Gamma_s} (0 for padded rows)
};

template <int DK>
__global__ void __launch_bounds__(kThreads)
fwd_tile_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                const __nv_bfloat16 *__restrict__ v, const float *__restrict__ gamma,
                const int32_t *__restrict__ cu, int T, int64_t tokens, int H, int dv,
                const float *__restrict__ h0, void *__restrict__ o, int o_f32,
                float *__restrict__ hT, float *__restrict__ ckpt, int ckpt_stride,
                int64_t n_slots)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    FwdSmem<DK> &sm = *reinterpret_cast<FwdSmem<DK> *>(smem_raw);
    const int tid = threadIdx.x;
    const int j0 = blockIdx.x * kDvSlice;
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const DocSpan d = doc_span(cu, n, T);
    if (!doc_valid(d, tokens))
        return;
    const size_t sstride = (size_t)DK * dv;
    const int64_t unit = (int64_t)n * H + h;

    for (int e = tid; e < DK * kDvSlice; e += kThreads) {
        const int i = e / kDvSlice, j = e % kDvSlice;
        sm.S[i][j] = h0 ? h0[unit * sstride + (size_t)i * dv + j0 + j] : 0.0f;
    }
    const int64_t ntiles = (d.len + kChunk - 1) / kChunk;
    for (int64_t c = 0; c < ntiles; ++c) {
        const int64_t t0 = d.start + c * kChunk;
        const int m = (int)(d.len - c * kChunk < kChunk ? d.len - c * kChunk : kChunk);
        __syncthreads();  // previous tile finished with the smem tiles and S
        if (ckpt && ((c * kChunk) % ckpt_stride) == 0) {
            const int64_t slot = ckpt_slot(d.start, n, c * kChunk / ckpt_stride, ckpt_stride);
            float *dst = ckpt + ((size_t)h * n_slots + slot) * sstride;
            for (int e = tid; e < DK * kDvSlice; e += kThreads) {
                const int i = e / kDvSlice, j = e % kDvSlice;
                dst[(size_t)i * dv + j0 + j] = sm.S[i][j];
            }
        }
        for (int e = tid; e < kChunk * DK; e += kThreads) {
            const int t = e / DK, i = e % DK;
            float qv = 0.0f, kv = 0.0f;
            if (t < m) {
                const size_t off = ((size_t)(t0 + t) * H + h) * DK + i;
                qv = bf2f(q[off]);
                kv = bf2f(k[off]);
            }
            sm.q[t][i] = qv;
            sm.k[t][i] = kv;
        }
        for (int e = tid; e < kChunk * kDvSlice; e += kThreads) {
            const int t = e / kDvSlice, j = e % kDvSlice;
            sm.v[t][j] = t < m ? bf2f(v[((size_t)(t0 + t) * H + h) * dv + j0 + j]) : 0.0f;
        }
        if (tid < kChunk) {
            const int t = tid < m ? tid : m - 1;
            sm.g[tid] = gamma[(int64_t)h * tokens + t0 + t];
        }
        __syncthreads();
        if (tid < kChunk)
            sm.wk[tid] = tid < m ? expf(sm.g[m - 1] - sm.g[tid]) : 0.0f;
        {   // A_ts = (q_t . k_s) e^{Gamma_t - Gamma_s}, causal inside the tile
            const int t = tid / kChunk, s = tid % kChunk;
            float acc = 0.0f;
#pragma unroll 8
            for (int i = 0; i < DK; ++i)
                acc += sm.q[t][i] * sm.k[s][i];
            sm.A[t][s] = (s <= t && t < m) ? acc * expf(sm.g[t] - sm.g[s]) : 0.0f;
        }
        __syncthreads();
        {   // o_t = e^{Gamma_t} S_in^T q_t + sum_s A_ts v_s
            const int j = tid % kDvSlice;
            const int tb = tid / kDvSlice;
#pragma unroll
            for (int r = 0; r < kChunk / 4; ++r) {
                const int t = tb + 4 * r;
                float acc = 0.0f;
#pragma unroll 8
                for (int i = 0; i < DK; ++i)
                    acc += sm.q[t][i] * sm.S[i][j];
                float out = acc * expf(sm.g[t]);
#pragma unroll
                for (int s = 0; s < kChunk; ++s)
                    out += sm.A[t][s] * sm.v[s][j];
                if (o && t < m) {
                    const size_t off = ((size_t)(t0 + t) * H + h) * dv + j0 + j;
                    if (o_f32)
                        reinterpret_cast<float *>(o)[off] = out;
                    else
                        reinterpret_cast<__nv_bfloat16 *>(o)[off] = __float2bfloat16_rn(out);
                }
            }
        }
        __syncthreads();
        {   // S_out = e^{gamma} S_in + sum_s e^{gamma - Gamma_s} k_s v_s^T
            const int j = tid % kDvSlice;
            const int ib = tid / kDvSlice;
            const float eg = expf(sm.g[m - 1]);
            for (int i = ib; i < DK; i += kThreads / kDvSlice) {
                float acc = sm.S[i][j] * eg;
#pragma unroll
                for (int s = 0; s < kChunk; ++s)
                    acc += sm.wk[s] * sm.k[s][i] * sm.v[s][j];
                sm.S[i][j] = acc;
            }
        }
    }
    __syncthreads();
    if (hT) {
        for (int e = tid; e < DK * kDvSlice; e += kThreads) {
            const int i = e / kDvSlice, j = e % kDvSlice;
            hT[unit * sstride + (size_t)i * dv + j0 + j] = sm.S[i][j];
        }
    }
}

template <int DK, int DV>
struct BwdSmem {
    float E[DK][DV];
    float q[kChunk][DK + 1];
    float k[kChunk][DK + 1];
    float v[kChunk][DV + 1];
    float dO[kChunk][DV + 1];
    float dqi[kChunk][DK];  // e^{Gamma_t} S_in dO_t
    float dki[kChunk][DK];  // e^{gamma - Gamma_s} E v_s
    float red[kThreads / DV][kChunk][DV];
    float P[kChunk][kChunk + 1];   // A_ts
    float dP[kChunk][kChunk + 1];  // dP_ts
    float W[kChunk][kChunk + 1];   // A_ts * (dO_t . v_s)
    float g[kChunk];
    float wq[kChunk];   // e^{Gamma_t}
    float wk[kChunk];   // e^{gamma - Gamma_s}
    float Y[kChunk];    // q_t . dq_inter_t
    float KD[kChunk];   // k_u . dk_inter_u
    float se[kThreads / 32];
};

// Sum of 32 per-lane values across the warp, scattered so that lane l ends
// with the total of value l.
__device__ __forceinline__ float warp_reduce_scatter32(float (&vals)[32], int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? vals[i] : vals[i + off];
            const float keep = upper ? vals[i + off] : vals[i];
            vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return vals[0];
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads)
bwd_tile_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                const __nv_bfloat16 *__restrict__ v, const float *__restrict__ a,
                const float *__restrict__ gamma, const __nv_bfloat16 *__restrict__ dO,
                const float *__restrict__ dhT, const float *__restrict__ states, int64_t n_slots,
                const int32_t *__restrict__ cu, int T, int64_t tokens, int H, float b, int mode,
                float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dv,
                float *__restrict__ da, float *__restrict__ dh0)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<DK, DV> &sm = *reinterpret_cast<BwdSmem<DK, DV> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x;
    const int n = blockIdx.y;
    const DocSpan d = doc_span(cu, n, T);
    if (!doc_valid(d, tokens))
        return;
    const size_t sstride = (size_t)DK * DV;
    const int64_t unit = (int64_t)n * H + h;

    for (int e = tid; e < DK * DV; e += kThreads)
        (&sm.E[0][0])[e] = dhT ? dhT[unit * sstride + e] : 0.0f;

    const int64_t ntiles = (d.len + kChunk - 1) / kChunk;
    for (int64_t c = ntiles - 1; c >= 0; --c) {
        const int64_t t0 = d.start + c * kChunk;
        const int m = (int)(d.len - c * kChunk < kChunk ? d.len - c * kChunk : kChunk);
        const float *Sin = states + ((size_t)h * n_slots + ckpt_slot(d.start, n, c, kChunk)) * sstride;
        __syncthreads();
        for (int e = tid; e < kChunk * DK; e += kThreads) {
            const int t = e / DK, i = e % DK;
            float qv = 0.0f, kv = 0.0f;
            if (t < m) {
                const size_t off = ((size_t)(t0 + t) * H + h) * DK + i;
                qv = bf2f(q[off]);
                kv = bf2f(k[off]);
            }
            sm.q[t][i] = qv;
            sm.k[t][i] = kv;
        }
        for (int e = tid; e < kChunk * DV; e += kThreads) {
            const int t = e / DV, j = e % DV;
            float vv = 0.0f, gv = 0.0f;
            if (t < m) {
                const size_t off = ((size_t)(t0 + t) * H + h) * DV + j;
                vv = bf2f(v[off]);
                gv = bf2f(dO[off]);
            }
            sm.v[t][j] = vv;
            sm.dO[t][j] = gv;
        }
        if (tid < kChunk) {
            const int t = tid < m ? tid : m - 1;
            sm.g[tid] = gamma[(int64_t)h * tokens + t0 + t];
        }
        __syncthreads();
        const float gam = sm.g[m - 1];
        if (tid < kChunk) {
            sm.wq[tid] = tid < m ? expf(sm.g[tid]) : 0.0f;
            sm.wk[tid] = tid < m ? expf(gam - sm.g[tid]) : 0.0f;
        }
        {   // pair products of the tile
            const int t = tid / kChunk, s = tid % kChunk;
            float qk = 0.0f, ov = 0.0f;
#pragma unroll 8
            for (int i = 0; i < DK; ++i)
                qk += sm.q[t][i] * sm.k[s][i];
#pragma unroll 8
            for (int j = 0; j < DV; ++j)
                ov += sm.dO[t][j] * sm.v[s][j];
            const bool live = s <= t && t < m;
            const float w = live ? expf(sm.g[t] - sm.g[s]) : 0.0f;
            sm.P[t][s] = qk * w;
            sm.dP[t][s] = ov * w;
            sm.W[t][s] = (s < t && live) ? qk * w * ov : 0.0f;
        }
        __syncthreads();
        {   // rows of S_in and E: dq_inter, dk_inter, <S_in, E>
            float se = 0.0f;
            for (int i = warp; i < DK; i += kThreads / 32) {
                float vals[32];
#pragma unroll
                for (int x = 0; x < 32; ++x)
                    vals[x] = 0.0f;
#pragma unroll
                for (int r = 0; r < DV / 32; ++r) {
                    const int j = lane + 32 * r;
                    const float sij = Sin[(size_t)i * DV + j];
                    const float eij = sm.E[i][j];
                    se += sij * eij;
#pragma unroll
                    for (int t = 0; t < kChunk; ++t) {
                        vals[t] += sij * sm.dO[t][j];
                        vals[kChunk + t] += eij * sm.v[t][j];
                    }
                }
                const float tot = warp_reduce_scatter32(vals, lane);
                if (lane < kChunk)
                    sm.dqi[lane][i] = tot * sm.wq[lane];
                else
                    sm.dki[lane - kChunk][i] = tot * sm.wk[lane - kChunk];
            }
            se = warp_sum(se);
            if (lane == 0)
                sm.se[warp] = se;
        }
        {   // dv_inter partials: sum_i E[i][j] k_s[i]
            constexpr int parts = kThreads / DV;
            const int j = tid % DV, part = tid / DV;
            float acc[kChunk];
#pragma unroll
            for (int s = 0; s < kChunk; ++s)
                acc[s] = 0.0f;
            for (int i = part * (DK / parts); i < (part + 1) * (DK / parts); ++i) {
                const float eij = sm.E[i][j];
#pragma unroll
                for (int s = 0; s < kChunk; ++s)
                    acc[s] += eij * sm.k[s][i];
            }
#pragma unroll
            for (int s = 0; s < kChunk; ++s)
                sm.red[part][s][j] = acc[s];
        }
        __syncthreads();
        // outputs dv, dq, dk
        for (int e = tid; e < kChunk * DV; e += kThreads) {
            const int s = e / DV, j = e % DV;
            float inter = 0.0f;
#pragma unroll
            for (int p = 0; p < kThreads / DV; ++p)
                inter += sm.red[p][s][j];
            float acc = inter * sm.wk[s];
#pragma unroll
            for (int t = 0; t < kChunk; ++t)
                acc += sm.P[t][s] * sm.dO[t][j];
            if (s < m)
                dv[((size_t)(t0 + s) * H + h) * DV + j] = acc;
        }
        for (int e = tid; e < kChunk * DK; e += kThreads) {
            const int t = e / DK, i = e % DK;
            float aq = sm.dqi[t][i], ak = sm.dki[t][i];
#pragma unroll
            for (int s = 0; s < kChunk; ++s) {
                aq += sm.dP[t][s] * sm.k[s][i];
                ak += sm.dP[s][t] * sm.q[s][i];
            }
            if (t < m) {
                const size_t off = ((size_t)(t0 + t) * H + h) * DK + i;
                dq[off] = aq;
                dk[off] = ak;
            }
        }
        // Y_t = q_t . dq_inter_t and k_u . dk_inter_u: 32 dot products, 4 per warp
        for (int x = warp; x < 2 * kChunk; x += kThreads / 32) {
            const int t = x % kChunk;
            float acc = 0.0f;
            for (int i = lane; i < DK; i += 32)
                acc += x < kChunk ? sm.q[t][i] * sm.dqi[t][i] : sm.k[t][i] * sm.dki[t][i];
            acc = warp_sum(acc);
            if (lane == 0) {
                if (x < kChunk)
                    sm.Y[t] = acc;
                else
                    sm.KD[t] = acc;
            }
        }
        __syncthreads();
        if (warp == 0) {
            float X = 0.0f, Y = 0.0f;
            if (lane < kChunk) {
                float row = 0.0f, col = 0.0f;
#pragma unroll
                for (int s = 0; s < kChunk; ++s) {
                    row += sm.W[lane][s];
                    col += sm.W[s][lane];
                }
                X = col - row + sm.KD[lane];
                Y = sm.Y[lane];
            }
            float se = 0.0f;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w)
                se += sm.se[w];
            const float C = expf(gam) * se;
            // exclusive prefix of X and inclusive suffix of Y over the tile
            float pre = 0.0f, suf = 0.0f;
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
                const float xu = __shfl_sync(0xffffffffu, X, u);
                const float yu = __shfl_sync(0xffffffffu, Y, u);
                if (u < lane)
                    pre += xu;
                if (u >= lane)
                    suf += yu;
            }
            if (lane < m) {
                const int64_t idx = (t0 + lane) * H + h;
                const float dl = pre + suf + C;
                da[idx] = dl * log_decay_deriv(a[idx], b, mode);
            }
        }
        // E <- e^{gamma} E + sum_t e^{Gamma_t} q_t dO_t^T   (all reads of E are done)
        {
            const float eg = expf(gam);
            for (int e = tid; e < DK * DV; e += kThreads) {
                const int i = e / DV, j = e % DV;
                float acc = sm.E[i][j] * eg;
#pragma unroll
                for (int t = 0; t < kChunk; ++t)
                    acc += sm.wq[t] * sm.q[t][i] * sm.dO[t][j];
                sm.E[i][j] = acc;
            }
        }
    }
    __syncthreads();
    if (dh0)
        for (int e = tid; e < DK * DV; e += kThreads)
            dh0[unit * sstride + e] = (&sm.E[0][0])[e];
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_fwd_tile(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                            const __nv_bfloat16 *v, const float *gamma, const float *h0, void *o,
                            int o_f32, float *hT, float *ckpt, int ckpt_stride)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    dim3 grid(p.dv / kDvSlice, p.H, p.n_docs);
    const int64_t n_slots = ckpt ? ckpt_slots(p, ckpt_stride) : 0;
    cudaError_t err;
    if (p.dk == 64) {
        auto kern = fwd_tile_kernel<64>;
        if ((err = set_smem(kern, sizeof(FwdSmem<64>))) != cudaSuccess)
            return err;
        kern<<<grid, kThreads, sizeof(FwdSmem<64>), p.stream>>>(q, k, v, gamma, p.cu, p.T, p.tokens,
            p.H, p.dv, h0, o, o_f32, hT, ckpt, ckpt_stride, n_slots);
    } else {
        auto kern = fwd_tile_kernel<128>;
        if ((err = set_smem(kern, sizeof(FwdSmem<128>))) != cudaSuccess)
            return err;
        kern<<<grid, kThreads, sizeof(FwdSmem<128>), p.stream>>>(q, k, v, gamma, p.cu, p.T,
            p.tokens, p.H, p.dv, h0, o, o_f32, hT, ckpt, ckpt_stride, n_slots);
    }
    return cudaGetLastError();
}

template <int DK, int DV>
static cudaError_t launch_bwd_tile_t(const Problem &p, const __nv_bfloat16 *q,
                                     const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                     const float *a, const float *gamma, const __nv_bfloat16 *dO,
                                     const float *dhT, const float *states, float *dq, float *dk,
                                     float *dv, float *da, float *dh0)
{
    auto kern = bwd_tile_kernel<DK, DV>;
    cudaError_t err = set_smem(kern, sizeof(BwdSmem<DK, DV>));
    if (err != cudaSuccess)
        return err;
    dim3 grid(p.H, p.n_docs);
    kern<<<grid, kThreads, sizeof(BwdSmem<DK, DV>), p.stream>>>(q, k, v, a, gamma, dO, dhT, states,
        ckpt_slots(p, kChunk), p.cu, p.T, p.tokens, p.H, p.b, p.mode, dq, dk, dv, da, dh0);
    return cudaGetLastError();
}

cudaError_t launch_bwd_tile(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                            const __nv_bfloat16 *v, const float *a, const float *gamma,
                            const __nv_bfloat16 *dO, const float *dhT, const float *states,
                            float *dq, float *dk, float *dv, float *da, float *dh0)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
#define BDLA_BWD_CASE(DK_, DV_)                                                                    \
    if (p.dk == DK_ && p.dv == DV_)                                                                \
        return launch_bwd_tile_t<DK_, DV_>(p, q, k, v, a, gamma, dO, dhT, states, dq, dk, dv, da,  \
                                           dh0);
    BDLA_BWD_CASE(64, 64)
    BDLA_BWD_CASE(64, 128)
    BDLA_BWD_CASE(64, 256)
    BDLA_BWD_CASE(128, 64)
    BDLA_BWD_CASE(128, 128)
    BDLA_BWD_CASE(128, 256)
#undef BDLA_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace bdla
