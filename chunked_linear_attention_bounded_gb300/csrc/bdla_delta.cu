// Gated delta rule with the bounded log-decay: the "Delta Net-style"
// structure that "Engineering Long-Context Training for Trillion-Parameter MoE
// Models: Three Key Breakthroughs" (sec. 3.1) names beside linear attention,
// with the same decay parameterisation (sec. 3.2).  The rule is the published
// gated delta rule ("Gated Delta Networks: Improving Mamba2 with Delta Rule",
// 2024) for a dk x dv state read by o = S^T q:
//     S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   g_t = e^{lambda_t}.
//
// Multiplying out the projection gives gated linear attention with the
// pseudo-values delta_t = beta_t (v_t - g_t S_{t-1}^T k_t).  Inside a 16-token
// tile (Gamma the tile-local cumsum of lambda, gamma its total, S_0 the state
// before the tile) they solve one unit lower-triangular system (the WY / UT
// form of the rule):
//   L     = diag(beta) strict_tril((K K^T) o E),   E_ts = e^{Gamma_t - Gamma_s} <= 1
//   T     = (I + L)^{-1} diag(beta)
//   Delta = T V - (T diag(e^{Gamma}) K) S_0
//   O     = diag(e^{Gamma}) Q S_0 + tril((Q K^T) o E) Delta
//   S_C   = e^{gamma} S_0 + K^T (diag(e^{gamma - Gamma}) Delta)
// Every decay factor is at most 1.  The 16 x 16 products Q K^T and K K^T are
// taken from the exact bf16 inputs and the pair factors applied to their fp32
// values; the solve, T V, T diag(e^Gamma) K and the causal product with Delta
// run in fp32 on CUDA cores (all contractions of length 16); the three
// products with the state (Q S_0, W S_0, K^T Delta) are bf16 warp MMAs (wmma
// 16x16x16, fp32 accumulate) against a bf16 copy of the fp32 state.  Folding
// e^{-Gamma} into bf16 key operands, as the linear-attention kernels do, is
// legal under the bound here too, but the rounding then passes through the
// triangular solve into every output (about 3e-3 relative error on o in an
// fp32 simulation, against 1e-4 this way).
#include <mma.h>

#include "bdla_internal.h"

namespace bdla {

namespace {

using namespace nvcuda;

constexpr int kT = kChunk;       // 16-token tile
constexpr int kDT = 256;         // forward threads (8 warps)
constexpr int kDvs = 64;         // value columns per forward CTA

template <int DK>
struct DeltaFwdSmem {
    static constexpr int LK = DK + 8;     // padded rows (bf16), so consecutive rows change banks
    static constexpr int LV = kDvs + 8;
    static constexpr int LF = kDvs + 4;   // padded rows (fp32)
    static constexpr int LS = kT + 4;     // 16 x 16 fp32 tiles
    float S32[DK * LF];                   // fp32 state (this CTA's value columns)
    __nv_bfloat16 S16[DK * LV];           // its bf16 copy (MMA operand)
    __nv_bfloat16 Q[kT * LK], K[kT * LK], Wb[kT * LK];
    __nv_bfloat16 V[kT * LV], Dh[kT * LV];
    float QK[kT * LS], KK[kT * LS], Tm[kT * LS];
    float QS[kT * LF], WS[kT * LF], Dl[kT * LF];
    float G[kT], eG[kT], beta[kT];
};

// 4 / 8 consecutive bf16 of a shared row as floats, by one 8- / 16-byte load
// (a bf16 is the upper half of the fp32 with the same bits).
__device__ __forceinline__ void ld_bf4(const __nv_bfloat16 *p, float (&x)[4])
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void ld_bf8(const __nv_bfloat16 *p, float (&x)[8])
{
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// C[16][16] (ld LS) = A B^T for two [16][DK] bf16 tiles (ld LK); one warp.
template <int DK, int LK, int LS>
__device__ __forceinline__ void gram16(float *C, const __nv_bfloat16 *A, const __nv_bfloat16 *B)
{
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
    wmma::fill_fragment(acc, 0.0f);
#pragma unroll
    for (int kk = 0; kk < DK / 16; ++kk) {
        wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
        wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
        wmma::load_matrix_sync(fa, A + 16 * kk, LK);
        wmma::load_matrix_sync(fb, B + 16 * kk, LK);   // B^T[kk][s] = B[s][kk]
        wmma::mma_sync(acc, fa, fb, acc);
    }
    wmma::store_matrix_sync(C, acc, LS, wmma::mem_row_major);
}

// C[16][16 ni .. +15] (ld LF) = A S for A [16][DK] bf16 (ld LK) and the bf16
// state S [DK][kDvs] (ld LV); one warp, one 16-column panel.
template <int DK, int LK, int LV, int LF>
__device__ __forceinline__ void times_state(float *C, const __nv_bfloat16 *A, const __nv_bfloat16 *S, int ni)
{
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
    wmma::fill_fragment(acc, 0.0f);
#pragma unroll
    for (int kk = 0; kk < DK / 16; ++kk) {
        wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
        wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
        wmma::load_matrix_sync(fa, A + 16 * kk, LK);
        wmma::load_matrix_sync(fb, S + 16 * kk * LV + 16 * ni, LV);
        wmma::mma_sync(acc, fa, fb, acc);
    }
    wmma::store_matrix_sync(C + 16 * ni, acc, LF, wmma::mem_row_major);
}

// One CTA per (64-column value slice, head, document), tiles in order.
// With `states` given the bf16 state before every tile goes there
// ([H][slots][DK][dv], slot = floor(doc_start / 16) + n + tile); STATES: no q
// and no output (the backward's own states pass).
template <int DK, bool STATES>
__global__ void __launch_bounds__(kDT)
delta_fwd_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                 const __nv_bfloat16 *__restrict__ v, const float *__restrict__ a,
                 const float *__restrict__ beta, float b, int mode, const int32_t *__restrict__ cu, int T,
                 int64_t tokens, int H, int dv, const float *__restrict__ h0, void *__restrict__ o, int o_f32,
                 float *__restrict__ hT, __nv_bfloat16 *__restrict__ states, int64_t n_slots, DeviceStatus *st,
               const int32_t *__restrict__ order)
{
    using Sm = DeltaFwdSmem<DK>;
    constexpr int LK = Sm::LK, LV = Sm::LV, LF = Sm::LF, LS = Sm::LS;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = blockIdx.x * kDvs, h = blockIdx.y, n = order != nullptr ? order[blockIdx.z] : (int)blockIdx.z;
    const DocSpan d = doc_span(cu, n, T);
    if (!doc_valid(d, tokens)) {
        if (tid == 0)
            set_status(st, BDLA_ERR_DEVICE, (unsigned)n);
        return;
    }
    const int64_t unit = (int64_t)n * H + h;
    const size_t sstride = (size_t)DK * dv;
    for (int e = tid; e < DK * kDvs; e += kDT) {
        const int i = e / kDvs, j = e % kDvs;
        const float x = h0 != nullptr ? h0[unit * sstride + (size_t)i * dv + j0 + j] : 0.0f;
        sm.S32[i * LF + j] = x;
        sm.S16[i * LV + j] = __float2bfloat16_rn(x);
    }
    __syncthreads();
    const int ntile = (int)((d.len + kT - 1) / kT);
    for (int c = 0; c < ntile; ++c) {
        const int64_t t0 = d.start + (int64_t)c * kT;
        const int nv = (int)(d.len - (int64_t)c * kT < kT ? d.len - (int64_t)c * kT : kT);
        // ---- the tile's inputs, the decay cumsum and the write strengths
        if (states != nullptr) {   // the state before this tile
            __nv_bfloat16 *dst = states + ((size_t)h * n_slots + (size_t)(d.start / kT + n + c)) * sstride + j0;
            for (int e = tid; e < DK * kDvs / 8; e += kDT) {
                const int row = e / (kDvs / 8), col = (e % (kDvs / 8)) * 8;
                *reinterpret_cast<uint4 *>(dst + (size_t)row * dv + col) =
                    *reinterpret_cast<const uint4 *>(sm.S16 + row * LV + col);
            }
        }
        {   // q, k and the value slice: every global load before the shared stores
            static_assert(kT * DK / 8 <= kDT && kT * kDvs / 8 <= kDT, "one chunk per thread");
            const uint4 z4 = make_uint4(0, 0, 0, 0);
            uint4 qv = z4, kv = z4, vv = z4;
            const int tk = tid / (DK / 8), ck = (tid % (DK / 8)) * 8;
            const int tq = tid / (kDvs / 8), cv = (tid % (kDvs / 8)) * 8;
            const bool hk = tid < kT * DK / 8, hv = tid < kT * kDvs / 8;
            if (hk && tk < nv) {
                const size_t off = ((size_t)(t0 + tk) * H + h) * DK + ck;
                if (!STATES)
                    qv = *reinterpret_cast<const uint4 *>(q + off);
                kv = *reinterpret_cast<const uint4 *>(k + off);
            }
            if (hv && tq < nv)
                vv = *reinterpret_cast<const uint4 *>(v + ((size_t)(t0 + tq) * H + h) * dv + j0 + cv);
            if (hk) {
                if (!STATES)
                    *reinterpret_cast<uint4 *>(sm.Q + tk * LK + ck) = qv;
                *reinterpret_cast<uint4 *>(sm.K + tk * LK + ck) = kv;
            }
            if (hv)
                *reinterpret_cast<uint4 *>(sm.V + tq * LV + cv) = vv;
        }
        if (warp == 0) {
            const bool in = lane < nv;
            float x = in ? log_decay(a[(t0 + lane) * H + h], b, mode) : 0.0f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {   // inclusive scan over the tile
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off)
                    x += y;
            }
            if (lane < kT) {
                sm.G[lane] = x;
                sm.eG[lane] = expf(x);
                sm.beta[lane] = in ? beta[(t0 + lane) * H + h] : 0.0f;
            }
        }
        __syncthreads();
        // ---- products from the exact inputs: K K^T, Q K^T, Q S_0
        if (warp == 0) {
            gram16<DK, LK, LS>(sm.KK, sm.K, sm.K);
        } else if (!STATES) {
            if (warp == 1)
                gram16<DK, LK, LS>(sm.QK, sm.Q, sm.K);
            for (int ni = warp - 2; ni < kDvs / 16; ni += kDT / 32 - 2)
                if (ni >= 0)
                    times_state<DK, LK, LV, LF>(sm.QS, sm.Q, sm.S16, ni);
        }
        __syncthreads();
        // ---- pair factors: L = beta_t (k_t.k_s) E_ts (s < t), P = (q_t.k_s) E_ts (s <= t)
        for (int e = tid; e < kT * kT; e += kDT) {
            const int t = e / kT, s = e % kT;
            const float E = s <= t ? expf(sm.G[t] - sm.G[s]) : 0.0f;
            sm.KK[t * LS + s] = s < t ? sm.beta[t] * sm.KK[t * LS + s] * E : 0.0f;
            if (!STATES)
                sm.QK[t * LS + s] *= E;
        }
        __syncthreads();
        // ---- T = (I + L)^{-1} diag(beta): lane j solves column j by forward substitution
        if (warp == 0 && lane < kT) {
            const int j = lane;
            float x[kT];
#pragma unroll
            for (int t = 0; t < kT; ++t) {
                float acc = 0.0f;
#pragma unroll
                for (int s = 0; s < t; ++s)
                    acc += sm.KK[t * LS + s] * x[s];
                x[t] = t < j ? 0.0f : (t == j ? sm.beta[j] : -acc);
                sm.Tm[t * LS + j] = x[t];
            }
        }
        __syncthreads();
        // ---- W = T diag(e^{Gamma}) K (bf16 operand), U = T V (fp32, into Dl); 4
        //      columns per item, T lower-triangular (s <= t)
        for (int e = tid; e < kT * DK / 4; e += kDT) {
            const int t = e / (DK / 4), i4 = (e % (DK / 4)) * 4;
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int s = 0; s <= t; ++s) {
                const float c = sm.Tm[t * LS + s] * sm.eG[s];
                float x[4];
                ld_bf4(sm.K + s * LK + i4, x);
#pragma unroll
                for (int y = 0; y < 4; ++y)
                    acc[y] += c * x[y];
            }
            *reinterpret_cast<uint2 *>(sm.Wb + t * LK + i4) = make_uint2(pack2_bf16(acc[0], acc[1]), pack2_bf16(acc[2], acc[3]));
        }
        for (int e = tid; e < kT * kDvs / 4; e += kDT) {
            const int t = e / (kDvs / 4), j4 = (e % (kDvs / 4)) * 4;
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int s = 0; s <= t; ++s) {
                const float c = sm.Tm[t * LS + s];
                float x[4];
                ld_bf4(sm.V + s * LV + j4, x);
#pragma unroll
                for (int y = 0; y < 4; ++y)
                    acc[y] += c * x[y];
            }
            *reinterpret_cast<float4 *>(sm.Dl + t * LF + j4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
        __syncthreads();
        // ---- W S_0
        for (int ni = warp; ni < kDvs / 16; ni += kDT / 32)
            times_state<DK, LK, LV, LF>(sm.WS, sm.Wb, sm.S16, ni);
        __syncthreads();
        // ---- Delta = U - W S_0 and its state-update operand diag(e^{gamma - Gamma}) Delta
        const float gam = sm.G[kT - 1];
        for (int e = tid; e < kT * (kDvs / 8); e += kDT) {
            const int t = e >> 3, c8 = (e & 7) * 8;   // one row segment of 8 per item
            const float w = expf(gam - sm.G[t]);
            __align__(16) __nv_bfloat16 h8[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float dl = sm.Dl[t * LF + c8 + x] - sm.WS[t * LF + c8 + x];
                sm.Dl[t * LF + c8 + x] = dl;
                h8[x] = __float2bfloat16_rn(w * dl);
            }
            *reinterpret_cast<uint4 *>(sm.Dh + t * LV + c8) = *reinterpret_cast<const uint4 *>(h8);
        }
        __syncthreads();
        // ---- O = diag(e^{Gamma}) Q S_0 + P Delta (rows t < nv)
        for (int e = tid; !STATES && e < kT * (kDvs / 8); e += kDT) {
            const int t = e >> 3, c8 = (e & 7) * 8;
            float out[8];
            const float eg = sm.eG[t];
#pragma unroll
            for (int x = 0; x < 8; ++x)
                out[x] = eg * sm.QS[t * LF + c8 + x];
            for (int s = 0; s <= t; ++s) {
                const float p = sm.QK[t * LS + s];
                const float4 d0 = *reinterpret_cast<const float4 *>(sm.Dl + s * LF + c8);
                const float4 d1 = *reinterpret_cast<const float4 *>(sm.Dl + s * LF + c8 + 4);
                out[0] += p * d0.x; out[1] += p * d0.y; out[2] += p * d0.z; out[3] += p * d0.w;
                out[4] += p * d1.x; out[5] += p * d1.y; out[6] += p * d1.z; out[7] += p * d1.w;
            }
            if (t < nv) {
                const size_t off = ((size_t)(t0 + t) * H + h) * dv + j0 + c8;
                if (o_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(o) + off);
                    dst[0] = make_float4(out[0], out[1], out[2], out[3]);
                    dst[1] = make_float4(out[4], out[5], out[6], out[7]);
                } else {
                    __align__(16) __nv_bfloat16 w8[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        w8[x] = __float2bfloat16_rn(out[x]);
                    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(o) + off) =
                        *reinterpret_cast<const uint4 *>(w8);
                }
            }
        }
        // ---- S <- e^{gamma} S + K^T (diag(e^{gamma - Gamma}) Delta)
        {
            const float eg = expf(gam);
            for (int tile = warp; tile < (DK / 16) * (kDvs / 16); tile += kDT / 32) {
                const int mi = tile / (kDvs / 16), ni = tile % (kDvs / 16);
                wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
                wmma::load_matrix_sync(acc, sm.S32 + 16 * mi * LF + 16 * ni, LF, wmma::mem_row_major);
#pragma unroll
                for (int x = 0; x < acc.num_elements; ++x)
                    acc.x[x] *= eg;
                wmma::load_matrix_sync(fa, sm.K + 16 * mi, LK);     // A[i][t] = K[t][16 mi + i]
                wmma::load_matrix_sync(fb, sm.Dh + 16 * ni, LV);    // B[t][j] = Dh[t][16 ni + j]
                wmma::mma_sync(acc, fa, fb, acc);
                wmma::store_matrix_sync(sm.S32 + 16 * mi * LF + 16 * ni, acc, LF, wmma::mem_row_major);
            }
        }
        __syncthreads();
        for (int e = tid; e < DK * kDvs; e += kDT) {
            const int i = e / kDvs, j = e % kDvs;
            sm.S16[i * LV + j] = __float2bfloat16_rn(sm.S32[i * LF + j]);
        }
        __syncthreads();
    }
    if (hT != nullptr)
        for (int e = tid; e < DK * kDvs; e += kDT) {
            const int i = e / kDvs, j = e % kDvs;
            hT[unit * sstride + (size_t)i * dv + j0 + j] = sm.S32[i * LF + j];
        }
}

// ---------------------------------------------------------------- backward
// Reverse walk over a document's tiles, one CTA per (head, document) holding
// all value columns, with the adjoint D of the state at the tile end kept in
// accumulator fragments (warp w owns the 16 x 16 tiles w, w + 8, ...).  Per
// tile, with S_0 the bf16 state before it (states pass), the forward
// quantities are recomputed (E, P, L, T, W, U, Delta) and then
//   dDelta = P^T dO + diag(w) K D                     (w_t = e^{gamma - Gamma_t})
//   dP     = tril(dO Delta^T),  dW = -dDelta S_0^T,  dT = dDelta V^T + dW (diag(e^Gamma) K)^T
//   dv     = T^T dDelta,        dM = T^T dW
//   X      = (I + L)^{-T} dT,   dL = -strict_tril(X T^T),  dbeta_t = X_tt + sum_s dL_ts (K K^T o E)_ts
//   dq     = diag(e^Gamma) dO S_0^T + (dP o E) K
//   dk     = (dP o E)^T Q + (diag(w) Delta) D^T + diag(e^Gamma) dM + (dA + dA^T) K,
//            dA = diag(beta) (dL o E)
//   D     <- e^{gamma} D + Q^T diag(e^Gamma) dO - W^T dDelta
// and the decay gradient as sums that never subtract large equal terms: over
// the pairs s < r <= t of the pair terms dP o P + dL o L, suffix sums of the
// terms through e^{Gamma_t}, prefix sums of the terms through w_t, and the
// state term e^{gamma} <S_0, D>.  Products with the state or the adjoint are
// bf16 warp MMAs; the 16-long contractions are fp32 on CUDA cores.
constexpr int kBT = 512;   // backward threads (16 warps)

template <int DK, int DV>
struct DeltaBwdSmem {
    static constexpr int LK = DK + 8, LV = DV + 8;
    static constexpr int LW = (DK > DV ? DK : DV) + 4;   // 16-row fp32 buffers
    static constexpr int LS = kT + 4;
    __nv_bfloat16 S16[DK * LV];   // state before the tile
    __nv_bfloat16 D16[DK * LV];   // bf16 copy of the adjoint at the tile end
    __nv_bfloat16 Q[kT * LK], K[kT * LK], Wb[kT * LK];
    __nv_bfloat16 V[kT * LV], dO[kT * LV], nDb[kT * LV], Dhb[kT * LV], eGdO[kT * LV];
    float B1[kT * LW];   // U, then Delta
    float B2[kT * LW];   // W S_0, then dO S_0^T
    float B3[kT * LW];   // Q S_0, then dW, then dM
    float B4[kT * LW];   // K D, then dDelta
    float B5[kT * LW];   // (diag(w) Delta) D^T
    float E[kT * LS], P[kT * LS], KE[kT * LS], Lm[kT * LS], Tm[kT * LS], dP[kT * LS], X[kT * LS], dL[kT * LS];
    float stage[kBT / 32][256];   // per-warp 16 x 16 fp32 staging
    float G[kT], eG[kT], w[kT], beta[kT], sq[kT], sm_[kT], wdw[kT], red[kBT / 32];
    float dlda[kT], cross[kT], dbeta[kT];   // d lambda / d a; pair sums and dbeta (P11)
};
static_assert(sizeof(DeltaBwdSmem<128, 128>) <= 227 * 1024, "delta backward tile exceeds shared memory");

template <int DK, int DV>
__global__ void __launch_bounds__(kBT, 1)
delta_bwd_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                 const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ dO,
                 const float *__restrict__ a, const float *__restrict__ beta, float b, int mode,
                 const int32_t *__restrict__ cu, int T, int64_t tokens, int H,
                 const __nv_bfloat16 *__restrict__ states, int64_t n_slots, const float *__restrict__ dhT,
                 float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dv, float *__restrict__ da,
                 float *__restrict__ dbeta, float *__restrict__ dh0, DeviceStatus *st,
               const int32_t *__restrict__ order)
{
    using Sm = DeltaBwdSmem<DK, DV>;
    constexpr int LK = Sm::LK, LV = Sm::LV, LW = Sm::LW, LS = Sm::LS;
    constexpr int NW = kBT / 32;
    constexpr int NFD = (DK / 16) * (DV / 16) / NW;   // adjoint fragments per warp
    static_assert(NFD >= 1 && (DK / 16) * (DV / 16) % NW == 0, "adjoint split");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, n = order != nullptr ? order[blockIdx.y] : (int)blockIdx.y;
    const DocSpan d = doc_span(cu, n, T);
    if (!doc_valid(d, tokens)) {
        if (tid == 0)
            set_status(st, BDLA_ERR_DEVICE, (unsigned)n);
        return;
    }
    const int64_t unit = (int64_t)n * H + h;
    const size_t sstride = (size_t)DK * DV;
    float *stg = sm.stage[warp];
    // ---- the adjoint at the document end: fragments and bf16 copy
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> Df[NFD];
#pragma unroll
    for (int x = 0; x < NFD; ++x) {
        const int tile = warp + NW * x, mi = tile / (DV / 16), ni = tile % (DV / 16);
        for (int e = lane; e < 256; e += 32) {
            const int r = e >> 4, c2 = e & 15;
            stg[e] = dhT != nullptr ? dhT[unit * sstride + (size_t)(16 * mi + r) * DV + 16 * ni + c2] : 0.0f;
        }
        __syncwarp();
        wmma::load_matrix_sync(Df[x], stg, 16, wmma::mem_row_major);
        for (int e = lane; e < 256; e += 32)
            sm.D16[(16 * mi + (e >> 4)) * LV + 16 * ni + (e & 15)] = __float2bfloat16_rn(stg[e]);
        __syncwarp();
    }
    const int ntile = (int)((d.len + kT - 1) / kT);
    for (int c = ntile - 1; c >= 0; --c) {
        const int64_t t0 = d.start + (int64_t)c * kT;
        const int nv = (int)(d.len - (int64_t)c * kT < kT ? d.len - (int64_t)c * kT : kT);
        // ---- P0: inputs, the state before the tile (every global load issued
        //      before the shared stores), decay scalars
        {
            constexpr int rows_k = DK / 8, rows_v = DV / 8;
            constexpr int NS = DK * rows_v / kBT;   // state chunks per thread
            static_assert(NS >= 1 && DK * rows_v % kBT == 0 && kT * rows_k <= kBT && kT * rows_v <= kBT, "loads");
            const __nv_bfloat16 *src = states + ((size_t)h * n_slots + (size_t)(d.start / kT + n + c)) * sstride;
            uint4 sv[NS];
#pragma unroll
            for (int x = 0; x < NS; ++x) {
                const int e = tid + x * kBT, row = e / rows_v, c8 = (e % rows_v) * 8;
                sv[x] = *reinterpret_cast<const uint4 *>(src + (size_t)row * DV + c8);
            }
            const uint4 z4 = make_uint4(0, 0, 0, 0);
            uint4 qv = z4, kv = z4, vv = z4, gv = z4;
            const int tk = tid / rows_k, ck = (tid % rows_k) * 8, tq = tid / rows_v, cv = (tid % rows_v) * 8;
            const bool hk = tid < kT * rows_k, hv = tid < kT * rows_v;
            if (hk && tk < nv) {
                const size_t off = ((size_t)(t0 + tk) * H + h) * DK + ck;
                qv = *reinterpret_cast<const uint4 *>(q + off);
                kv = *reinterpret_cast<const uint4 *>(k + off);
            }
            if (hv && tq < nv) {
                const size_t off = ((size_t)(t0 + tq) * H + h) * DV + cv;
                vv = *reinterpret_cast<const uint4 *>(v + off);
                gv = *reinterpret_cast<const uint4 *>(dO + off);
            }
#pragma unroll
            for (int x = 0; x < NS; ++x) {
                const int e = tid + x * kBT, row = e / rows_v, c8 = (e % rows_v) * 8;
                *reinterpret_cast<uint4 *>(sm.S16 + row * LV + c8) = sv[x];
            }
            if (hk) {
                *reinterpret_cast<uint4 *>(sm.Q + tk * LK + ck) = qv;
                *reinterpret_cast<uint4 *>(sm.K + tk * LK + ck) = kv;
            }
            if (hv) {
                *reinterpret_cast<uint4 *>(sm.V + tq * LV + cv) = vv;
                *reinterpret_cast<uint4 *>(sm.dO + tq * LV + cv) = gv;
            }
            if (warp == 0) {
                const bool in = lane < nv;
                const float av = in ? a[(t0 + lane) * H + h] : 0.0f;
                float x = in ? log_decay(av, b, mode) : 0.0f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off)
                        x += y;
                }
                const float gam = __shfl_sync(0xffffffffu, x, kT - 1);
                if (lane < kT) {
                    sm.G[lane] = x;
                    sm.eG[lane] = expf(x);
                    sm.w[lane] = expf(gam - x);
                    sm.beta[lane] = in ? beta[(t0 + lane) * H + h] : 0.0f;
                    sm.dlda[lane] = in ? log_decay_deriv(av, b, mode) : 0.0f;
                }
            }
        }
        __syncthreads();
        const float gam = sm.G[kT - 1];
        // ---- P1: K K^T, Q K^T, Q S_0, K D (MMAs); the state term <S_0, D>
        {
            constexpr int J = 2 + 2 * (DV / 16);
            for (int job = warp; job < J; job += NW) {
                if (job == 0)
                    gram16<DK, LK, LS>(sm.KE, sm.K, sm.K);
                else if (job == 1)
                    gram16<DK, LK, LS>(sm.P, sm.Q, sm.K);
                else if (job < 2 + DV / 16)
                    times_state<DK, LK, LV, LW>(sm.B3, sm.Q, sm.S16, job - 2);
                else
                    times_state<DK, LK, LV, LW>(sm.B4, sm.K, sm.D16, job - 2 - DV / 16);
            }
            float part = 0.0f;
#pragma unroll
            for (int x = 0; x < NFD; ++x) {
                const int tile = warp + NW * x, mi = tile / (DV / 16), ni = tile % (DV / 16);
                wmma::store_matrix_sync(stg, Df[x], 16, wmma::mem_row_major);
                __syncwarp();
                for (int e = lane; e < 256; e += 32)
                    part += stg[e] * __bfloat162float(sm.S16[(16 * mi + (e >> 4)) * LV + 16 * ni + (e & 15)]);
                __syncwarp();
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                part += __shfl_xor_sync(0xffffffffu, part, off);
            if (lane == 0)
                sm.red[warp] = part;
        }
        __syncthreads();
        // ---- P2: pair factors; row sums (Q S_0) . dO
        for (int e = tid; e < kT * kT; e += kBT) {
            const int t = e / kT, s = e % kT;
            const float E = s <= t ? expf(sm.G[t] - sm.G[s]) : 0.0f;
            sm.E[t * LS + s] = E;
            sm.P[t * LS + s] *= E;
            const float ke = s < t ? sm.KE[t * LS + s] * E : 0.0f;
            sm.KE[t * LS + s] = ke;
            sm.Lm[t * LS + s] = sm.beta[t] * ke;
        }
        for (int t = warp; t < kT; t += NW) {
            float part = 0.0f;
            for (int j = lane; j < DV; j += 32)
                part += sm.B3[t * LW + j] * __bfloat162float(sm.dO[t * LV + j]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                part += __shfl_xor_sync(0xffffffffu, part, off);
            if (lane == 0)
                sm.sq[t] = part;
        }
        __syncthreads();
        // ---- P3: T = (I + L)^{-1} diag(beta); bf16 e^{Gamma} o dO
        if (warp == 0 && lane < kT) {
            const int j = lane;
            float x[kT];
#pragma unroll
            for (int t = 0; t < kT; ++t) {
                float acc = 0.0f;
#pragma unroll
                for (int s = 0; s < t; ++s)
                    acc += sm.Lm[t * LS + s] * x[s];
                x[t] = t < j ? 0.0f : (t == j ? sm.beta[j] : -acc);
                sm.Tm[t * LS + j] = x[t];
            }
        }
        for (int e = tid; e < kT * DV; e += kBT) {
            const int t = e / DV, j = e % DV;
            sm.eGdO[t * LV + j] = __float2bfloat16_rn(sm.eG[t] * __bfloat162float(sm.dO[t * LV + j]));
        }
        __syncthreads();
        // ---- P4: W = T diag(e^Gamma) K (bf16), U = T V (fp32); 4 columns per item,
        //      T lower-triangular (s <= t)
        for (int e = tid; e < kT * DK / 4; e += kBT) {
            const int t = e / (DK / 4), i4 = (e % (DK / 4)) * 4;
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int s = 0; s <= t; ++s) {
                const float c = sm.Tm[t * LS + s] * sm.eG[s];
                float x[4];
                ld_bf4(sm.K + s * LK + i4, x);
#pragma unroll
                for (int y = 0; y < 4; ++y)
                    acc[y] += c * x[y];
            }
            *reinterpret_cast<uint2 *>(sm.Wb + t * LK + i4) = make_uint2(pack2_bf16(acc[0], acc[1]), pack2_bf16(acc[2], acc[3]));
        }
        for (int e = tid; e < kT * DV / 4; e += kBT) {
            const int t = e / (DV / 4), j4 = (e % (DV / 4)) * 4;
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int s = 0; s <= t; ++s) {
                const float c = sm.Tm[t * LS + s];
                float x[4];
                ld_bf4(sm.V + s * LV + j4, x);
#pragma unroll
                for (int y = 0; y < 4; ++y)
                    acc[y] += c * x[y];
            }
            *reinterpret_cast<float4 *>(sm.B1 + t * LW + j4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
        __syncthreads();
        // ---- P5: W S_0
        for (int ni = warp; ni < DV / 16; ni += NW)
            times_state<DK, LK, LV, LW>(sm.B2, sm.Wb, sm.S16, ni);
        __syncthreads();
        // ---- P6: Delta, diag(w) Delta (bf16), dDelta = P^T dO + diag(w) K D, -dDelta (bf16)
        for (int e = tid; e < kT * DV; e += kBT) {
            const int t = e / DV, j = e % DV;
            const float dl = sm.B1[t * LW + j] - sm.B2[t * LW + j];
            sm.B1[t * LW + j] = dl;
            sm.Dhb[t * LV + j] = __float2bfloat16_rn(sm.w[t] * dl);
            float acc = sm.w[t] * sm.B4[t * LW + j];
            for (int s2 = t; s2 < kT; ++s2)
                acc += sm.P[s2 * LS + t] * __bfloat162float(sm.dO[s2 * LV + j]);
            sm.B4[t * LW + j] = acc;
            sm.nDb[t * LV + j] = __float2bfloat16_rn(-acc);
        }
        __syncthreads();
        // ---- P7: dW = (-dDelta) S_0^T, dO S_0^T, (diag(w) Delta) D^T  (N = DK panels)
        for (int job = warp; job < 3 * (DK / 16); job += NW) {
            const int kind = job / (DK / 16), ni = job % (DK / 16);
            const __nv_bfloat16 *A = kind == 0 ? sm.nDb : (kind == 1 ? sm.dO : sm.Dhb);
            const __nv_bfloat16 *Bm = kind == 2 ? sm.D16 : sm.S16;
            float *C = kind == 0 ? sm.B3 : (kind == 1 ? sm.B2 : sm.B5);
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.0f);
#pragma unroll
            for (int kk = 0; kk < DV / 16; ++kk) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
                wmma::load_matrix_sync(fa, A + 16 * kk, LV);
                wmma::load_matrix_sync(fb, Bm + 16 * ni * LV + 16 * kk, LV);   // B[j][i] = M[16 ni + i][j]
                wmma::mma_sync(acc, fa, fb, acc);
            }
            wmma::store_matrix_sync(C + 16 * ni, acc, LW, wmma::mem_row_major);
        }
        __syncthreads();
        // ---- P8: dP, dT: warp t, lane (s, part): the two lanes s and s + 16 take
        //      alternate 4-column chunks of the sums (a quarter warp then reads 8
        //      different rows in 8 different bank groups); dv below
        static_assert(NW == kT, "one warp per row t");
        {
            const int t = warp, s = lane & 15, part = lane >> 4;
            float acc = 0.0f, dt = 0.0f, dw = 0.0f;
#pragma unroll 4
            for (int m = 0; m < DV / 8; ++m) {
                const int j = 8 * m + 4 * part;
                float o4[4], v4[4];
                ld_bf4(sm.dO + t * LV + j, o4);
                ld_bf4(sm.V + s * LV + j, v4);
                const float4 d4 = *reinterpret_cast<const float4 *>(sm.B1 + s * LW + j);
                const float4 g4 = *reinterpret_cast<const float4 *>(sm.B4 + t * LW + j);
                acc += o4[0] * d4.x + o4[1] * d4.y + o4[2] * d4.z + o4[3] * d4.w;
                dt += g4.x * v4[0] + g4.y * v4[1] + g4.z * v4[2] + g4.w * v4[3];
            }
#pragma unroll 4
            for (int m = 0; m < DK / 8; ++m) {
                const int i = 8 * m + 4 * part;
                float k4[4];
                ld_bf4(sm.K + s * LK + i, k4);
                const float4 w4 = *reinterpret_cast<const float4 *>(sm.B3 + t * LW + i);
                dw += w4.x * k4[0] + w4.y * k4[1] + w4.z * k4[2] + w4.w * k4[3];
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 16);
            dt += __shfl_xor_sync(0xffffffffu, dt, 16);
            dw += __shfl_xor_sync(0xffffffffu, dw, 16);
            if (part == 0) {
                sm.dP[t * LS + s] = s <= t ? acc : 0.0f;
                sm.X[t * LS + s] = dt + sm.eG[s] * dw;
            }
        }
        for (int e = tid; e < kT * DV; e += kBT) {
            const int t = e / DV, j = e % DV;
            float acc = 0.0f;
            for (int s = t; s < kT; ++s)
                acc += sm.Tm[s * LS + t] * sm.B4[s * LW + j];
            if (t < nv)
                dv[((size_t)(t0 + t) * H + h) * DV + j] = acc;
        }
        __syncthreads();
        // ---- P9: dM = T^T dW in place (thread = column); X = (I + L)^{-T} dT (lane = column)
        if (tid < DK) {
            const int i = tid;
            float col[kT];
#pragma unroll
            for (int s = 0; s < kT; ++s)
                col[s] = sm.B3[s * LW + i];
#pragma unroll
            for (int t = 0; t < kT; ++t) {
                float acc = 0.0f;
#pragma unroll
                for (int s = t; s < kT; ++s)
                    acc += sm.Tm[s * LS + t] * col[s];
                sm.B3[t * LW + i] = acc;
            }
        } else if (tid >= kBT - 32 && lane < kT) {
            const int j = lane;
            float x[kT];
#pragma unroll
            for (int t = kT - 1; t >= 0; --t) {
                float acc = sm.X[t * LS + j];
#pragma unroll
                for (int s = t + 1; s < kT; ++s)
                    acc -= sm.Lm[s * LS + t] * x[s];
                x[t] = acc;
            }
            __syncwarp(0x0000ffffu);
#pragma unroll
            for (int t = 0; t < kT; ++t)
                sm.X[t * LS + j] = x[t];
        }
        __syncthreads();
        // ---- P10: dL = -strict_tril(X T^T)
        for (int e = tid; e < kT * kT; e += kBT) {
            const int t = e / kT, s = e % kT;
            float acc = 0.0f;
            if (s < t)
                for (int u = 0; u <= s; ++u)   // T is lower-triangular: T_su = 0 for u > s
                    acc -= sm.X[t * LS + u] * sm.Tm[s * LS + u];
            sm.dL[t * LS + s] = acc;
        }
        __syncthreads();
        // ---- P11: dq, dk; per-row sums for the decay gradient; the last warp
        //      (no dq/dk items) takes the pair sums and dbeta
        static_assert(kT * (DK / 8) <= kBT - 32, "the last warp is free in P11");
        if (warp == NW - 1 && lane < kT) {
            const int r = lane;
            float cr = 0.0f;
            for (int t = r; t < kT; ++t)
                for (int s = 0; s < r; ++s)
                    cr += sm.dP[t * LS + s] * sm.P[t * LS + s] + sm.dL[t * LS + s] * sm.Lm[t * LS + s];
            sm.cross[r] = cr;
            float db = sm.X[r * LS + r];
            for (int s = 0; s < r; ++s)
                db += sm.dL[r * LS + s] * sm.KE[r * LS + s];
            sm.dbeta[r] = db;
        }
        {
            constexpr int IPR = DK / 8;   // items per row, contiguous lanes
            for (int e = tid; e < kT * IPR; e += kBT) {
                const int t = e / IPR, c8 = (e % IPR) * 8;
                float gq[8], gk[8];
                const float eg = sm.eG[t];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    gq[x] = eg * sm.B2[t * LW + c8 + x];
                    gk[x] = sm.B5[t * LW + c8 + x] + eg * sm.B3[t * LW + c8 + x];
                }
                for (int s = 0; s < kT; ++s) {
                    const float dpe_ts = s <= t ? sm.dP[t * LS + s] * sm.E[t * LS + s] : 0.0f;   // as (t, s)
                    const float dpe_st = t <= s ? sm.dP[s * LS + t] * sm.E[s * LS + t] : 0.0f;   // as (s, t)
                    const float da_ts = s < t ? sm.beta[t] * sm.dL[t * LS + s] * sm.E[t * LS + s] : 0.0f;
                    const float da_st = t < s ? sm.beta[s] * sm.dL[s * LS + t] * sm.E[s * LS + t] : 0.0f;
                    const float ck = da_ts + da_st;
                    float ks[8], qs[8];
                    ld_bf8(sm.K + s * LK + c8, ks);
                    ld_bf8(sm.Q + s * LK + c8, qs);
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        gq[x] += dpe_ts * ks[x];
                        gk[x] += dpe_st * qs[x] + ck * ks[x];
                    }
                }
                float pm = 0.0f, pw = 0.0f;
                {
                    float kt[8];
                    ld_bf8(sm.K + t * LK + c8, kt);
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        pm += sm.B3[t * LW + c8 + x] * kt[x];
                        pw += sm.B5[t * LW + c8 + x] * kt[x];
                    }
                }
#pragma unroll
                for (int off = 1; off < IPR; off <<= 1) {
                    pm += __shfl_xor_sync(0xffffffffu, pm, off);
                    pw += __shfl_xor_sync(0xffffffffu, pw, off);
                }
                if (e % IPR == 0) {
                    sm.sm_[t] = pm;
                    sm.wdw[t] = pw;
                }
                if (t < nv) {
                    const size_t off = ((size_t)(t0 + t) * H + h) * DK + c8;
                    float4 *pq = reinterpret_cast<float4 *>(dq + off);
                    float4 *pk = reinterpret_cast<float4 *>(dk + off);
                    pq[0] = make_float4(gq[0], gq[1], gq[2], gq[3]);
                    pq[1] = make_float4(gq[4], gq[5], gq[6], gq[7]);
                    pk[0] = make_float4(gk[0], gk[1], gk[2], gk[3]);
                    pk[1] = make_float4(gk[4], gk[5], gk[6], gk[7]);
                }
            }
        }
        __syncthreads();
        // ---- P12: decay and write-strength gradients; D <- e^gamma D + Q^T (e^Gamma o dO) - W^T dDelta
        if (warp == 0 && lane < kT) {
            const int r = lane;
            const float cross = sm.cross[r];
            float suffix = 0.0f, prefix = 0.0f;
            for (int t = r; t < kT; ++t)
                suffix += sm.eG[t] * (sm.sq[t] + sm.sm_[t]);
            for (int t = 0; t < r; ++t)
                prefix += sm.wdw[t];
            float state = 0.0f;
#pragma unroll
            for (int x = 0; x < NW; ++x)
                state += sm.red[x];
            if (r < nv) {
                const size_t off = (size_t)(t0 + r) * H + h;
                const float dl = cross + suffix + prefix + expf(gam) * state;
                da[off] = dl * sm.dlda[r];
                dbeta[off] = sm.dbeta[r];
            }
        }
        {
            const float eg = expf(gam);
#pragma unroll
            for (int x = 0; x < NFD; ++x) {
                const int tile = warp + NW * x, mi = tile / (DV / 16), ni = tile % (DV / 16);
#pragma unroll
                for (int e = 0; e < Df[x].num_elements; ++e)
                    Df[x].x[e] *= eg;
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
                wmma::load_matrix_sync(fa, sm.Q + 16 * mi, LK);      // A[i][t] = Q[t][16 mi + i]
                wmma::load_matrix_sync(fb, sm.eGdO + 16 * ni, LV);
                wmma::mma_sync(Df[x], fa, fb, Df[x]);
                wmma::load_matrix_sync(fa, sm.Wb + 16 * mi, LK);     // A[i][t] = W[t][16 mi + i]
                wmma::load_matrix_sync(fb, sm.nDb + 16 * ni, LV);
                wmma::mma_sync(Df[x], fa, fb, Df[x]);
                wmma::store_matrix_sync(stg, Df[x], 16, wmma::mem_row_major);
                __syncwarp();
                for (int e = lane; e < 256; e += 32)
                    sm.D16[(16 * mi + (e >> 4)) * LV + 16 * ni + (e & 15)] = __float2bfloat16_rn(stg[e]);
                __syncwarp();
            }
        }
        __syncthreads();
    }
    if (dh0 != nullptr) {
#pragma unroll
        for (int x = 0; x < NFD; ++x) {
            const int tile = warp + NW * x, mi = tile / (DV / 16), ni = tile % (DV / 16);
            wmma::store_matrix_sync(stg, Df[x], 16, wmma::mem_row_major);
            __syncwarp();
            for (int e = lane; e < 256; e += 32)
                dh0[unit * sstride + (size_t)(16 * mi + (e >> 4)) * DV + 16 * ni + (e & 15)] = stg[e];
            __syncwarp();
        }
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

int64_t delta_state_slots(const Problem &p) { return p.tokens / kT + p.n_docs + 1; }

cudaError_t launch_delta_fwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const float *a, const float *beta, const float *h0, void *o,
                             int o_f32, float *hT, __nv_bfloat16 *states, const int32_t *order)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    dim3 grid(p.dv / kDvs, p.H, p.n_docs);
    const int64_t slots = delta_state_slots(p);
    cudaError_t err;
#define BDLA_DELTA_FWD(DK_, ST_)                                                                    \
    do {                                                                                            \
        auto kern = delta_fwd_kernel<DK_, ST_>;                                                     \
        if ((err = set_smem(kern, sizeof(DeltaFwdSmem<DK_>))) != cudaSuccess)                       \
            return err;                                                                             \
        kern<<<grid, kDT, sizeof(DeltaFwdSmem<DK_>), p.stream>>>(q, k, v, a, beta, p.b, p.mode, p.cu, p.T,   \
                                                                 p.tokens, p.H, p.dv, h0, o, o_f32, hT,     \
                                                                 states, slots, p.st, order);               \
    } while (0)
    const bool st = o == nullptr;   // states pass only
    if (p.dk == 64) {
        if (st)
            BDLA_DELTA_FWD(64, true);
        else
            BDLA_DELTA_FWD(64, false);
    } else {
        if (st)
            BDLA_DELTA_FWD(128, true);
        else
            BDLA_DELTA_FWD(128, false);
    }
#undef BDLA_DELTA_FWD
    return cudaGetLastError();
}

cudaError_t launch_delta_bwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const __nv_bfloat16 *dO, const float *a, const float *beta,
                             const __nv_bfloat16 *states, const float *dhT, float *dq, float *dk, float *dv,
                             float *da, float *dbeta, float *dh0, const int32_t *order)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    dim3 grid(p.H, p.n_docs);
    const int64_t slots = delta_state_slots(p);
    cudaError_t err;
#define BDLA_DELTA_BWD(DK_, DV_)                                                                    \
    do {                                                                                            \
        auto kern = delta_bwd_kernel<DK_, DV_>;                                                     \
        if ((err = set_smem(kern, sizeof(DeltaBwdSmem<DK_, DV_>))) != cudaSuccess)                  \
            return err;                                                                             \
        kern<<<grid, kBT, sizeof(DeltaBwdSmem<DK_, DV_>), p.stream>>>(                              \
            q, k, v, dO, a, beta, p.b, p.mode, p.cu, p.T, p.tokens, p.H, states, slots, dhT, dq, dk, dv, da, \
            dbeta, dh0, p.st, order);                                                               \
    } while (0)
    if (p.dk == 64 && p.dv == 64)
        BDLA_DELTA_BWD(64, 64);
    else if (p.dk == 64)
        BDLA_DELTA_BWD(64, 128);
    else if (p.dv == 64)
        BDLA_DELTA_BWD(128, 64);
    else
        BDLA_DELTA_BWD(128, 128);
#undef BDLA_DELTA_BWD
    return cudaGetLastError();
}

}  // namespace bdla
