// Per-channel (vector) decay: one log-decay per (token, head, key channel),
//     lambda_t[i] = b * sigmoid(a_t[i])   or   -softplus(a_t[i]),
//     S_t = diag(e^{lambda_t}) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t,
// the variant the first page's "per-position cumulative decay" also admits
// ("Engineering Long-Context Training for Trillion-Parameter MoE Models:
// Three Key Breakthroughs", sec. 3.1), with its sec. 3.2 bound applied
// channel by channel.
//
// Evaluated tile by tile (16 tokens, the unit of the bound).  With Gamma the
// tile-local inclusive cumsum of lambda per channel and gamma its tile total:
//   Qt = q o e^{Gamma}        (<= 1)
//   Kt = k o e^{-Gamma}       (<= e^{16 |b|} = e^{80}: the bound makes it finite)
//   Kh = k o e^{gamma - Gamma} (<= 1)
//   O  = Qt S_in + tril(Qt Kt^T) V
//   S  <- diag(e^{gamma}) S_in + Kh^T V
// Per channel the decay factors differ, so they cannot be pulled out of the
// products as row and column scalars (the scalar kernels' two-level factors
// for 128-token blocks do not apply); the diagonal tile's reciprocal goes
// onto the bf16 operands instead, which is exactly what the bound makes
// legal.  Products are 16-row bf16 warp MMAs (wmma 16x16x16, fp32
// accumulate), the state an fp32 master in shared memory with a bf16 copy.
//
// Backward (reverse tile walk), with D the adjoint of the state at the tile
// end and S_in the state before the tile (bf16, written by a states pass):
//   dq = e^{Gamma} o (dO S_in^T + tril(dO V^T) Kt)
//   dk = e^{-Gamma} o (tril(dO V^T)^T Qt) + e^{gamma - Gamma} o (V D^T)
//   dv = tril(Qt Kt^T)^T dO + Kh D
//   dlambda_t[i] = sum_{u < t} X_u[i] + sum_{r >= t} Y_r[i] + e^{gamma_i} <S_in[i,:], D[i,:]>
//     X_u = Kt_u o (dP^T Qt)_u - Qt_u o (dP Kt)_u + k_u o dk_inter_u,  Y_r = q_r o dq_inter_r
//   D <- diag(e^{gamma}) D + Qt^T dO
// The decay gradient sums, channel by channel, only the token pairs whose
// weight holds lambda_t (one token before t, one at or after it): across the
// tile start (Y), the tile end (the last part of X), both (the state term), or
// inside the tile (the dP parts of X, built from the same bf16 operands as the
// GEMMs, so pairs on one side of t cancel in the telescoped sum).  The
// equivalent q.dq - k.dk form would subtract large, nearly equal terms.
#include <mma.h>

#include "bdla_internal.h"

namespace bdla {

namespace {

using namespace nvcuda;

constexpr int kT = kChunk;       // 16-token tile
constexpr int kVecFwdThreads = 256;   // forward: 8 warps
constexpr int kVecBwdThreads = 512;   // backward: 16 warps (one CTA per SM)

// Row strides in shared memory, padded by 16 bytes so that the 16 rows a
// warp MMA fragment touches fall in different banks.
constexpr int padb(int d) { return d + 8; }   // bf16 rows
constexpr int padf(int d) { return d + 4; }   // fp32 rows

// Rows [t0, t0 + nv) of a token-major bf16 tensor [tokens][H][d] (columns
// [c0, c0 + w)) into a [16][ld] tile; rows past nv are zero.  w % 8 == 0.
__device__ __forceinline__ void load_rows(__nv_bfloat16 *dst, int ld, const __nv_bfloat16 *src, int64_t t0, int nv,
                                          int H, int h, int d, int c0, int w)
{
    const int chunks = kT * w / 8;
    for (int e = threadIdx.x; e < chunks; e += blockDim.x) {
        const int t = e / (w / 8), c = (e % (w / 8)) * 8;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (t < nv)
            val = *reinterpret_cast<const uint4 *>(src + ((t0 + t) * H + h) * (int64_t)d + c0 + c);
        *reinterpret_cast<uint4 *>(dst + t * ld + c) = val;
    }
}

// Channel pass of a tile: NT / DK threads per channel (adjacent lanes), each
// taking a run of the 16 tokens; their partial cumulative sums are joined by a
// warp scan of width NT / DK.  Writes Qt, Kt, Kh (bf16, in place over the raw
// q, k where given), the tile-local Gamma, d lambda / d a and gamma (all
// optional) and g = e^{gamma}.  Rows past nv have lambda = 0 and zero q, k, so they
// change nothing.  Every thread of the block takes part.
template <int DK, int NT>
__device__ __forceinline__ void channel_pass(const float *__restrict__ a, int64_t t0, int nv, int H, int h, float b,
                                             int mode, __nv_bfloat16 *Qt, __nv_bfloat16 *Kt, __nv_bfloat16 *Kh,
                                             float *gam_out, float *g, float *dlam_out = nullptr,
                                             float *gam_total = nullptr)
{
    constexpr int LK = padb(DK);
    constexpr int PARTS = NT / DK;       // threads per channel
    constexpr int TPP = kT / PARTS;      // tokens per thread
    static_assert(NT % DK == 0 && kT % PARTS == 0 && 32 % PARTS == 0, "channel split");
    const int i = threadIdx.x / PARTS, part = threadIdx.x % PARTS;
    const int tb = part * TPP;           // first token of this thread's run
    float av[TPP];
#pragma unroll
    for (int x = 0; x < TPP; ++x)
        av[x] = tb + x < nv ? a[((t0 + tb + x) * H + h) * (int64_t)DK + i] : 0.0f;
    float G[TPP];
    float run = 0.0f;
#pragma unroll
    for (int x = 0; x < TPP; ++x) {
        const bool in = tb + x < nv;
        run += in ? log_decay(av[x], b, mode) : 0.0f;
        G[x] = run;
        if (dlam_out != nullptr)
            dlam_out[(tb + x) * DK + i] = in ? log_decay_deriv(av[x], b, mode) : 0.0f;
    }
    // exclusive prefix of the earlier runs of this channel, and the channel's total
    float incl = run;
#pragma unroll
    for (int off = 1; off < PARTS; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off, PARTS);
        if (part >= off)
            incl += y;
    }
    const float before = incl - run;
    const float gam = __shfl_sync(0xffffffffu, incl, PARTS - 1, PARTS);
#pragma unroll
    for (int x = 0; x < TPP; ++x) {
        const int t = tb + x;
        const float Gt = before + G[x];
        const float kr = __bfloat162float(Kt[t * LK + i]);
        if (Qt != nullptr)
            Qt[t * LK + i] = __float2bfloat16_rn(__bfloat162float(Qt[t * LK + i]) * expf(Gt));
        Kt[t * LK + i] = __float2bfloat16_rn(kr * expf(-Gt));
        Kh[t * LK + i] = __float2bfloat16_rn(kr * expf(gam - Gt));
        if (gam_out != nullptr)
            gam_out[t * DK + i] = Gt;
    }
    if (part == 0) {
        g[i] = expf(gam);
        if (gam_total != nullptr)
            gam_total[i] = gam;
    }
}

// S32 <- diag(g) S32 + Kh^T V (fp32 master), then S16 <- bf16(S32).
template <int DK, int DV>
__device__ __forceinline__ void state_update(float *S32, __nv_bfloat16 *S16, const __nv_bfloat16 *Kh,
                                             const __nv_bfloat16 *V, const float *g)
{
    constexpr int LK = padb(DK), LV = padb(DV), LF = padf(DV);
    const int warp = threadIdx.x >> 5;
    for (int tile = warp; tile < (DK / 16) * (DV / 16); tile += (blockDim.x / 32)) {
        const int mi = tile / (DV / 16), ni = tile % (DV / 16);
        wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
        wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> fa;
        wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
        // rows of one fragment: 16 * mi + r, each decayed by its own channel's factor
        for (int e = threadIdx.x & 31; e < 256; e += 32)
            S32[(16 * mi + (e >> 4)) * LF + 16 * ni + (e & 15)] *= g[16 * mi + (e >> 4)];
        __syncwarp();
        wmma::load_matrix_sync(acc, S32 + 16 * mi * LF + 16 * ni, LF, wmma::mem_row_major);
        wmma::load_matrix_sync(fa, Kh + 16 * mi, LK);          // A[m][t] = Kh[t][16 mi + m]
        wmma::load_matrix_sync(fb, V + 16 * ni, LV);           // B[t][n] = V[t][16 ni + n]
        wmma::mma_sync(acc, fa, fb, acc);
        wmma::store_matrix_sync(S32 + 16 * mi * LF + 16 * ni, acc, LF, wmma::mem_row_major);
        __syncwarp();
        for (int e = threadIdx.x & 31; e < 256; e += 32) {
            const int x = (16 * mi + (e >> 4)) * LF + 16 * ni + (e & 15);
            S16[(16 * mi + (e >> 4)) * LV + 16 * ni + (e & 15)] = __float2bfloat16_rn(S32[x]);
        }
    }
    __syncthreads();
}

template <int DK, int DV>
struct VecFwdSmem {
    float S32[DK * padf(DV)];
    __nv_bfloat16 S16[DK * padb(DV)];
    __nv_bfloat16 Qt[kT * padb(DK)], Kt[kT * padb(DK)], Kh[kT * padb(DK)];
    __nv_bfloat16 V[kT * padb(DV)];
    __nv_bfloat16 P[kT * kT];
    float A[kT * kT];
    float O[kT * padf(DV)];
    float g[DK];
};

// One CTA per (dv slice of DV columns, head, document).  With `states` given
// the bf16 state before every tile goes there ([H][slots][DK][dv], slot =
// floor(doc_start / 16) + n + tile); STATES: no q and no output (the
// backward's own states pass).
template <int DK, int DV, bool STATES>
__global__ void __launch_bounds__(kVecFwdThreads)
vec_fwd_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
               const __nv_bfloat16 *__restrict__ v, const float *__restrict__ a, float b, int mode,
               const int32_t *__restrict__ cu, int T, int64_t tokens, int H, int dv,
               const float *__restrict__ h0, void *__restrict__ o, int o_f32, float *__restrict__ hT,
               __nv_bfloat16 *__restrict__ states, int64_t n_slots, DeviceStatus *st,
               const int32_t *__restrict__ order)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    VecFwdSmem<DK, DV> &sm = *reinterpret_cast<VecFwdSmem<DK, DV> *>(smem_raw);
    constexpr int LK = padb(DK), LV = padb(DV), LF = padf(DV);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int j0 = blockIdx.x * DV, h = blockIdx.y, n = order != nullptr ? order[blockIdx.z] : (int)blockIdx.z;
    const DocSpan d = doc_span(cu, n, T);
    if (!doc_valid(d, tokens)) {
        if (tid == 0)
            set_status(st, BDLA_ERR_DEVICE, (unsigned)n);
        return;
    }
    const int64_t unit = (int64_t)n * H + h;
    const size_t sstride = (size_t)DK * dv;
    for (int e = tid; e < DK * DV; e += kVecFwdThreads) {
        const int i = e / DV, j = e % DV;
        const float x = h0 != nullptr ? h0[unit * sstride + (size_t)i * dv + j0 + j] : 0.0f;
        sm.S32[i * LF + j] = x;
        sm.S16[i * LV + j] = __float2bfloat16_rn(x);
    }
    __syncthreads();
    const int ntile = (int)((d.len + kT - 1) / kT);
    for (int c = 0; c < ntile; ++c) {
        const int64_t t0 = d.start + (int64_t)c * kT;
        const int nv = (int)(d.len - (int64_t)c * kT < kT ? d.len - (int64_t)c * kT : kT);
        if (states != nullptr) {   // the state before this tile
            __nv_bfloat16 *dst = states + ((size_t)h * n_slots + (size_t)(d.start / kT + n + c)) * sstride + j0;
            for (int e = tid; e < DK * DV / 8; e += kVecFwdThreads) {
                const int row = e / (DV / 8), col = (e % (DV / 8)) * 8;
                *reinterpret_cast<uint4 *>(dst + (size_t)row * dv + col) =
                    *reinterpret_cast<const uint4 *>(sm.S16 + row * LV + col);
            }
        }
        if (!STATES)
            load_rows(sm.Qt, LK, q, t0, nv, H, h, DK, 0, DK);
        load_rows(sm.Kt, LK, k, t0, nv, H, h, DK, 0, DK);
        load_rows(sm.V, LV, v, t0, nv, H, h, dv, j0, DV);
        __syncthreads();
        channel_pass<DK, kVecFwdThreads>(a, t0, nv, H, h, b, mode, STATES ? nullptr : sm.Qt, sm.Kt, sm.Kh, nullptr, sm.g);
        __syncthreads();
        if (!STATES) {
            if (warp == 0) {   // diagonal tile: A = Qt Kt^T
                wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
                wmma::fill_fragment(acc, 0.0f);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                    wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
                    wmma::load_matrix_sync(fa, sm.Qt + 16 * kk, LK);
                    wmma::load_matrix_sync(fb, sm.Kt + 16 * kk, LK);   // B[kk][s] = Kt[s][kk]
                    wmma::mma_sync(acc, fa, fb, acc);
                }
                wmma::store_matrix_sync(sm.A, acc, kT, wmma::mem_row_major);
            }
            __syncthreads();
            for (int e = tid; e < kT * kT; e += kVecFwdThreads) {
                const int t = e / kT, s = e % kT;
                sm.P[e] = __float2bfloat16_rn(s <= t ? sm.A[e] : 0.0f);
            }
            __syncthreads();
            // O = Qt S_in + P V, one 16-column panel per warp pass
            for (int ni = warp; ni < DV / 16; ni += kVecFwdThreads / 32) {
                wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
                wmma::fill_fragment(acc, 0.0f);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                    wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
                    wmma::load_matrix_sync(fa, sm.Qt + 16 * kk, LK);
                    wmma::load_matrix_sync(fb, sm.S16 + 16 * kk * LV + 16 * ni, LV);
                    wmma::mma_sync(acc, fa, fb, acc);
                }
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fp;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fv;
                wmma::load_matrix_sync(fp, sm.P, kT);
                wmma::load_matrix_sync(fv, sm.V + 16 * ni, LV);
                wmma::mma_sync(acc, fp, fv, acc);
                wmma::store_matrix_sync(sm.O + 16 * ni, acc, LF, wmma::mem_row_major);
            }
            __syncthreads();
            // rows t < nv of o
            for (int e = tid; e < kT * DV / 8; e += kVecFwdThreads) {
                const int t = e / (DV / 8), col = (e % (DV / 8)) * 8;
                if (t >= nv)
                    continue;
                const float *src = sm.O + t * LF + col;
                const size_t off = ((size_t)(t0 + t) * H + h) * dv + j0 + col;
                if (o_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(o) + off);
                    dst[0] = make_float4(src[0], src[1], src[2], src[3]);
                    dst[1] = make_float4(src[4], src[5], src[6], src[7]);
                } else {
                    __align__(16) __nv_bfloat16 w8[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        w8[x] = __float2bfloat16_rn(src[x]);
                    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(o) + off) =
                        *reinterpret_cast<const uint4 *>(w8);
                }
            }
        }
        state_update<DK, DV>(sm.S32, sm.S16, sm.Kh, sm.V, sm.g);
    }
    if (hT != nullptr)
        for (int e = tid; e < DK * DV; e += kVecFwdThreads)
            hT[unit * sstride + (size_t)(e / DV) * dv + j0 + e % DV] = sm.S32[(e / DV) * LF + e % DV];
}

template <int DK, int DV>
struct VecBwdSmem {
    float D32[DK * padf(DV)];
    __nv_bfloat16 D16[DK * padb(DV)];
    __nv_bfloat16 S16[DK * padb(DV)];   // state before the tile
    __nv_bfloat16 Qr[kT * padb(DK)], Kr[kT * padb(DK)];   // raw q, k
    __nv_bfloat16 Qt[kT * padb(DK)], Kt[kT * padb(DK)], Kh[kT * padb(DK)];
    __nv_bfloat16 V[kT * padb(DV)], dO[kT * padb(DV)];
    __nv_bfloat16 P[kT * kT], dP[kT * kT];
    float A[kT * kT], dA[kT * kT];
    float Gm[kT * DK];     // tile-local Gamma
    float Dl[kT * DK];     // d lambda / d a
    float X1[kT * padf(DK)];   // dO S_in^T (inter dq, unscaled)
    float X2[kT * padf(DK)];   // dP^T Qt (intra dk, unscaled), then the pair terms X
    float X3[kT * padf(DK)];   // V D^T (inter dk, unscaled), then the terms Y
    float X4[kT * padf(DK)];   // dP Kt (intra dq, unscaled)
    float Y[kT * padf(DV)];    // dv
    float g[DK], gam[DK], cst[DK];
};
static_assert(sizeof(VecBwdSmem<128, 128>) <= 227 * 1024, "per-channel backward tile exceeds shared memory");
static_assert(sizeof(VecFwdSmem<128, 64>) <= 227 * 1024, "per-channel forward tile exceeds shared memory");

// One CTA per (head, document), all dv columns (dv <= 128).  Reverse walk
// over the document's tiles; the state before each tile comes from the
// states pass (bf16, [H][slots][DK][dv]).
template <int DK, int DV>
__global__ void __launch_bounds__(kVecBwdThreads)
vec_bwd_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
               const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ dO,
               const float *__restrict__ a, float b, int mode, const int32_t *__restrict__ cu, int T,
               int64_t tokens, int H, const __nv_bfloat16 *__restrict__ states, int64_t n_slots,
               const float *__restrict__ dhT, float *__restrict__ dq, float *__restrict__ dk,
               float *__restrict__ dv, float *__restrict__ da, float *__restrict__ dh0, DeviceStatus *st,
               const int32_t *__restrict__ order)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    VecBwdSmem<DK, DV> &sm = *reinterpret_cast<VecBwdSmem<DK, DV> *>(smem_raw);
    constexpr int LK = padb(DK), LV = padb(DV), LF = padf(DV), LX = padf(DK);
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
    for (int e = tid; e < DK * DV; e += kVecBwdThreads) {
        const int i = e / DV, j = e % DV;
        const float x = dhT != nullptr ? dhT[unit * sstride + e] : 0.0f;
        sm.D32[i * LF + j] = x;
        sm.D16[i * LV + j] = __float2bfloat16_rn(x);
    }
    const int ntile = (int)((d.len + kT - 1) / kT);
    for (int c = ntile - 1; c >= 0; --c) {
        const int64_t t0 = d.start + (int64_t)c * kT;
        const int nv = (int)(d.len - (int64_t)c * kT < kT ? d.len - (int64_t)c * kT : kT);
        // ---- loads: every global load of the tile is issued before the shared stores
        {
            constexpr int NS = DK * DV / 8 / kVecBwdThreads;   // state chunks per thread
            static_assert(NS >= 1 && DK * DV / 8 % kVecBwdThreads == 0, "state chunks");
            static_assert(kT * DK / 8 <= kVecBwdThreads && kT * DV / 8 <= kVecBwdThreads, "row chunks");
            const __nv_bfloat16 *src = states + ((size_t)h * n_slots + (size_t)(d.start / kT + n + c)) * sstride;
            uint4 sv[NS];
#pragma unroll
            for (int x = 0; x < NS; ++x) {
                const int e = tid + x * kVecBwdThreads, row = e / (DV / 8), c8 = (e % (DV / 8)) * 8;
                sv[x] = *reinterpret_cast<const uint4 *>(src + (size_t)row * DV + c8);
            }
            const uint4 z4 = make_uint4(0, 0, 0, 0);
            uint4 qv = z4, kv = z4, vv = z4, gv = z4;
            const int tk = tid / (DK / 8), ck = (tid % (DK / 8)) * 8;
            const int tvv = tid / (DV / 8), cv = (tid % (DV / 8)) * 8;
            const bool hk = tid < kT * DK / 8, hv = tid < kT * DV / 8;
            if (hk && tk < nv) {
                const size_t off = ((size_t)(t0 + tk) * H + h) * DK + ck;
                qv = *reinterpret_cast<const uint4 *>(q + off);
                kv = *reinterpret_cast<const uint4 *>(k + off);
            }
            if (hv && tvv < nv) {
                const size_t off = ((size_t)(t0 + tvv) * H + h) * DV + cv;
                vv = *reinterpret_cast<const uint4 *>(v + off);
                gv = *reinterpret_cast<const uint4 *>(dO + off);
            }
#pragma unroll
            for (int x = 0; x < NS; ++x) {
                const int e = tid + x * kVecBwdThreads, row = e / (DV / 8), c8 = (e % (DV / 8)) * 8;
                *reinterpret_cast<uint4 *>(sm.S16 + row * LV + c8) = sv[x];
            }
            if (hk) {
                *reinterpret_cast<uint4 *>(sm.Qr + tk * LK + ck) = qv;
                *reinterpret_cast<uint4 *>(sm.Kr + tk * LK + ck) = kv;
            }
            if (hv) {
                *reinterpret_cast<uint4 *>(sm.V + tvv * LV + cv) = vv;
                *reinterpret_cast<uint4 *>(sm.dO + tvv * LV + cv) = gv;
            }
        }
        __syncthreads();
        for (int e = tid; e < kT * DK; e += kVecBwdThreads) {
            const int x = (e / DK) * LK + e % DK;
            sm.Qt[x] = sm.Qr[x];
            sm.Kt[x] = sm.Kr[x];
        }
        __syncthreads();
        channel_pass<DK, kVecBwdThreads>(a, t0, nv, H, h, b, mode, sm.Qt, sm.Kt, sm.Kh, sm.Gm, sm.g, sm.Dl, sm.gam);
        __syncthreads();
        // ---- scores: A = Qt Kt^T (warp 0), dA = dO V^T (warp 1)
        if (warp < 2) {
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.0f);
            const __nv_bfloat16 *xa = warp == 0 ? sm.Qt : sm.dO;
            const __nv_bfloat16 *xb = warp == 0 ? sm.Kt : sm.V;
            const int kd = warp == 0 ? DK : DV;
            const int ld = warp == 0 ? LK : LV;
            for (int kk = 0; kk < kd / 16; ++kk) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
                wmma::load_matrix_sync(fa, xa + 16 * kk, ld);
                wmma::load_matrix_sync(fb, xb + 16 * kk, ld);
                wmma::mma_sync(acc, fa, fb, acc);
            }
            wmma::store_matrix_sync(warp == 0 ? sm.A : sm.dA, acc, kT, wmma::mem_row_major);
        }
        __syncthreads();
        for (int e = tid; e < kT * kT; e += kVecBwdThreads) {
            const int t = e / kT, s = e % kT;
            sm.P[e] = __float2bfloat16_rn(s <= t ? sm.A[e] : 0.0f);
            sm.dP[e] = __float2bfloat16_rn(s <= t ? sm.dA[e] : 0.0f);
        }
        __syncthreads();
        // ---- X1 = dO S_in^T;  X2 = dP^T Qt;  X3 = V D^T;  X4 = dP Kt  (N = DK panels)
        for (int job = warp; job < 4 * (DK / 16); job += kVecBwdThreads / 32) {
            const int kind = job / (DK / 16), ni = job % (DK / 16);
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.0f);
            if (kind == 0) {
                for (int kk = 0; kk < DV / 16; ++kk) {
                    wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                    wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
                    wmma::load_matrix_sync(fa, sm.dO + 16 * kk, LV);
                    wmma::load_matrix_sync(fb, sm.S16 + 16 * ni * LV + 16 * kk, LV);   // B[j][i] = S[i][j]
                    wmma::mma_sync(acc, fa, fb, acc);
                }
                wmma::store_matrix_sync(sm.X1 + 16 * ni, acc, LX, wmma::mem_row_major);
            } else if (kind == 3) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fp;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fk;
                wmma::load_matrix_sync(fp, sm.dP, kT);
                wmma::load_matrix_sync(fk, sm.Kt + 16 * ni, LK);
                wmma::mma_sync(acc, fp, fk, acc);
                wmma::store_matrix_sync(sm.X4 + 16 * ni, acc, LX, wmma::mem_row_major);
            } else if (kind == 1) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> fp;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fq;
                wmma::load_matrix_sync(fp, sm.dP, kT);   // A[s][t] = dP[t][s]
                wmma::load_matrix_sync(fq, sm.Qt + 16 * ni, LK);
                wmma::mma_sync(acc, fp, fq, acc);
                wmma::store_matrix_sync(sm.X2 + 16 * ni, acc, LX, wmma::mem_row_major);
            } else {   // kind 2
                for (int kk = 0; kk < DV / 16; ++kk) {
                    wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                    wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
                    wmma::load_matrix_sync(fa, sm.V + 16 * kk, LV);
                    wmma::load_matrix_sync(fb, sm.D16 + 16 * ni * LV + 16 * kk, LV);   // B[j][i] = D[i][j]
                    wmma::mma_sync(acc, fa, fb, acc);
                }
                wmma::store_matrix_sync(sm.X3 + 16 * ni, acc, LX, wmma::mem_row_major);
            }
        }
        // ---- dv = P^T dO + Kh D  (N = DV panels)
        for (int ni = warp; ni < DV / 16; ni += kVecBwdThreads / 32) {
            wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
            wmma::fill_fragment(acc, 0.0f);
            wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> fp;
            wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fo;
            wmma::load_matrix_sync(fp, sm.P, kT);   // A[s][t] = P[t][s]
            wmma::load_matrix_sync(fo, sm.dO + 16 * ni, LV);
            wmma::mma_sync(acc, fp, fo, acc);
            for (int kk = 0; kk < DK / 16; ++kk) {
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
                wmma::load_matrix_sync(fa, sm.Kh + 16 * kk, LK);
                wmma::load_matrix_sync(fb, sm.D16 + 16 * kk * LV + 16 * ni, LV);
                wmma::mma_sync(acc, fa, fb, acc);
            }
            wmma::store_matrix_sync(sm.Y + 16 * ni, acc, LF, wmma::mem_row_major);
        }
        __syncthreads();
        // ---- gradients of q, k, v (rows t < nv); the pair terms X (into X2) and Y (into X3)
        for (int e = tid; e < kT * DK; e += kVecBwdThreads) {
            const int t = e / DK, i = e % DK;
            const int x = t * LX + i, xb = t * LK + i;   // fp32 / bf16 rows
            const float G = sm.Gm[e];
            const float eG = expf(G);
            const float qinter = eG * sm.X1[x];
            const float dqv = qinter + eG * sm.X4[x];
            const float kinter = expf(sm.gam[i] - G) * sm.X3[x];
            const float dkv = expf(-G) * sm.X2[x] + kinter;
            const float kr = __bfloat162float(sm.Kr[xb]);
            sm.X2[x] = __bfloat162float(sm.Kt[xb]) * sm.X2[x] - __bfloat162float(sm.Qt[xb]) * sm.X4[x] + kr * kinter;
            sm.X3[x] = __bfloat162float(sm.Qr[xb]) * qinter;
            if (t < nv) {
                const size_t off = ((size_t)(t0 + t) * H + h) * DK + i;
                dq[off] = dqv;
                dk[off] = dkv;
            }
        }
        for (int e = tid; e < kT * DV; e += kVecBwdThreads) {
            const int t = e / DV, j = e % DV;
            if (t < nv)
                dv[((size_t)(t0 + t) * H + h) * DV + j] = sm.Y[t * LF + j];
        }
        // pairs across the whole tile: e^{gamma_i} <S_in[i,:], D[i,:]>; one warp per row group
        for (int i = warp; i < DK; i += kVecBwdThreads / 32) {
            float acc = 0.0f;
            for (int j = lane; j < DV; j += 32)
                acc = fmaf(__bfloat162float(sm.S16[i * LV + j]), sm.D32[i * LF + j], acc);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0)
                sm.cst[i] = sm.g[i] * acc;
        }
        __syncthreads();
        // ---- decay gradient: thread = channel, sum_{u<t} X_u + sum_{r>=t} Y_r + state term
        if (tid < DK) {
            const int i = tid;
            float ytot = 0.0f;
#pragma unroll
            for (int t = 0; t < kT; ++t)
                ytot += sm.X3[t * LX + i];
            float xb = 0.0f, yb = 0.0f;   // sums over the tokens before t
            for (int t = 0; t < kT; ++t) {
                if (t < nv) {
                    const size_t off = ((size_t)(t0 + t) * H + h) * DK + i;
                    da[off] = (xb + (ytot - yb) + sm.cst[i]) * sm.Dl[t * DK + i];
                }
                xb += sm.X2[t * LX + i];
                yb += sm.X3[t * LX + i];
            }
        }
        __syncthreads();
        // ---- adjoint: D <- diag(g) D + Qt^T dO; each warp owns NTW tiles and
        //      takes every step for all of them before the next step
        {
            constexpr int NTW = (DK / 16) * (DV / 16) / (kVecBwdThreads / 32);
            static_assert(NTW >= 1 && (DK / 16) * (DV / 16) % (kVecBwdThreads / 32) == 0, "adjoint tiles");
#pragma unroll
            for (int x = 0; x < NTW; ++x) {
                const int tile = warp + x * (kVecBwdThreads / 32), mi = tile / (DV / 16), ni = tile % (DV / 16);
#pragma unroll
                for (int e = lane; e < 256; e += 32)
                    sm.D32[(16 * mi + (e >> 4)) * LF + 16 * ni + (e & 15)] *= sm.g[16 * mi + (e >> 4)];
            }
            __syncwarp();
#pragma unroll
            for (int x = 0; x < NTW; ++x) {
                const int tile = warp + x * (kVecBwdThreads / 32), mi = tile / (DV / 16), ni = tile % (DV / 16);
                wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
                wmma::load_matrix_sync(acc, sm.D32 + 16 * mi * LF + 16 * ni, LF, wmma::mem_row_major);
                wmma::load_matrix_sync(fa, sm.Qt + 16 * mi, LK);   // A[i][t] = Qt[t][16 mi + i]
                wmma::load_matrix_sync(fb, sm.dO + 16 * ni, LV);
                wmma::mma_sync(acc, fa, fb, acc);
                wmma::store_matrix_sync(sm.D32 + 16 * mi * LF + 16 * ni, acc, LF, wmma::mem_row_major);
            }
            __syncwarp();
#pragma unroll
            for (int x = 0; x < NTW; ++x) {
                const int tile = warp + x * (kVecBwdThreads / 32), mi = tile / (DV / 16), ni = tile % (DV / 16);
#pragma unroll
                for (int e = lane; e < 256; e += 32) {
                    const int r = 16 * mi + (e >> 4), c2 = 16 * ni + (e & 15);
                    sm.D16[r * LV + c2] = __float2bfloat16_rn(sm.D32[r * LF + c2]);
                }
            }
        }
        __syncthreads();
    }
    if (dh0 != nullptr)
        for (int e = tid; e < DK * DV; e += kVecBwdThreads)
            dh0[unit * sstride + e] = sm.D32[(e / DV) * LF + e % DV];
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

int64_t vec_state_slots(const Problem &p) { return p.tokens / kT + p.n_docs + 1; }

cudaError_t launch_vec_fwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, const float *a, const float *h0, void *o, int o_f32,
                           float *hT, __nv_bfloat16 *states, const int32_t *order)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    constexpr int DVS = 64;   // value columns per CTA
    dim3 grid(p.dv / DVS, p.H, p.n_docs);
    const int64_t slots = vec_state_slots(p);
    cudaError_t err;
#define BDLA_VEC_FWD(DK_, ST_)                                                                      \
    do {                                                                                            \
        auto kern = vec_fwd_kernel<DK_, DVS, ST_>;                                                  \
        if ((err = set_smem(kern, sizeof(VecFwdSmem<DK_, DVS>))) != cudaSuccess)                    \
            return err;                                                                             \
        kern<<<grid, kVecFwdThreads, sizeof(VecFwdSmem<DK_, DVS>), p.stream>>>(                        \
            q, k, v, a, p.b, p.mode, p.cu, p.T, p.tokens, p.H, p.dv, h0, o, o_f32, hT, states, slots, \
            p.st, order);                                                                           \
    } while (0)
    const bool st = o == nullptr;   // states pass only
    if (p.dk == 64) {
        if (st)
            BDLA_VEC_FWD(64, true);
        else
            BDLA_VEC_FWD(64, false);
    } else {
        if (st)
            BDLA_VEC_FWD(128, true);
        else
            BDLA_VEC_FWD(128, false);
    }
#undef BDLA_VEC_FWD
    return cudaGetLastError();
}

cudaError_t launch_vec_bwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, const __nv_bfloat16 *dO, const float *a,
                           const __nv_bfloat16 *states, const float *dhT, float *dq, float *dk, float *dv,
                           float *da, float *dh0, const int32_t *order)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    dim3 grid(p.H, p.n_docs);
    const int64_t slots = vec_state_slots(p);
    cudaError_t err;
#define BDLA_VEC_BWD(DK_, DV_)                                                                      \
    do {                                                                                            \
        auto kern = vec_bwd_kernel<DK_, DV_>;                                                       \
        if ((err = set_smem(kern, sizeof(VecBwdSmem<DK_, DV_>))) != cudaSuccess)                    \
            return err;                                                                             \
        kern<<<grid, kVecBwdThreads, sizeof(VecBwdSmem<DK_, DV_>), p.stream>>>(                        \
            q, k, v, dO, a, p.b, p.mode, p.cu, p.T, p.tokens, p.H, states, slots, dhT, dq, dk, dv, da, \
            dh0, p.st, order);                                                                      \
    } while (0)
    if (p.dk == 64 && p.dv == 64)
        BDLA_VEC_BWD(64, 64);
    else if (p.dk == 64)
        BDLA_VEC_BWD(64, 128);
    else if (p.dv == 64)
        BDLA_VEC_BWD(128, 64);
    else
        BDLA_VEC_BWD(128, 128);
#undef BDLA_VEC_BWD
    return cudaGetLastError();
}

}  // namespace bdla
