// Tile-serial forward on CUDA cores (fp32 arithmetic), used to write state
// checkpoints whose stride is below the tensor-core kernels' 128-token block
// (the per-16-token-chunk checkpoints of the 256K stage).
//
// One CTA walks one (document, head, 64-wide dv slice) through its 16-token
// tiles ("Engineering Long-Context Training for Trillion-Parameter MoE
// Models", sec. 3.1: products inside a tile, recurrent state between tiles):
//   Gamma_t   tile-local inclusive cumsum of log-decay (decay kernel output,
//             head-major [H][tokens])
//   A_ts      = (q_t . k_s) e^{Gamma_t - Gamma_s},  s <= t in the tile
//   o_t       = e^{Gamma_t} S_in^T q_t + sum_s A_ts v_s          (when o is given)
//   S_out     = e^{gamma} S_in + sum_s e^{gamma - Gamma_s} k_s v_s^T,
// gamma = Gamma at the tile's last token; S is written to the checkpoint
// array at every multiple of the stride.
#include <mma.h>

#include "bdla_internal.h"
#include "bdla_sm100.cuh"

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
                int64_t n_slots, int n_docs, int seg_blk, const float *__restrict__ seg_init)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FwdSmem<DK> &sm = *reinterpret_cast<FwdSmem<DK> *>(smem_raw);
    const int tid = threadIdx.x;
    const int j0 = blockIdx.x * kDvSlice;
    const int h = blockIdx.y;
    // one document, or one segment of it (initial state from seg_init)
    const SegSpan span = seg_span(cu, T, tokens, n_docs, blockIdx.z, seg_blk);
    if (!span.valid)
        return;
    const int n = span.n;
    DocSpan d;
    d.start = span.start;
    d.len = span.len;
    const int64_t off0 = (int64_t)span.blk_base * 128;   // doc-local offset of the segment
    const size_t sstride = (size_t)DK * dv;
    const int64_t unit = (int64_t)n * H + h;
    const float *init = seg_blk > 0 ? seg_init : h0;
    const int64_t init_unit = seg_blk > 0 ? (int64_t)blockIdx.z * H + h : unit;

    for (int e = tid; e < DK * kDvSlice; e += kThreads) {
        const int i = e / kDvSlice, j = e % kDvSlice;
        sm.S[i][j] = init ? init[init_unit * sstride + (size_t)i * dv + j0 + j] : 0.0f;
    }
    const int64_t ntiles = (d.len + kChunk - 1) / kChunk;
    for (int64_t c = 0; c < ntiles; ++c) {
        const int64_t t0 = d.start + c * kChunk;
        const int m = (int)(d.len - c * kChunk < kChunk ? d.len - c * kChunk : kChunk);
        __syncthreads();  // previous tile finished with the smem tiles and S
        if (ckpt && ((off0 + c * kChunk) % ckpt_stride) == 0) {
            const int64_t slot = ckpt_slot(span.doc_start, n, (off0 + c * kChunk) / ckpt_stride, ckpt_stride);
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
    if (hT && span.last) {
        for (int e = tid; e < DK * kDvSlice; e += kThreads) {
            const int i = e / kDvSlice, j = e % kDvSlice;
            hT[unit * sstride + (size_t)i * dv + j0 + j] = sm.S[i][j];
        }
    }
}

// Checkpoints inside the 128-token blocks.  The tensor-core forward has
// written the state at every block start (fp32, same slot layout); this
// kernel fills the states at the block's inner multiples of the stride, one
// CTA per (block, head), all blocks at once: from the block start S, each
// 16-token tile c applies
//   S <- e^{gamma_c} S + (K o w)_c^T V_c,   w_t = e^{gamma_c - Gamma_t} <= 1
// (Gamma tile-local, gamma_c its value at the tile's last token).  The update
// is one 16-token bf16 warp MMA per 16 x 16 state tile (wmma, fp32
// accumulate).  Warp w keeps rows 16 (w mod DK/16) .. +15 of the state over
// its share of the columns in accumulator fragments, scales them by
// e^{gamma_c} (one factor for every element), and writes each inner state
// through a staging panel in shared memory with bulk async copies, one per
// row.  The work is all output bandwidth: the CTA reads k, v and the
// block-start state once (bulk async copies onto one mbarrier, k weighted in
// place afterwards) and writes up to seven states of DK x DV fp32.  Rows in
// shared memory are padded by 16 bytes so that the fragment loads and stores
// of consecutive rows fall in different banks.
constexpr int kExpThreads = 256;
constexpr int kExpWarps = kExpThreads / 32;
constexpr int kExpRows = 128 - kChunk;   // tokens feeding the inner states (the last tile feeds none)

template <int DK, int DV>
struct ExpSmem {
    static constexpr int kRG = DK / 16;                 // row groups
    static constexpr int kNC = DV * kRG / kExpWarps;    // columns per warp
    static constexpr int kLdS = kNC + 4;                // padded panel row (floats)
    static constexpr int kLdK = DK + 8, kLdV = DV + 8;  // padded bf16 rows
    float stage[kExpWarps][16 * kLdS];                  // one panel per warp
    __nv_bfloat16 kw[kExpRows][kLdK];                   // k_t o w_t
    __nv_bfloat16 v[kExpRows][kLdV];
    float w[kExpRows];   // e^{gamma_c - Gamma_t} for the token's tile c
    float eg[128 / kChunk];
    alignas(8) uint64_t bar;   // the block's loads
};
static_assert(sizeof(ExpSmem<128, 256>) <= 227 * 1024, "expansion tile exceeds shared memory");

template <int DK, int DV>
__global__ void __launch_bounds__(kExpThreads, 1)
ckpt_expand_kernel(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                   const float *__restrict__ gamma, const int32_t *__restrict__ cu, int T,
                   int64_t tokens, int n_docs, int H, float *__restrict__ ckpt, int ckpt_stride,
                   int64_t n_slots, uint64_t wait_ns, DeviceStatus *st)
{
    using namespace nvcuda;
    using Sm = ExpSmem<DK, DV>;
    constexpr int RG = Sm::kRG, NC = Sm::kNC, NF = NC / 16, LDS = Sm::kLdS;
    static_assert(NC % 16 == 0 && kExpWarps % RG == 0, "warp split");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const SegSpan blk = seg_span(cu, T, tokens, n_docs, (int)blockIdx.x, 1);   // one 128-token block
    if (!blk.valid || blk.len <= kChunk)
        return;   // no tile boundary inside the block
    const int n = blk.n;
    const int64_t off0 = (int64_t)blk.blk_base * 128;   // doc-local first token
    const int ntiles = (int)((blk.len + kChunk - 1) / kChunk);
    const int m = (ntiles - 1) * kChunk;   // tokens feeding the inner states (full tiles)
    constexpr uint32_t kPanelBytes = 16u * NC * 4u;   // bytes of one warp's panel
    if (tid == 0) {
        sm100::mbar_init(&sm.bar, 1);
        sm100::mbar_fence_init();
    }
    if (tid < m) {
        const float gt = gamma[(int64_t)h * tokens + blk.start + tid];
        const float gend = gamma[(int64_t)h * tokens + blk.start + (tid | (kChunk - 1))];
        sm.w[tid] = expf(gend - gt);
        if ((tid & (kChunk - 1)) == kChunk - 1)
            sm.eg[tid / kChunk] = expf(gend);
    }
    __syncthreads();
    if (tid == 0)
        sm100::mbar_arrive_expect_tx(&sm.bar, (uint32_t)m * (DK + DV) * 2u + kExpWarps * kPanelBytes);
    __syncthreads();   // the expected bytes are posted before any copy can complete
    // keys and values of the block's first ntiles - 1 tiles, one row per thread
    if (tid < m) {
        sm100::bulk_load(&sm.kw[tid][0], k + ((size_t)(blk.start + tid) * H + h) * DK, DK * 2u, &sm.bar);   // row stride padded
        sm100::bulk_load(&sm.v[tid][0], v + ((size_t)(blk.start + tid) * H + h) * DV, DV * 2u, &sm.bar);
    }
    // this warp's panel of the block-start state: rows r0 .. r0 + 15, columns c0 .. c0 + NC - 1
    const int r0 = 16 * (warp % RG), c0 = (warp / RG) * NC;
    const size_t sstride = (size_t)DK * DV;
    float *stg = sm.stage[warp];
    if (lane < 16) {   // one panel row per lane
        const int64_t slot = ckpt_slot(blk.doc_start, n, off0 / ckpt_stride, ckpt_stride);
        const float *src = ckpt + ((size_t)h * n_slots + slot) * sstride + (size_t)r0 * DV + c0;
        sm100::bulk_load(stg + lane * LDS, src + (size_t)lane * DV, NC * 4u, &sm.bar);
    }
    const bool ok = sm100::mbar_wait(&sm.bar, 0, wait_ns);
    if (__syncthreads_or(!ok)) {
        if (tid == 0)
            set_status(st, BDLA_ERR_TIMEOUT, (unsigned)blockIdx.x);
        if (!ok)   // let the copies land before the CTA leaves (full limit, whatever the trigger's)
            sm100::mbar_wait(&sm.bar, 0, kDefaultWaitNs);
        return;
    }
    // weight the keys in place: k_t o w_t
    for (int e = tid; e < m * (DK / 8); e += kExpThreads) {
        const int t = e / (DK / 8), c8 = e % (DK / 8);
        uint4 *p = reinterpret_cast<uint4 *>(&sm.kw[t][0]) + c8;
        const uint4 raw = *p;
        const float wt = sm.w[t];
        const uint32_t x[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            y[i] = sm100::pack_bf16(sm100::bf16_lo(x[i]) * wt, sm100::bf16_hi(x[i]) * wt);
        *p = make_uint4(y[0], y[1], y[2], y[3]);
    }
    __syncthreads();   // kw weighted
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f)
        wmma::load_matrix_sync(acc[f], stg + 16 * f, LDS, wmma::mem_row_major);
    __syncwarp();
    for (int c = 0; c + 1 < ntiles; ++c) {   // the last tile ends the block: not needed here
        const float eg = sm.eg[c];
        wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major> fa;
        wmma::load_matrix_sync(fa, &sm.kw[16 * c][r0], Sm::kLdK);            // A[i][t] = kw[t][r0 + i]
#pragma unroll
        for (int f = 0; f < NF; ++f) {
#pragma unroll
            for (int e = 0; e < acc[f].num_elements; ++e)
                acc[f].x[e] *= eg;
            wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major> fb;
            wmma::load_matrix_sync(fb, &sm.v[16 * c][c0 + 16 * f], Sm::kLdV);  // B[t][j] = v[t][c0 + j]
            wmma::mma_sync(acc[f], fa, fb, acc[f]);
        }
        const int64_t tl = off0 + (int64_t)(c + 1) * kChunk;   // doc-local token the state precedes
        if (tl % ckpt_stride != 0)
            continue;
        if (lane < 16)
            sm100::tma_store_wait_read();   // the previous panel has left the staging buffer
        __syncwarp();
#pragma unroll
        for (int f = 0; f < NF; ++f)
            wmma::store_matrix_sync(stg + 16 * f, acc[f], LDS, wmma::mem_row_major);
        sm100::fence_proxy_async_smem();
        __syncwarp();
        if (lane < 16) {   // one panel row per lane
            float *dst = ckpt + ((size_t)h * n_slots + (size_t)ckpt_slot(blk.doc_start, n, tl / ckpt_stride, ckpt_stride)) *
                                    sstride + (size_t)(r0 + lane) * DV + c0;
            sm100::bulk_store(dst, stg + lane * LDS, NC * 4u);
            sm100::tma_store_commit();
        }
    }
    if (lane < 16)
        sm100::tma_store_wait_read();   // shared memory stays valid until the copies have read it
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_fwd_tile(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                            const __nv_bfloat16 *v, const float *gamma, const float *h0, void *o,
                            int o_f32, float *hT, float *ckpt, int ckpt_stride, const SegPlan &seg)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    dim3 grid(p.dv / kDvSlice, p.H, seg.seg_blk > 0 ? (unsigned)seg.n_slots : (unsigned)p.n_docs);
    const int64_t n_slots = ckpt ? ckpt_slots(p, ckpt_stride) : 0;
    cudaError_t err;
    if (p.dk == 64) {
        auto kern = fwd_tile_kernel<64>;
        if ((err = set_smem(kern, sizeof(FwdSmem<64>))) != cudaSuccess)
            return err;
        kern<<<grid, kThreads, sizeof(FwdSmem<64>), p.stream>>>(q, k, v, gamma, p.cu, p.T, p.tokens,
            p.H, p.dv, h0, o, o_f32, hT, ckpt, ckpt_stride, n_slots, p.n_docs,
            seg.seg_blk, seg.buf);
    } else {
        auto kern = fwd_tile_kernel<128>;
        if ((err = set_smem(kern, sizeof(FwdSmem<128>))) != cudaSuccess)
            return err;
        kern<<<grid, kThreads, sizeof(FwdSmem<128>), p.stream>>>(q, k, v, gamma, p.cu, p.T,
            p.tokens, p.H, p.dv, h0, o, o_f32, hT, ckpt, ckpt_stride, n_slots, p.n_docs,
            seg.seg_blk, seg.buf);
    }
    return cudaGetLastError();
}

cudaError_t launch_ckpt_expand(const Problem &p, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                               const float *gamma, float *ckpt, int ckpt_stride)
{
    if (p.n_docs <= 0 || p.tokens <= 0)
        return cudaSuccess;
    const int64_t n_slots = ckpt_slots(p, ckpt_stride);
    const int64_t blocks = (p.tokens + 127) / 128 + p.n_docs;   // block slots (seg_span with 1-block segments)
    if (blocks > INT32_MAX || p.H > 65535)
        return cudaErrorInvalidValue;
    dim3 grid((unsigned)blocks, p.H);
    const WaitCfg wc = wait_cfg(BDLA_KERNEL_STATES);
    cudaError_t err;
#define BDLA_EXPAND(DK_, DV_)                                                                       \
    do {                                                                                            \
        auto kern = ckpt_expand_kernel<DK_, DV_>;                                                   \
        if ((err = set_smem(kern, sizeof(ExpSmem<DK_, DV_>))) != cudaSuccess)                       \
            return err;                                                                             \
        kern<<<grid, kExpThreads, sizeof(ExpSmem<DK_, DV_>), p.stream>>>(                           \
            k, v, gamma, p.cu, p.T, p.tokens, p.n_docs, p.H, ckpt, ckpt_stride, n_slots, wc.ns, p.st); \
    } while (0)
    if (p.dk == 64) {
        if (p.dv == 64)
            BDLA_EXPAND(64, 64);
        else if (p.dv == 128)
            BDLA_EXPAND(64, 128);
        else
            BDLA_EXPAND(64, 256);
    } else {
        if (p.dv == 64)
            BDLA_EXPAND(128, 64);
        else if (p.dv == 128)
            BDLA_EXPAND(128, 128);
        else
            BDLA_EXPAND(128, 256);
    }
#undef BDLA_EXPAND
    return cudaGetLastError();
}

// bf16 copies of the states at the 128-token block starts, taken from fp32
// checkpoints whose stride divides 128, in the layout of the forward's bf16
// block checkpoints ([H][slots of stride 128][dk][dv]): the backward then
// loads each block's S_in by one TMA copy.  One CTA per (block slot, head);
// block slot b is the 128-token span of seg_span(..., b, 1), gaps return.
__global__ void __launch_bounds__(256)
states_bf16_kernel(const float *__restrict__ ck, int stride, int64_t ck_slots, __nv_bfloat16 *__restrict__ out,
                   int64_t out_slots, const int32_t *__restrict__ cu, int T, int64_t tokens, int n_docs, int dk,
                   int dv)
{
    const SegSpan sl = seg_span(cu, T, tokens, n_docs, (int)blockIdx.x, 1);
    if (!sl.valid || sl.len <= 0)
        return;
    const int h = blockIdx.y;
    const int64_t src = ckpt_slot(sl.doc_start, sl.n, (int64_t)sl.s * 128 / stride, stride);
    const int64_t dst = ckpt_slot(sl.doc_start, sl.n, sl.s, 128);
    const float4 *s4 = reinterpret_cast<const float4 *>(ck + ((size_t)h * ck_slots + src) * dk * dv);
    uint2 *d2 = reinterpret_cast<uint2 *>(out + ((size_t)h * out_slots + dst) * dk * dv);
    const int n4 = dk * dv / 4;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 x = s4[i];
        d2[i] = make_uint2(sm100::pack_bf16(x.x, x.y), sm100::pack_bf16(x.z, x.w));
    }
}

cudaError_t launch_states_bf16(const Problem &p, const float *ckpt, int ckpt_stride, __nv_bfloat16 *out)
{
    if (p.n_docs <= 0 || p.tokens <= 0)
        return cudaSuccess;
    const int64_t blocks = (p.tokens + 127) / 128 + p.n_docs;
    states_bf16_kernel<<<dim3((unsigned)blocks, (unsigned)p.H), 256, 0, p.stream>>>(
        ckpt, ckpt_stride, ckpt_slots(p, ckpt_stride), out, ckpt_slots(p, 128), p.cu, p.T, p.tokens, p.n_docs,
        p.dk, p.dv);
    return cudaGetLastError();
}

}  // namespace bdla
