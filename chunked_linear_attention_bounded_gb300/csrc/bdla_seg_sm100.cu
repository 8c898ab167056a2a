// Sequence segments: parallelism along the sequence inside one GPU.
//
// A state passes between chunks ("Engineering Long-Context Training for
// Trillion-Parameter MoE Models", sec. 3.1), so one CTA per (document, head)
// walks its document block after block.  When those units are fewer than the
// SMs, each document is cut into segments and the state entering every
// segment is found first, from two facts of the recurrence S_t = e^{lam_t}
// S_{t-1} + k_t v_t^T:
//   S_end = e^{Lam_end} S_start + sum_t e^{Lam_end - Lam_t} k_t v_t^T
// (Lam the inclusive cumulative log-decay from the segment start), and, for
// the adjoint D of the backward pass (D += q_t dO_t^T, then D <- e^{lam_t} D),
//   D_start = e^{Lam_end} D_end + sum_t e^{Lam_t} q_t dO_t^T.
// seg_summary computes the sums (one tensor-core GEMM per 128-token block,
// accumulated in tensor memory); seg_scan chains them over the segments of a
// document, in token order for S and in reverse for D, and leaves in place
// the state each segment starts from.  The forward and backward kernels then
// run one CTA per segment from those states.
//
// Every weight e^{...} is <= 1: the summary walks the forward's blocks from
// the segment end (suffix sums) and the backward's from the start (prefix
// sums), so no partial sum is ever rescaled.
#include <cudaTypedefs.h>

#include "bdla_internal.h"
#include "bdla_sm100.cuh"

namespace bdla {

bool make_token_map(CUtensorMap *map, const void *ptr, int d, int H, int64_t tokens);

std::atomic<int> g_seq_split{0};

namespace {

using namespace sm100;

constexpr int BT = 128;
constexpr int kStages = 3;
constexpr int kRowThreads = 128;                       // warps 2-5: one token row each
constexpr int kSegThreads = 64 + 2 * kRowThreads;      // + producer, MMA and 4 epilogue warps
constexpr uint32_t kPanel = 16384;
// drains of a CTA's own copies and MMAs before it exits keep the full limit
constexpr uint64_t kWaitNs = kDefaultWaitNs;

template <int DV>
struct SegSmem {
    alignas(1024) unsigned char x[kStages][2 * kPanel];          // rows: tokens, panels: dk
    alignas(1024) unsigned char y[kStages][(DV / 64) * kPanel];  // rows: tokens, panels: dv
    float gam[BT / kChunk];
    uint64_t full[kStages], xready[kStages], empty[kStages], acc_full[2], acc_free[2], drain;
    uint64_t never;   // nothing arrives here: the wait of the stall test hook
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kMaxSmem = 232448;
static_assert(sizeof(SegSmem<128>) <= kMaxSmem, "segment summary shared memory exceeds the limit");

__device__ __forceinline__ void row_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool row_all(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint4 scale_row8(uint4 x, float s)
{
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = pack_bf16(bf16_lo(w[i]) * s, bf16_hi(w[i]) * s);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Persistent: each CTA walks the (segment slot, head, dv slice) items
// blockIdx.x, blockIdx.x + gridDim.x, ...; the TMA ring and the MMA
// pipeline run on across items, two TMEM accumulators let one item's sums
// drain while the next accumulates.  Warp 0 loads, warp 1 issues the MMAs,
// warps 2-5 scale the x rows, warps 6-9 write the sums.  BWD selects the
// weights e^{Lam_t} (blocks in token order) instead of e^{Lam_end - Lam_t}
// (blocks from the segment end).
template <int DV, bool BWD>
__global__ void __launch_bounds__(kSegThreads, 1)
seg_summary_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap ty,
                   const float *__restrict__ gamma, const int32_t *__restrict__ cu, int T,
                   int64_t tokens, int n_docs, int H, int dk, int dv, int seg_blk, int64_t n_items,
                   float *__restrict__ sums, float *__restrict__ lsum, DeviceStatus *st,
                   uint64_t wait_ns, int stall)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    SegSmem<DV> &sm = *reinterpret_cast<SegSmem<DV> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        if (tid == 0)
            set_status(st, BDLA_ERR_DEVICE, 0xC11u);
        return;
    }
    const int kpan = dk / 64;
    const int slices = dv / DV;
    // item -> (slot, head, slice) and its segment (len < 0: nothing to do)
    auto item = [&](int64_t i, int &slot, int &h, int &j0, SegSpan &g) -> int {
        j0 = (int)(i % slices) * DV;
        h = (int)((i / slices) % H);
        slot = (int)(i / ((int64_t)slices * H));
        g = seg_span(cu, T, tokens, n_docs, slot, seg_blk);
        return g.valid ? (int)((g.len + BT - 1) / BT) : -1;
    };

    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 2 * DV);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.xready[s], kRowThreads);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_free[a], kRowThreads);
        }
        mbar_init(&sm.drain, 1);
        mbar_init(&sm.never, 1);
        sm.abort_flag = 0;
        mbar_fence_init();
    }
    if (kpan == 1) {   // dk = 64: the upper key panel of every stage stays zero
        for (int e = tid; e < kStages * (int)(kPanel / 16); e += kSegThreads) {
            const int s = e / (kPanel / 16), i = e % (kPanel / 16);
            reinterpret_cast<uint4 *>(sm.x[s] + kPanel)[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tx);
            tma_prefetch_desc(&ty);
            const uint32_t bytes = (uint32_t)(kpan + DV / 64) * kPanel;
            int64_t gb = 0;   // blocks loaded by this CTA
            bool ok = true;
            for (int64_t i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
                int slot, h, j0;
                SegSpan g;
                const int nblk = item(i, slot, h, j0, g);
                for (int b = 0; b < nblk; ++b, ++gb) {
                    const int j = BWD ? b : nblk - 1 - b;
                    const int s = (int)(gb % kStages);
                    // (test hook: the stalling role waits at its CTA's second block)
                    if (*abort_flag || (stall == BDLA_STALL_PRODUCER && gb == 1 && !mbar_wait(&sm.never, 0, wait_ns)) ||
                        (gb >= kStages && !mbar_wait(&sm.empty[s], ((gb / kStages) - 1) & 1, wait_ns))) {
                        ok = false;
                        break;
                    }
                    const int t0 = (int)(g.start + (int64_t)j * BT);
                    mbar_arrive_expect_tx(&sm.full[s], bytes);
                    for (int p = 0; p < kpan; ++p)
                        tma_load_3d(sm.x[s] + p * kPanel, &tx, &sm.full[s], p * 64, h, t0);
                    for (int p = 0; p < DV / 64; ++p)
                        tma_load_3d(sm.y[s] + p * kPanel, &ty, &sm.full[s], j0 + p * 64, h, t0);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(st, BDLA_ERR_TIMEOUT, 21u);
            }
            // the copies this thread started have landed before the CTA exits
            for (int64_t b = gb - kStages < 0 ? 0 : gb - kStages; b < gb; ++b)
                mbar_wait(&sm.full[b % kStages], (b / kStages) & 1, kWaitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id = idesc_bf16_f32(128, DV, true, true);   // [dk x dv] += X^T Y
            int64_t gb = 0, la = 0;   // blocks consumed, items accumulated
            bool ok = true;
            for (int64_t i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
                int slot, h, j0;
                SegSpan g;
                const int nblk = item(i, slot, h, j0, g);
                if (nblk <= 0)
                    continue;
                const int a = (int)(la & 1);
                if (la >= 2 && !mbar_wait(&sm.acc_free[a], ((la / 2) - 1) & 1, wait_ns)) {
                    ok = false;
                    break;
                }
                for (int b = 0; b < nblk; ++b, ++gb) {
                    const int s = (int)(gb % kStages);
                    if (*abort_flag || (stall == BDLA_STALL_MMA && gb == 1 && !mbar_wait(&sm.never, 0, wait_ns)) ||
                        !mbar_wait(&sm.xready[s], (gb / kStages) & 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sx = smem_u32(sm.x[s]), sy = smem_u32(sm.y[s]);
                    for (int ks = 0; ks < BT / 16; ++ks)
                        umma_bf16(tmem + a * DV, sdesc_sw128(sx + ks * 2048, kPanel, 1024),
                                  sdesc_sw128(sy + ks * 2048, kPanel, 1024), id, (b > 0 || ks > 0) ? 1 : 0);
                    umma_commit(&sm.empty[s]);
                }
                if (!ok)
                    break;
                umma_commit(&sm.acc_full[a]);
                ++la;
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(st, BDLA_ERR_TIMEOUT, 22u);
            }
            // every MMA issued above completes before TMEM is released
            umma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, kWaitNs);
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------------- row warps
        const int r = 32 * (warp & 3) + lane;   // token row of the block
        int64_t gb = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
            int slot, h, j0;
            SegSpan g;
            const int nblk = item(i, slot, h, j0, g);
            if (nblk < 0)
                continue;
            float run = 0.0f;   // summed log-decay of the blocks already taken
            // Gamma of the row in block j (0 past the segment end); each block's
            // value is loaded while the block before it is scaled
            auto gamma_of = [&](int j) -> float {
                const bool in = (int64_t)j * BT + r < g.len;
                return in ? gamma[(int64_t)h * tokens + g.start + (int64_t)j * BT + r] : 0.0f;
            };
            float gv_next = nblk > 0 ? gamma_of(BWD ? 0 : nblk - 1) : 0.0f;
            for (int b = 0; b < nblk; ++b, ++gb) {
                const int j = BWD ? b : nblk - 1 - b;
                const int s = (int)(gb % kStages);
                const int Lb = (int)(g.len - (int64_t)j * BT < BT ? g.len - (int64_t)j * BT : BT);
                const bool valid = r < Lb;
                const int tau = r >> 4;
                const float gv = gv_next;
                if (b + 1 < nblk)
                    gv_next = gamma_of(BWD ? b + 1 : nblk - 2 - b);
                const int lastr = min(16 * tau + 15, Lb - 1);
                const float g_last = __shfl_sync(0xffffffffu, gv, lastr & 31);
                row_sync();   // every row has read the previous block's tile totals
                if ((r & 15) == 0)
                    sm.gam[tau] = (16 * tau < Lb) ? g_last : 0.0f;
                row_sync();
                float Gt = 0.0f, lend = 0.0f;
#pragma unroll
                for (int u = 0; u < BT / kChunk; ++u) {
                    Gt += (u < tau) ? sm.gam[u] : 0.0f;
                    lend += sm.gam[u];
                }
                const float lam = Gt + gv;   // inclusive cumulative log-decay inside the block
                const float c = BWD ? run + lam : run + (lend - lam);
                const float w = valid ? expf(c) : 0.0f;
                run += lend;
                ok = row_all(mbar_wait(&sm.full[s], (gb / kStages) & 1, wait_ns) &&
                             !(stall == BDLA_STALL_EPILOGUE && gb == 1 && !mbar_wait(&sm.never, 0, wait_ns))) &&
                     !*abort_flag;
                if (!ok)
                    break;
#pragma unroll 1
                for (int p = 0; p < kpan; ++p)
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint4 *xa = reinterpret_cast<uint4 *>(sm.x[s] + p * kPanel + sw128_offset(r, c8));
                        *xa = scale_row8(*xa, w);
                    }
                fence_proxy_async_smem();
                mbar_arrive(&sm.xready[s]);
            }
            if (ok && r == 0 && j0 == 0)
                lsum[(size_t)slot * H + h] = run;
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0)
                set_status(st, BDLA_ERR_TIMEOUT, 23u);
        }
    } else {
        // ---------------------------------------------------------------- sum writers
        const int q4 = warp & 3;               // TMEM lane quarter this warp may access
        const int r = 32 * q4 + lane;          // key row of the sums
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        int64_t la = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
            int slot, h, j0;
            SegSpan g;
            const int nblk = item(i, slot, h, j0, g);
            if (nblk < 0)
                continue;
            const size_t base = ((size_t)slot * H + h) * (size_t)dk * dv;
            const int a = (int)(la & 1);
            if (nblk > 0) {
                if (!mbar_wait(&sm.acc_full[a], (la / 2) & 1, wait_ns) || *abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (r < dk) {
#pragma unroll 1
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t x[32];
                    if (nblk > 0) {
                        tmem_ld32(tmem + a * DV + lane_off + c * 32, x);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            x[e] = 0u;
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(sums + base + (size_t)r * dv + j0 + c * 32);
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        dst[k4] = make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
                }
            }
            if (nblk > 0) {
                tc_fence_before();
                mbar_arrive(&sm.acc_free[a]);
                ++la;
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0)
                set_status(st, BDLA_ERR_TIMEOUT, 24u);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem, 2 * DV);
}

// One thread per 4 consecutive state entries of one (document, head); the
// loop over the document's segments carries the state.
template <bool BWD>
__global__ void __launch_bounds__(256)
seg_scan_kernel(const int32_t *__restrict__ cu, int T, int64_t tokens, int H, int dk, int dv,
                int seg_blk, const float *__restrict__ init, float *__restrict__ buf,
                const float *__restrict__ lsum)
{
    const int h = blockIdx.y, n = blockIdx.z;
    const int64_t sz = (int64_t)dk * dv;
    const int64_t e = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (e >= sz)
        return;
    const DocSpan d = doc_span(cu, n, T);
    if (!doc_valid(d, tokens))
        return;
    const int64_t L = (int64_t)seg_blk * 128;
    const int64_t base = d.start / L + n;
    const int nseg = (int)(d.len > 0 ? (d.len + L - 1) / L : 1);
    float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init != nullptr)
        S = *reinterpret_cast<const float4 *>(init + ((int64_t)n * H + h) * sz + e);
    for (int i = 0; i < nseg; ++i) {
        const int64_t slot = base + (BWD ? nseg - 1 - i : i);
        float4 *p = reinterpret_cast<float4 *>(buf + (slot * H + h) * sz + e);
        const float4 dsum = *p;
        const float a = expf(lsum[slot * H + h]);
        *p = S;
        S.x = fmaf(a, S.x, dsum.x);
        S.y = fmaf(a, S.y, dsum.y);
        S.z = fmaf(a, S.z, dsum.z);
        S.w = fmaf(a, S.w, dsum.w);
    }
}

int sm_count()
{
    static int cached = 0;
    if (cached == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            cached = v;
        else
            return 152;
    }
    return cached;
}

}  // namespace

SegPlan plan_segments(const Problem &p)
{
    SegPlan sp;
    const int split = g_seq_split.load();
    // the slot count (at most 65535) must leave room for at least one token
    // block beside the documents
    if (p.tokens <= 0 || p.n_docs <= 0 || split < 0 || p.n_docs >= 65535 - 1)
        return sp;
    const int slices = p.dv > 128 ? p.dv / 128 : 1;
    const int64_t units = (int64_t)p.n_docs * p.H * slices;
    const int64_t nblk = (p.tokens + BT - 1) / BT;
    int64_t sb;
    if (split > 0) {
        sb = split;
    } else {
        const int sms = sm_count();
        if (units >= sms)
            return sp;
        // about four segments per SM, at least 4 blocks each
        const int64_t total = (nblk + p.n_docs) * p.H * slices;
        sb = (total + 4 * sms - 1) / (4 * sms);
        sb = sb < 4 ? 4 : sb;
    }
    // the slot count is a grid extent (at most 65535)
    const int64_t min_sb = (nblk + 65535 - p.n_docs - 1) / (65535 - p.n_docs);
    sb = sb < min_sb ? min_sb : sb;
    sp.seg_blk = (int)sb;
    sp.n_slots = (p.tokens + BT * sb - 1) / (BT * sb) + p.n_docs;
    return sp;
}

cudaError_t launch_seg_summary(const Problem &p, const __nv_bfloat16 *x, const __nv_bfloat16 *y,
                               const float *gamma, bool backward, const SegPlan &seg)
{
    if (seg.seg_blk <= 0 || p.tokens <= 0)
        return cudaSuccess;
    CUtensorMap mx, my;
    if (!make_token_map(&mx, x, p.dk, p.H, p.tokens) || !make_token_map(&my, y, p.dv, p.H, p.tokens))
        return cudaErrorInvalidValue;
    const int DVs = p.dv >= 128 ? 128 : 64;
    const int64_t n_items = (int64_t)(p.dv / DVs) * p.H * seg.n_slots;
    const int64_t n_cta = n_items < sm_count() ? n_items : sm_count();
    dim3 grid((unsigned)n_cta);
    const WaitCfg wc = wait_cfg(BDLA_KERNEL_SEG);
    cudaError_t err;
#define BDLA_SEG_GO(DV_, B_)                                                                       \
    do {                                                                                           \
        auto kern = seg_summary_kernel<DV_, B_>;                                                   \
        const size_t smem = sizeof(SegSmem<DV_>);                                                  \
        if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,         \
                                        (int)smem)) != cudaSuccess)                                \
            return err;                                                                            \
        kern<<<grid, kSegThreads, smem, p.stream>>>(mx, my, gamma, p.cu, p.T, p.tokens, p.n_docs, \
                                                    p.H, p.dk, p.dv, seg.seg_blk, n_items,         \
                                                    seg.buf, seg.lsum, p.st, wc.ns, wc.stall);     \
    } while (0)
    if (DVs == 64) {
        if (backward)
            BDLA_SEG_GO(64, true);
        else
            BDLA_SEG_GO(64, false);
    } else {
        if (backward)
            BDLA_SEG_GO(128, true);
        else
            BDLA_SEG_GO(128, false);
    }
#undef BDLA_SEG_GO
    return cudaGetLastError();
}

cudaError_t launch_seg_scan(const Problem &p, const float *init, bool backward, const SegPlan &seg)
{
    if (seg.seg_blk <= 0 || p.tokens <= 0)
        return cudaSuccess;
    const int64_t sz = (int64_t)p.dk * p.dv;
    dim3 grid((unsigned)((sz / 4 + 255) / 256), p.H, p.n_docs);
    if (backward)
        seg_scan_kernel<true><<<grid, 256, 0, p.stream>>>(p.cu, p.T, p.tokens, p.H, p.dk, p.dv,
                                                          seg.seg_blk, init, seg.buf, seg.lsum);
    else
        seg_scan_kernel<false><<<grid, 256, 0, p.stream>>>(p.cu, p.T, p.tokens, p.H, p.dk, p.dv,
                                                           seg.seg_blk, init, seg.buf, seg.lsum);
    return cudaGetLastError();
}

}  // namespace bdla
