// Forward pass on the sm_100-family tensor cores: TMA tile loads,
// tcgen05.mma with fp32 accumulators in tensor memory, one CTA per
// (document, head, dv slice) walking the document in 128-token blocks.
//
// Method ("Engineering Long-Context Training for Trillion-Parameter MoE
// Models", sec. 3.1-3.3; "Engineering Stability in Ultra-Long Context and
// Trillion-Parameter Sparse Models", sec. 2.2): inside a chunk the products
// are dense GEMMs and a state passes between chunks; the bounded log-decay
// keeps the reciprocal of the in-tile cumulative decay finite so that the
// diagonal tiles go through the same GEMM as every other tile.
//
// Per block of 128 tokens (8 decay tiles of 16) with Gamma the tile-local
// cumulative log-decay, gamma_tau the tile totals, G_tau their exclusive
// prefix inside the block and Lam = G + Gamma:
//   score = Q K^T                                            (tensor cores)
//   P_ts  = score_ts e^{-Gamma_s} e^{Gamma_t}                 same tile, s <= t
//   P_ts  = score_ts e^{gamma_sig - Gamma_s} e^{G_tau - G_sig+1} e^{Gamma_t}   sig < tau
//   O     = P V + (Q o e^{Lam}) S_in                          (tensor cores)
//   S_out = e^{Lam_end} S_in + (K o e^{Lam_end - Lam})^T V    (tensor cores)
// Every factor is <= 1 except e^{-Gamma_s} on the diagonal tile, which the
// bound keeps <= e^{16 |b|} = e^{80}.  The unbounded ablation instead
// computes the diagonal tile pair by pair on CUDA cores,
//   P_ts = (q_t . k_s) e^{Gamma_t - Gamma_s}   (explicit position-pair path),
// and keeps the GEMM result only for the off-diagonal tiles.
//
// Warp roles: warp 0 issues TMA loads (Q, K double-buffered, V single),
// warp 1 allocates TMEM and issues the MMAs, warps 2-9 (two per TMEM lane
// quarter, splitting the columns) turn scores into P, fold the decay into Q
// and K in place, move the state between TMEM and its bf16 shared copy, and
// store O.  P is written back (bf16) into its block's score buffer in TMEM,
// from where the P V GEMM reads its A operand; the score GEMM of block j+2
// reuses that buffer once block j's P V GEMM has completed.
// Every wait is bounded; on expiry the CTA records BDLA_ERR_TIMEOUT, drains
// its own copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "bdla_internal.h"
#include "bdla_sm100.cuh"

namespace bdla {

namespace {

using namespace sm100;

constexpr int BT = 128;             // tokens per block
constexpr int kEpiWarps = 8;        // two per TMEM lane quarter
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kFwdThreads = 64 + kEpiThreads;   // producer warp, MMA warp, epilogue
constexpr uint32_t kPanel = 16384;  // one 128-row x 128-byte swizzled panel
// drains of a CTA's own copies and MMAs before it exits keep the full limit
constexpr uint64_t kWaitNs = kDefaultWaitNs;

template <int DV>
struct FwdSmem {
    alignas(1024) unsigned char q[2][2 * kPanel];   // stages x dk panels
    alignas(1024) unsigned char k[2][2 * kPanel];
    alignas(1024) unsigned char v[(DV / 64) * kPanel];
    alignas(1024) unsigned char sb[(DV / 64) * kPanel];  // state bf16: rows dk, panels over dv
    float cdiag[BT];     // e^{-Gamma_s}
    float coff[BT];      // e^{gamma_sig - Gamma_s}
    float gq[BT];        // Gamma per row (ablation diagonal path)
    float gam[BT / kChunk];
    float eg[BT / kChunk];   // e^{gamma_tau}
    uint32_t abl_pair[BT][4];   // ablation: one half's 8 position-pair values of a row (bf16 pairs)
    uint64_t full_qk[2], empty_qk[2], score_full[2];
    uint64_t full_v, empty_v, p_ready, o_full, p_free, drain;
    uint64_t never;
    uint64_t wait_ns;     // limit of the pipeline waits
    int stall_at[3];      // test hook: block at which producer / MMA / epilogue stall (-1: never)   // nothing arrives here: the wait of the stall test hook
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kMaxSmem = 232448;   // 227 KB opt-in shared memory per CTA
static_assert(sizeof(FwdSmem<128>) <= kMaxSmem && sizeof(FwdSmem<64>) <= kMaxSmem,
              "forward shared memory exceeds the per-CTA limit");

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ bool epi_all(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint4 scale_bf16x8(uint4 x, float s)
{
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = pack_bf16(bf16_lo(w[i]) * s, bf16_hi(w[i]) * s);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float dot_bf16x8(uint4 a, uint4 b, float acc)
{
    const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = fmaf(bf16_lo(x[i]), bf16_lo(y[i]), acc);
        acc = fmaf(bf16_hi(x[i]), bf16_hi(y[i]), acc);
    }
    return acc;
}

// STATES: only the state chain runs (no Q, no scores, no output); it writes
// the checkpoints the backward reads.
template <int DV, bool ABL, bool STATES>
__global__ void __launch_bounds__(kFwdThreads, 1)
fwd_sm100_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tck,
                 int ck_tma, const float *__restrict__ a, float b, int mode,
                 const int32_t *__restrict__ cu, int T, int64_t tokens, int H, int dk, int dv,
                 const float *__restrict__ h0, void *__restrict__ o, int o_f32,
                 float *__restrict__ hT, void *__restrict__ ckpt, int ck_bf16, int ckpt_stride,
                 int64_t n_slots, int n_docs, int seg_blk, const float *__restrict__ seg_init,
                 const int32_t *__restrict__ doc_order, DeviceStatus *st, uint64_t wait_ns, int stall)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    FwdSmem<DV> &sm = *reinterpret_cast<FwdSmem<DV> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = blockIdx.x * DV, h = blockIdx.y;
    // one document, or one segment of it (then the initial state comes from seg_init)
    const SegSpan span = seg_span(cu, T, tokens, n_docs,
                                   (seg_blk <= 0 && doc_order != nullptr) ? doc_order[blockIdx.z] : (int)blockIdx.z,
                                   seg_blk);
    if (!span.valid)
        return;
    const int n = span.n;
    DocSpan d;
    d.start = span.start;
    d.len = span.len;
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        if (tid == 0)
            set_status(st, BDLA_ERR_DEVICE, 0xA11u);
        return;
    }
    const int nblk = (int)((d.len + BT - 1) / BT);
    // test hook: the stalling role waits at this block (its second, or its only one)
    const int stall_blk = nblk > 1 ? 1 : 0;
    const int kpan = dk / 64;
    const size_t sstride = (size_t)dk * dv;
    const int64_t unit = (int64_t)n * H + h;
    const float *init = seg_blk > 0 ? seg_init : h0;
    const int64_t init_unit = seg_blk > 0 ? (int64_t)blockIdx.z * H + h : unit;

    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.full_qk[s], 1);
            mbar_init(&sm.empty_qk[s], 1);
            mbar_init(&sm.score_full[s], 1);
        }
        mbar_init(&sm.full_v, 1);
        mbar_init(&sm.empty_v, 1);
        mbar_init(&sm.p_ready, kEpiThreads);
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.p_free, 1);
        mbar_init(&sm.drain, 1);
        mbar_init(&sm.never, 1);
        sm.abort_flag = 0;
        sm.wait_ns = wait_ns;
        for (int r = 0; r < 3; ++r)
            sm.stall_at[r] = stall == r + 1 ? stall_blk : -1;
        mbar_fence_init();
    }
    if (kpan == 1) {   // dk = 64: the second dk panel of Q and K stays zero
        for (int e = tid; e < 2 * (int)(kPanel / 16); e += kFwdThreads) {
            const int s = e / (kPanel / 16), i = e % (kPanel / 16);
            reinterpret_cast<uint4 *>(sm.q[s] + kPanel)[i] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(sm.k[s] + kPanel)[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t t_score0 = tmem, t_o = tmem + 256, t_s = tmem + 384;
    volatile int *abort_flag = &sm.abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            const uint32_t qk_bytes = (uint32_t)kpan * (STATES ? 1u : 2u) * kPanel;
            const uint32_t v_bytes = (uint32_t)(DV / 64) * kPanel;
            int last_qk[2] = {-1, -1}, last_v = -1;
            bool consumed = true;
            for (int j = 0; j < nblk; ++j) {
                if (*abort_flag)
                    break;
                const int s = j & 1;
                const int t0 = (int)(d.start + (int64_t)j * BT);
                if (j >= 2 && !mbar_wait_lim(&sm.empty_qk[s], ((j >> 1) - 1) & 1, &sm.wait_ns)) {
                    consumed = false;
                    break;
                }
                mbar_arrive_expect_tx(&sm.full_qk[s], qk_bytes);
                for (int p = 0; p < kpan; ++p) {
                    if (!STATES)
                        tma_load_3d(sm.q[s] + p * kPanel, &tq, &sm.full_qk[s], p * 64, h, t0);
                    tma_load_3d(sm.k[s] + p * kPanel, &tk, &sm.full_qk[s], p * 64, h, t0);
                }
                last_qk[s] = j;
                // (test hook: the stalling producer waits on `never` here instead)
                const bool sp = j == sm.stall_at[0];
                if ((j >= 1 || sp) && !mbar_wait_lim(sp ? &sm.never : &sm.empty_v, sp ? 0u : (uint32_t)((j - 1) & 1), &sm.wait_ns)) {
                    consumed = false;
                    break;
                }
                mbar_arrive_expect_tx(&sm.full_v, v_bytes);
                for (int p = 0; p < DV / 64; ++p)
                    tma_load_3d(sm.v + p * kPanel, &tv, &sm.full_v, j0 + p * 64, h, t0);
                last_v = j;
            }
            if (!consumed || *abort_flag) {
                *abort_flag = 1;
                set_status(st, BDLA_ERR_TIMEOUT, 1u);
                // let the copies this thread started land before the CTA exits
                for (int s = 0; s < 2; ++s)
                    if (last_qk[s] >= 0)
                        mbar_wait(&sm.full_qk[s], (last_qk[s] >> 1) & 1, kWaitNs);
                if (last_v >= 0)
                    mbar_wait(&sm.full_v, last_v & 1, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_pv = idesc_bf16_f32(128, DV, false, true);
            const uint32_t id_kv = idesc_bf16_f32(128, DV, true, true);
            const uint32_t sq[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
            const uint32_t sk[2] = {smem_u32(sm.k[0]), smem_u32(sm.k[1])};
            const uint32_t sv = smem_u32(sm.v), ssb = smem_u32(sm.sb);
            bool ok = true;
            auto issue_qk = [&](int j) -> bool {
                const int s = j & 1;
                if (!mbar_wait_lim(&sm.full_qk[s], (j >> 1) & 1, &sm.wait_ns))
                    return false;
                // the P of block j - 2 (in this score buffer) has been read by its P V GEMM
                if (j >= 2 && !mbar_wait_lim(&sm.p_free, j & 1, &sm.wait_ns))
                    return false;
                tc_fence_after();
                for (int ks = 0; ks < dk / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * kPanel + (ks & 3) * 32;
                    umma_bf16(t_score0 + 128 * s, sdesc_sw128(sq[s] + off, 16, 1024),
                              sdesc_sw128(sk[s] + off, 16, 1024), id_qk, ks > 0);
                }
                umma_commit(&sm.score_full[s]);
                return true;
            };
            if (nblk > 0 && !STATES)
                ok = issue_qk(0);
            for (int j = 0; ok && j < nblk; ++j) {
                const int s = j & 1;
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                if (!STATES && j + 1 < nblk && !(ok = issue_qk(j + 1)))
                    break;
                // (test hook: the stalling MMA warp waits on `never` here instead)
                const bool sm_ = j == sm.stall_at[1];
                if (!mbar_wait_lim(sm_ ? &sm.never : &sm.p_ready, sm_ ? 0u : (uint32_t)(j & 1), &sm.wait_ns) ||
                    !mbar_wait_lim(&sm.full_v, j & 1, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (!STATES) {
                    // O = P V, P from tensor memory
                    for (int ks = 0; ks < BT / 16; ++ks)
                        umma_bf16_ts(t_o, t_score0 + 128 * s + ks * 8,
                                     sdesc_sw128(sv + ks * 2048, kPanel, 1024), id_pv, ks > 0);
                    umma_commit(&sm.p_free);   // the score buffer may take new scores once this GEMM is done
                    // O += (Q o e^{Lam}) S_in
                    for (int ks = 0; ks < dk / 16; ++ks)
                        umma_bf16(t_o, sdesc_sw128(sq[s] + (ks >> 2) * kPanel + (ks & 3) * 32, 16, 1024),
                                  sdesc_sw128(ssb + ks * 2048, kPanel, 1024), id_pv, 1);
                }
                // S += (K o e^{Lam_end - Lam})^T V
                for (int ks = 0; ks < BT / 16; ++ks)
                    umma_bf16(t_s, sdesc_sw128(sk[s] + ks * 2048, kPanel, 1024),
                              sdesc_sw128(sv + ks * 2048, kPanel, 1024), id_kv, 1);
                umma_commit(&sm.o_full);
                umma_commit(&sm.empty_qk[s]);
                umma_commit(&sm.empty_v);
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(st, BDLA_ERR_TIMEOUT, 2u);
            }
            // every MMA issued above has completed before TMEM is released
            umma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, kWaitNs);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        // Thread = row r (TMEM lane); the two warps of a lane quarter split the
        // columns: `half` takes 32-column chunks c with c % 2 == half.
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        {   // initial state
            uint32_t x[32];
#pragma unroll
            for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float val = (init != nullptr && r < dk)
                                          ? init[init_unit * sstride + (size_t)r * dv + j0 + c * 32 + i]
                                          : 0.0f;
                    x[i] = __float_as_uint(val);
                }
                tmem_st32(t_s + lane_off + c * 32, x);
            }
            tmem_st_wait();
        }

        // Output rows of block jb.  bf16: each half takes 64-column pairs; a
        // warp stages its 32 rows x 128 bytes in sb (free between the Q S GEMM
        // of block jb and the state copy of block jb+1) and 8 lanes write each
        // row's contiguous 128 bytes.  fp32 (parity workload): per-row stores.
        auto store_o = [&](int jb) {
            const int64_t t = d.start + (int64_t)jb * BT + r;
            const bool valid = (int64_t)jb * BT + r < d.len;
            if (o_f32) {
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                    uint32_t x[32];
                    tmem_ld32(t_o + lane_off + c * 32, x);
                    tmem_ld_wait();
                    if (!valid)
                        continue;
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<float *>(o) +
                                                           ((size_t)t * H + h) * dv + j0 + c * 32);
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        dst[k4] = make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
                }
                return;
            }
            const int64_t t_w = d.start + (int64_t)jb * BT + 32 * q4;
            const int n_valid = (int)(d.len - ((int64_t)jb * BT + 32 * q4));
            uint4 *st4 = reinterpret_cast<uint4 *>(sm.sb + (q4 + 4 * half) * 4096);
#pragma unroll
            for (int c2 = 0; c2 < DV / 64; ++c2) if ((c2 & 1) == half) {
                uint32_t xa[32], xb[32];
                tmem_ld32(t_o + lane_off + (2 * c2) * 32, xa);
                tmem_ld32(t_o + lane_off + (2 * c2 + 1) * 32, xb);
                tmem_ld_wait();
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    st4[lane * 8 + (k4 ^ (lane & 7))] =
                        make_uint4(pack_bf16(__uint_as_float(xa[8 * k4]), __uint_as_float(xa[8 * k4 + 1])),
                                   pack_bf16(__uint_as_float(xa[8 * k4 + 2]), __uint_as_float(xa[8 * k4 + 3])),
                                   pack_bf16(__uint_as_float(xa[8 * k4 + 4]), __uint_as_float(xa[8 * k4 + 5])),
                                   pack_bf16(__uint_as_float(xa[8 * k4 + 6]), __uint_as_float(xa[8 * k4 + 7])));
                    st4[lane * 8 + ((4 + k4) ^ (lane & 7))] =
                        make_uint4(pack_bf16(__uint_as_float(xb[8 * k4]), __uint_as_float(xb[8 * k4 + 1])),
                                   pack_bf16(__uint_as_float(xb[8 * k4 + 2]), __uint_as_float(xb[8 * k4 + 3])),
                                   pack_bf16(__uint_as_float(xb[8 * k4 + 4]), __uint_as_float(xb[8 * k4 + 5])),
                                   pack_bf16(__uint_as_float(xb[8 * k4 + 6]), __uint_as_float(xb[8 * k4 + 7])));
                }
                __syncwarp();
                __nv_bfloat16 *gbase = reinterpret_cast<__nv_bfloat16 *>(o) + ((size_t)t_w * H + h) * dv + j0 + c2 * 64;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int row = 4 * it + (lane >> 3), c8 = lane & 7;
                    const uint4 v = st4[row * 8 + (c8 ^ (row & 7))];
                    if (row < n_valid)
                        *reinterpret_cast<uint4 *>(gbase + (size_t)row * H * dv + 8 * c8) = v;
                }
                __syncwarp();
            }
        };

        bool ok = true;
        // logits of the first block; later blocks are fetched one block ahead
        float a_next = (nblk > 0 && r < d.len) ? a[(d.start + r) * H + h] : 0.0f;
        for (int j = 0; j < nblk; ++j) {
            const int s = j & 1;
            const int Lb = (int)(d.len - (int64_t)j * BT < BT ? d.len - (int64_t)j * BT : BT);
            const bool valid = r < Lb;
            const int tau = r >> 4;
            // ---- decay scalars of this block: Gamma from the logits
            // (the state-only pass serves both decay modes; the others are ABL-specific)
            const int md = STATES ? mode : (ABL ? BDLA_DECAY_NEG_SOFTPLUS : BDLA_DECAY_BOUNDED_SIGMOID);
            const float g = tile_gamma(valid ? log_decay(a_next, b, md) : 0.0f, lane);
            if (j + 1 < nblk) {
                const int64_t tn = (int64_t)(j + 1) * BT + r;
                a_next = tn < d.len ? a[(d.start + tn) * H + h] : 0.0f;
            }
            const int last = min(16 * tau + 15, Lb - 1);
            const float g_last = __shfl_sync(0xffffffffu, g, last & 31);
            const float gam_tau = (16 * tau < Lb) ? g_last : 0.0f;
            epi_sync();   // both halves are done with the previous block's column factors
            if (half == 0 && (r & 15) == 0) {
                sm.gam[tau] = gam_tau;
                sm.eg[tau] = expf(gam_tau);
            }
            if (half == 0) {
                if (ABL)
                    sm.gq[r] = g;
                sm.cdiag[r] = (valid && !ABL) ? expf(-g) : 0.0f;
                sm.coff[r] = valid ? expf(gam_tau - g) : 0.0f;
            }
            epi_sync();
            float G[BT / kChunk + 1];
            G[0] = 0.0f;
#pragma unroll
            for (int i = 0; i < BT / kChunk; ++i)
                G[i + 1] = G[i] + sm.gam[i];
            float Gt = 0.0f;
#pragma unroll
            for (int i = 0; i < BT / kChunk; ++i)
                Gt = (i == tau) ? G[i] : Gt;
            const float lend = G[BT / kChunk];
            const float lam_r = Gt + g;
            const float rt = valid ? expf(g) : 0.0f;
            const float qsc = valid ? expf(lam_r) : 0.0f;
            const float ksc = valid ? expf(lend - lam_r) : 0.0f;

            {
                // (test hook: the stalling epilogue waits on `never` here instead)
                const bool se = j == sm.stall_at[2];
                uint64_t *bar = se ? &sm.never : (STATES ? &sm.full_qk[s] : &sm.score_full[s]);
                ok = epi_all(mbar_wait_lim(bar, se ? 0u : (uint32_t)((j >> 1) & 1), &sm.wait_ns)) && !*abort_flag;
            }
            if (!ok)
                break;
            tc_fence_after();

            // explicit position-pair path for the diagonal tile (ablation): the
            // two warps of a lane quarter each compute 8 of the 16 pairs of a
            // row (half 0 the first 8), reading each 16-byte chunk of the q row
            // once; the values replace the GEMM ones in P below, in the warp
            // whose columns hold the rows' diagonal tile (chunk q4)
            uint32_t pair[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (ABL) {
                float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
                const int s0 = 16 * tau + 8 * half;   // first key row of this half's pairs
#pragma unroll 1
                for (int p = 0; p < kpan; ++p)
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const uint4 qa = *reinterpret_cast<const uint4 *>(sm.q[s] + p * kPanel + sw128_offset(r, c8));
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint4 kk = *reinterpret_cast<const uint4 *>(sm.k[s] + p * kPanel + sw128_offset(s0 + i, c8));
                            acc[i] = dot_bf16x8(qa, kk, acc[i]);
                        }
                    }
                uint32_t mine[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int sa = s0 + 2 * i, sb = sa + 1;
                    const float va = (valid && sa <= r) ? acc[2 * i] * expf(g - sm.gq[sa]) : 0.0f;
                    const float vb = (valid && sb <= r) ? acc[2 * i + 1] * expf(g - sm.gq[sb]) : 0.0f;
                    mine[i] = pack_bf16(va, vb);
                }
                const bool owner = (q4 & 1) == half;
                if (!owner) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        sm.abl_pair[r][i] = mine[i];
                }
                epi_sync();   // every thread is done with the raw K rows; the other half's pairs are in
                if (owner) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        pair[4 * half + i] = mine[i];
                        pair[4 * (1 - half) + i] = sm.abl_pair[r][i];
                    }
                }
            }
            // ---- fold the decay into Q and K in place (row r, half the chunks)
#pragma unroll 1
            for (int p = 0; p < kpan; ++p)
#pragma unroll
                for (int c8 = 4 * half; c8 < 4 * half + 4; ++c8) {
                    uint4 *ka = reinterpret_cast<uint4 *>(sm.k[s] + p * kPanel + sw128_offset(r, c8));
                    *ka = scale_bf16x8(*ka, ksc);
                    if (!STATES) {
                        uint4 *qa = reinterpret_cast<uint4 *>(sm.q[s] + p * kPanel + sw128_offset(r, c8));
                        *qa = scale_bf16x8(*qa, qsc);
                    }
                }
            // ---- P = decay-weighted causal scores, bf16 pairs written back into
            //      this block's score buffer (columns 16c .. 16c + 15 for chunk
            //      c), where the P V GEMM reads them
            if (!STATES) {
                uint32_t uu[2][16];
                // per source tile sg < tau: e^{G_tau - G_sg+1} e^{Gamma_t}, the
                // product of the tile decays e^{gamma} between sg and tau
                float f[BT / kChunk];
                {
                    float run = rt;
#pragma unroll
                    for (int sg = BT / kChunk - 1; sg >= 0; --sg) {
                        const bool below = sg < tau;
                        f[sg] = below ? run : (sg == tau ? rt : 0.0f);
                        run = below ? run * sm.eg[sg] : run;
                    }
                }
#pragma unroll
                for (int c = 0; c < BT / 32; ++c) if ((c & 1) == half) {
                    uint32_t (&u)[16] = uu[c >> 1];
                    if (c <= q4) {   // chunks above the warp's rows are causally zero
                        uint32_t x[32];
                        tmem_ld32(t_score0 + 128 * s + lane_off + c * 32, x);
                        tmem_ld_wait();
                        float pv[32];
#pragma unroll
                        for (int i4 = 0; i4 < 8; ++i4) {
                            const float4 co = *reinterpret_cast<const float4 *>(&sm.coff[c * 32 + 4 * i4]);
                            const float4 cd = *reinterpret_cast<const float4 *>(&sm.cdiag[c * 32 + 4 * i4]);
                            const float cov[4] = {co.x, co.y, co.z, co.w};
                            const float cdv[4] = {cd.x, cd.y, cd.z, cd.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 4 * i4 + e;
                                const int col = c * 32 + i;
                                const int sg = col >> 4;
                                const float sc = __uint_as_float(x[i]);
                                // branch-free: rows of one warp sit in two different tiles
                                const bool diag = (sg == tau);
                                const bool live = (sg < tau) || (!ABL && diag && col <= r);
                                const float w = diag ? cdv[e] * rt : cov[e] * f[sg];
                                pv[i] = live ? sc * w : 0.0f;
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            u[i] = pack_bf16(pv[2 * i], pv[2 * i + 1]);
                        if (ABL && c == q4) {
                            // the row's diagonal tile: columns 16 (tau & 1) .. + 15 of this chunk
                            const bool upper = (tau & 1) != 0;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                u[i] = upper ? u[i] : pair[i];
                                u[8 + i] = upper ? pair[i] : u[8 + i];
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            u[i] = 0u;
                    }
                }
                epi_sync();   // every score of the buffer is read before P lands on it
#pragma unroll
                for (int c = 0; c < BT / 32; ++c) if ((c & 1) == half)
                    tmem_st16(t_score0 + 128 * s + lane_off + 16 * c, uu[c >> 1]);
                tmem_st_wait();
            }

            // ---- output of the previous block
            if (j > 0) {
                if (ck_tma && warp == 2 && lane == 0)
                    tma_store_wait_read();   // previous checkpoint store is done with sb
                ok = epi_all(mbar_wait_lim(&sm.o_full, (j - 1) & 1, &sm.wait_ns)) && !*abort_flag;
                if (!ok)
                    break;
                tc_fence_after();
                if (!STATES) {
                    store_o(j - 1);
                    epi_sync();   // every warp's staging in sb is done before the state copy
                }
            }
            // ---- state: checkpoint, bf16 copy for the Q S GEMM, decay for the K V update
            {
                const float el = expf(lend);
                const int64_t jd = span.blk_base + j;   // doc-local block
                // checkpoints at block starts: strides that are multiples of the
                // block (every stride-th token) or divide it (every block start;
                // the states inside the block are filled in afterwards)
                const bool ck_block = ckpt != nullptr && (jd * BT) % ckpt_stride == 0 &&
                                      (ckpt_stride % BT == 0 || BT % ckpt_stride == 0);
                const bool wck = ck_block && !ck_tma && r < dk;   // fp32 checkpoints: per-row stores
                const size_t ckoff = wck ? ((size_t)h * n_slots +
                                            ckpt_slot(span.doc_start, n, jd * BT / ckpt_stride, ckpt_stride)) *
                                               sstride + (size_t)r * dv + j0
                                         : 0;
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                    uint32_t x[32];
                    tmem_ld32(t_s + lane_off + c * 32, x);
                    tmem_ld_wait();
                    uint32_t u[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        u[i] = pack_bf16(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
                    if (wck && !ck_bf16) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<float *>(ckpt) + ckoff + c * 32);
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4)
                            dst[k4] = make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
                    } else if (wck) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(ckpt) + ckoff + c * 32);
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            dst[k4] = make_uint4(u[4 * k4], u[4 * k4 + 1], u[4 * k4 + 2], u[4 * k4 + 3]);
                    }
                    if (!STATES || (ck_block && ck_tma)) {
                        unsigned char *sp = sm.sb + (c >> 1) * kPanel;
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            *reinterpret_cast<uint4 *>(sp + sw128_offset(r, (c & 1) * 4 + k4)) =
                                make_uint4(u[4 * k4], u[4 * k4 + 1], u[4 * k4 + 2], u[4 * k4 + 3]);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        x[i] = __float_as_uint(__uint_as_float(x[i]) * el);
                    tmem_st32(t_s + lane_off + c * 32, x);
                }
                tmem_st_wait();
                if (ck_block && ck_tma) {
                    // bf16 checkpoint: one TMA store of the swizzled state tile
                    fence_proxy_async_smem();
                    epi_sync();
                    if (warp == 2 && lane == 0) {
                        const int64_t slot = ckpt_slot(span.doc_start, n, jd * BT / ckpt_stride, ckpt_stride);
                        for (int p = 0; p < DV / 64; ++p)
                            tma_store_3d(&tck, sm.sb + p * kPanel, j0 + p * 64, 0, (int)((int64_t)h * n_slots + slot));
                        tma_store_commit();
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.p_ready);
        }
        if (ck_tma && warp == 2 && lane == 0)
            tma_store_wait_read();
        if (ok && nblk > 0) {
            ok = epi_all(mbar_wait_lim(&sm.o_full, (nblk - 1) & 1, &sm.wait_ns)) && !*abort_flag;
            if (ok) {
                tc_fence_after();
                if (!STATES)
                    store_o(nblk - 1);
            }
        }
        if (ok && hT != nullptr && span.last && r < dk) {
#pragma unroll
            for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                uint32_t x[32];
                tmem_ld32(t_s + lane_off + c * 32, x);
                tmem_ld_wait();
                float *row = hT + unit * sstride + (size_t)r * dv + j0 + c * 32;
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4)
                    reinterpret_cast<uint4 *>(row)[k4] =
                        make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0)
                set_status(st, BDLA_ERR_TIMEOUT, 3u);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem, 512);
}

// hT = h0 (or 0) for documents without tokens when the whole call has none.
__global__ void copy_state_kernel(const float *__restrict__ h0, float *__restrict__ hT, size_t n)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        hT[i] = h0 ? h0[i] : 0.0f;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

// 3-D map over a token-major bf16 tensor [tokens][H][d]: box = 64 features x
// 1 head x 128 tokens, 128-byte swizzle, zero fill past the last token.
bool make_token_map(CUtensorMap *map, const void *ptr, int d, int H, int64_t tokens)
{
    auto fn = encode_fn();
    if (fn == nullptr || ptr == nullptr || tokens <= 0)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)BT};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over bf16 state matrices [n_mats][dk][dv] (checkpoints): box = 64
// value columns x 128 key rows x 1 matrix, 128-byte swizzle (rows past dk
// read as zero), so a state lands in shared memory as a GEMM operand tile.
bool make_state_map(CUtensorMap *map, const void *ptr, int dk, int dv, int64_t n_mats)
{
    auto fn = encode_fn();
    if (fn == nullptr || ptr == nullptr || n_mats <= 0)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)dv, (cuuint64_t)dk, (cuuint64_t)n_mats};
    cuuint64_t strides[2] = {(cuuint64_t)dv * 2, (cuuint64_t)dk * dv * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)BT, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DV, bool ABL, bool STATES>
static cudaError_t launch_fwd_sm100_t(const Problem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                      const CUtensorMap &mv, const CUtensorMap &mck, int ck_tma,
                                      const float *a, const float *h0,
                                      void *o, int o_f32, float *hT, void *ckpt, int ck_bf16,
                                      int ckpt_stride, const SegPlan &seg)
{
    auto kern = fwd_sm100_kernel<DV, ABL, STATES>;
    const size_t smem = sizeof(FwdSmem<DV>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    const int64_t n_slots = ckpt ? ckpt_slots(p, ckpt_stride) : 0;
    dim3 grid(p.dv / DV, p.H, seg.seg_blk > 0 ? (unsigned)seg.n_slots : (unsigned)p.n_docs);
    const WaitCfg wc = wait_cfg(STATES ? BDLA_KERNEL_STATES : BDLA_KERNEL_FWD);
    kern<<<grid, kFwdThreads, smem, p.stream>>>(mq, mk, mv, mck, ck_tma, a, p.b, p.mode, p.cu, p.T, p.tokens, p.H, p.dk,
                                                p.dv, h0, o, o_f32, hT, ckpt, ck_bf16, ckpt_stride,
                                                n_slots, p.n_docs, seg.seg_blk, seg.buf, seg.order, p.st,
                                                wc.ns, wc.stall);
    return cudaGetLastError();
}

cudaError_t launch_fwd_sm100(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const float *a, const float *h0, void *o,
                             int o_f32, float *hT, void *ckpt, int ck_bf16, int ckpt_stride,
                             const SegPlan &seg)
{
    if (p.n_docs <= 0)
        return cudaSuccess;
    if (p.tokens == 0) {
        if (hT == nullptr)
            return cudaSuccess;
        const size_t nst = (size_t)p.n_docs * p.H * p.dk * p.dv;
        copy_state_kernel<<<(unsigned)((nst + 255) / 256 < 4096 ? (nst + 255) / 256 : 4096), 256, 0,
                            p.stream>>>(h0, hT, nst);
        return cudaGetLastError();
    }
    CUtensorMap mq, mk, mv;
    const bool states_only = (o == nullptr);
    if ((!states_only && !make_token_map(&mq, q, p.dk, p.H, p.tokens)) ||
        !make_token_map(&mk, k, p.dk, p.H, p.tokens) || !make_token_map(&mv, v, p.dv, p.H, p.tokens))
        return cudaErrorInvalidValue;
    if (states_only)
        mq = mk;
    const bool abl = p.mode == BDLA_DECAY_NEG_SOFTPLUS;
    // bf16 checkpoints at block starts leave by TMA store from the state tile
    CUtensorMap mck = mk;
    int ck_tma = 0;
    if (ckpt != nullptr && ck_bf16 && ckpt_stride % BT == 0) {
        if (!make_state_map(&mck, ckpt, p.dk, p.dv, (int64_t)p.H * ckpt_slots(p, ckpt_stride)))
            return cudaErrorInvalidValue;
        ck_tma = 1;
    }
#define BDLA_FWD_GO(DV_, ABL_, ST_)                                                                 \
    return launch_fwd_sm100_t<DV_, ABL_, ST_>(p, mq, mk, mv, mck, ck_tma, a, h0, o, o_f32, hT,      \
                                              ckpt, ck_bf16, ckpt_stride, seg)
    if (states_only) {
        if (p.dv == 64)
            BDLA_FWD_GO(64, false, true);
        BDLA_FWD_GO(128, false, true);
    }
    if (p.dv == 64) {
        if (abl)
            BDLA_FWD_GO(64, true, false);
        BDLA_FWD_GO(64, false, false);
    }
    if (abl)
        BDLA_FWD_GO(128, true, false);
    BDLA_FWD_GO(128, false, false);
#undef BDLA_FWD_GO
}

}  // namespace bdla
