// Backward pass on the sm_100-family tensor cores: one CTA per (document,
// head) walks the document's 128-token blocks in reverse, carrying the state
// adjoint E (gradient w.r.t. the state at the block end from all later tokens)
// as an fp32 accumulator in tensor memory.
//
// Per block, with the pair weights w_ts = e^{Lam_t - Lam_s} built from the
// same two-level tile factors as the forward ("Engineering Long-Context
// Training for Trillion-Parameter MoE Models", sec. 3.2-3.3: with the bounded
// decay the diagonal 16-token tiles use the in-tile reciprocal like every
// other tile) and w_s = e^{Lam_end - Lam_s}:
//   P  = M o w o (Q K^T),  dA = dO V^T,  dP = M o w o dA
//   dq = e^{Lam_t} dO S_in^T + dP K
//   dk = (V o w_s) E^T + dP^T Q
//   dv = (K o w_s) E + P^T dO
//   E <- e^{Lam_end} E + (Q o e^{Lam})^T dO
// and the decay gradient from pair sums (W = P o dA):
//   dlam_r = sum_{u<r} X_u + sum_{t>=r} Y_t + e^{Lam_end} <S_in, E>
//   X_u = sum_{t>u} W_tu - sum_{s<u} W_us + k_u . dk_inter_u,   Y_t = q_t . dq_inter_t
//   da = dlam * d lambda / d a.
// P is causal, so the column sums come from the P^T dO GEMM:
//   sum_{t>=u} W_tu = v_u . (P^T dO)_u,   X_u = v_u . (P^T dO)_u - sum_{s<=u} W_us + k_u . dk_inter_u
// (the diagonal term cancels).  The row sums take the same bf16 P as that GEMM,
// so every pair inside the block cancels exactly in the prefix sums.
// S_in (the state before the block) comes from forward checkpoints.
//
// Phases of one block (MMA warp <-> eight epilogue warps, two per TMEM lane
// quarter splitting the columns).  Each GEMM is issued as soon as its operands
// and its accumulator are ready, in this order:
//   M1  C2 = dO V^T, C1 = Q K^T, C3 = dO S_in^T (each once the previous
//       block's output in that accumulator has been read out)
//   EA  P (smem) and dP (registers), W row sums, E -> bf16 copy;
//       E <- e^{Lam_end} E, C3 <- e^{Lam_t} C3 and Y
//   Mb  C2 = P^T dO (once P is in smem), C1 = V E^T (after EA)
//   Eb  dO -> e^{Lam} o dO, dP -> smem, C1 <- w_s o C1, k . dk_inter; then,
//       while Md runs, the W column sums v . (P^T dO) and K o w_s into V's
//       tile (V is not read again in the block; when dv < dk it does not
//       hold K, and K is scaled in place once Md has read it)
//   Mf1 E += Q^T (e^{Lam} o dO)        (once dO is rescaled)
//   Md  C3 += dP K (once dP is in smem), C1 += dP^T Q (after Eb)
//   Mf2 C2 += (K o w_s) E              (after the column sums)
//   Eg  dv = C2, dk = C1, dq = C3, da  (overlaps the next block's loads)
#include <cudaTypedefs.h>

#include "bdla_internal.h"
#include "bdla_sm100.cuh"

namespace bdla {

bool make_token_map(CUtensorMap *map, const void *ptr, int d, int H, int64_t tokens);
bool make_state_map(CUtensorMap *map, const void *ptr, int dk, int dv, int64_t n_mats);

namespace {
// 3-D map over a token-major fp32 gradient [tokens][H][d] for TMA stores:
// box = 32 features (128 bytes) x 1 head x 128 tokens, 128-byte swizzle.
bool make_grad_map(CUtensorMap *map, void *ptr, int d, int H, int64_t tokens)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    if (ptr == nullptr || tokens <= 0)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
    cuuint32_t box[3] = {32, 1, 128};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

namespace {

using namespace sm100;

constexpr int BT = 128;
constexpr int kEpiThreads = 256;                 // 8 epilogue warps, two per TMEM lane quarter
constexpr int kBwdThreads = 64 + kEpiThreads;    // + producer warp and MMA warp
constexpr uint32_t kPanel = 16384;
// drains of a CTA's own copies and MMAs before it exits keep the full limit
constexpr uint64_t kWaitNs = kDefaultWaitNs;

template <int DV>
struct BwdSmem {
    alignas(1024) unsigned char q[2 * kPanel];
    alignas(1024) unsigned char k[2 * kPanel];
    alignas(1024) unsigned char v[(DV / 64) * kPanel];
    alignas(1024) unsigned char dO[(DV / 64) * kPanel];
    // z and x are adjacent: together they stage fp32 output panels for TMA stores
    alignas(1024) unsigned char z[(DV / 64) * kPanel];   // S_in, then E: rows dk, panels dv
    alignas(1024) unsigned char x[2 * kPanel];           // P, then dP: rows t, panels s
    float cdiag[BT];
    float coff[BT];
    // per block parity, row and column half: v_s . (P^T dO)_s, sum_{s<=t} W_ts,
    // k.dk_inter, q.dq_inter, and per parity and epilogue warp <S_in, E>: a
    // block's decay gradient is summed up while the next block runs
    float colpart[2][2][BT];
    float rowpart[2][2][BT];
    float kdpart[2][2][BT];
    float ypart[2][2][BT];
    float scan[2][4];
    float gam[BT / kChunk];
    float se[2][8];
    float gq[BT];                  // Gamma per row (ablation diagonal path)
    float dgp[BT][kChunk + 1];     // ablation: diagonal-tile P, computed pair by pair
    float dgd[BT][kChunk + 1];     // ablation: diagonal-tile dP
    uint64_t full_in, free_in, z_ready, m1a_done, m1b_done, p_ready, ea_done, mb_done, dp_ready, eb_done, md_done,
        do_ready, ee_done, mf_done, acc_free_c1, acc_free_c2, acc_free_c3, drain, full_z, z_free;
    uint64_t never;       // nothing arrives here: the wait of the stall test hook
    uint64_t wait_ns;     // limit of the pipeline waits
    int stall_at[3];      // test hook: block at which producer / MMA / epilogue stall (-1: never)
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kMaxSmem = 232448;   // 227 KB opt-in shared memory per CTA
static_assert(sizeof(BwdSmem<128>) <= kMaxSmem && sizeof(BwdSmem<64>) <= kMaxSmem,
              "backward shared memory exceeds the per-CTA limit");

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

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// fp32 -> nearest bf16 -> fp32
__device__ __forceinline__ float bf16_round(float x)
{
    unsigned short h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return __uint_as_float((uint32_t)h << 16);
}

// Exclusive prefix sum over the 128 epilogue rows (row = 32 * q4 + lane).
__device__ __forceinline__ float block_exclusive_scan(float x, float *warp_tot, int q4, int lane, float &total)
{
    float incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off)
            incl += y;
    }
    if (lane == 31)
        warp_tot[q4] = incl;
    epi_sync();
    float before = 0.0f;
    total = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        before += (w < q4) ? warp_tot[w] : 0.0f;
        total += warp_tot[w];
    }
    return before + incl - x;
}

// Coalesced store of a warp's 32 rows x 32 fp32 values (lane = row):
// transposed through a 4 KB shared staging tile (16-byte chunks XOR-swizzled
// by row, conflict-free) so that each group of 8 lanes writes one row's 128
// contiguous bytes (ADD: adds them to what memory holds).  Rows >= n_valid
// are not written.
template <bool ADD = false>
__device__ __forceinline__ void warp_store_rows_f32(unsigned char *stage, const uint32_t (&x)[32],
                                                    float *gbase, size_t row_stride, int n_valid,
                                                    int lane)
{
    uint4 *st4 = reinterpret_cast<uint4 *>(stage);
#pragma unroll
    for (int k4 = 0; k4 < 8; ++k4)
        st4[lane * 8 + (k4 ^ (lane & 7))] = make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int row = 4 * it + (lane >> 3), c4 = lane & 7;
        const uint4 v = st4[row * 8 + (c4 ^ (row & 7))];
        if (ADD) {
            if (row < n_valid) {
                float *dst = gbase + (size_t)row * row_stride + 4 * c4;
                atomicAdd(dst, __uint_as_float(v.x));
                atomicAdd(dst + 1, __uint_as_float(v.y));
                atomicAdd(dst + 2, __uint_as_float(v.z));
                atomicAdd(dst + 3, __uint_as_float(v.w));
            }
        } else if (row < n_valid) {
            *reinterpret_cast<uint4 *>(gbase + (size_t)row * row_stride + 4 * c4) = v;
        }
    }
    __syncwarp();
}

// Row r (of dk rows) of the state before block j from the checkpoint array.
__device__ __forceinline__ void load_state_row(const void *states, int st_bf16, int stride,
                                               int64_t n_slots, int64_t doc_start, int n, int h, int64_t jd,
                                               int dk, int dv, int j0, int r, float (&out)[32], int c)
{
    const int64_t slot = ckpt_slot(doc_start, n, jd * BT / stride, stride);
    const size_t off = (((size_t)h * n_slots + slot) * dk + r) * dv + j0 + c * 32;
    if (st_bf16) {
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(states) + off);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const uint4 u = src[k4];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                out[8 * k4 + 2 * i] = bf16_lo(w[i]);
                out[8 * k4 + 2 * i + 1] = bf16_hi(w[i]);
            }
        }
    } else {
        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(states) + off);
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
            const float4 u = src[k4];
            out[4 * k4] = u.x;
            out[4 * k4 + 1] = u.y;
            out[4 * k4 + 2] = u.z;
            out[4 * k4 + 3] = u.w;
        }
    }
}

// ABL: unbounded -softplus decay; the diagonal 16-token tiles of P and dP
// are computed pair by pair on CUDA cores (explicit position-pair path).
// dv = 256 runs as two value slices of 128 columns, one launch each in stream
// order: dv is exact per slice, while dq, dk and da are partial sums; the
// first launch (ADD = false) stores them and the second (ADD = true, columns
// 128..255) adds its own to them, by TMA reduce-add for full blocks and by
// atomics for da and a document's last partial block.  (The kernel can still
// split slices over gridDim.z with partial sums written to `part`; the
// launcher does not use that.)
template <int DV, bool ABL, bool ADD>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_sm100_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap tst, int st_tma,
                 const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                 const __grid_constant__ CUtensorMap tdv, const __grid_constant__ CUtensorMap tdq1,
                 const __grid_constant__ CUtensorMap tdk1, int out_tma,
                 const float *__restrict__ gamma, const float *__restrict__ dfac,
                 const int32_t *__restrict__ cu, int T, int64_t tokens, int H, int dk, int dv,
                 const void *__restrict__ states, int st_bf16, int st_stride, int64_t n_slots,
                 const float *__restrict__ dhT, float *__restrict__ dq_base, float *__restrict__ dk_base,
                 float *__restrict__ dvv, float *__restrict__ da_base, float *__restrict__ dh0,
                 float *__restrict__ part, int64_t part_qk, int64_t part_a, int n_docs, int seg_blk,
                 const float *__restrict__ seg_init, const int32_t *__restrict__ doc_order,
                 DeviceStatus *st, uint64_t wait_ns, int stall)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BwdSmem<DV> &sm = *reinterpret_cast<BwdSmem<DV> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x;
    const int j0 = (ADD ? 1 : blockIdx.z) * DV;
    // slice 0 writes dq, dk, da; later slices write partial sums into `part`
    float *dq = (ADD || blockIdx.z == 0) ? dq_base : part + (size_t)(blockIdx.z - 1) * (2 * part_qk + part_a);
    float *dkk = (ADD || blockIdx.z == 0) ? dk_base : dq + part_qk;
    float *da = (ADD || blockIdx.z == 0) ? da_base : dq + 2 * part_qk;
    // TMA maps of this slice's dq and dk (slice 1: its partial sums), formed
    // where a store needs them
#define BDLA_MAP_DQ ((ADD || blockIdx.z == 0) ? &tdq : &tdq1)
#define BDLA_MAP_DK ((ADD || blockIdx.z == 0) ? &tdk : &tdk1)
    // one document, or one segment of it (then the adjoint after its last
    // token comes from seg_init)
    const SegSpan span = seg_span(cu, T, tokens, n_docs,
                                   (seg_blk <= 0 && doc_order != nullptr) ? doc_order[blockIdx.y] : (int)blockIdx.y,
                                   seg_blk);
    if (!span.valid)
        return;
    const int n = span.n;
    DocSpan d;
    d.start = span.start;
    d.len = span.len;
    if ((smem_u32(smem_raw) & 1023u) != 0u) {
        if (tid == 0)
            set_status(st, BDLA_ERR_DEVICE, 0xB11u);
        return;
    }
    const int nblk = (int)((d.len + BT - 1) / BT);
    // test hook: the stalling role waits at this block (its second, or its only one)
    const int stall_blk = nblk > 1 ? 1 : 0;
    const int kpan = dk / 64;
    // Mf reads K o w_s from V's tile when that tile has room for K
    const bool khat_v = DV / 64 >= kpan;
    const size_t sstride = (size_t)dk * dv;
    const int64_t unit = (int64_t)n * H + h;
    const float *einit = seg_blk > 0 ? seg_init : dhT;
    const int64_t einit_unit = seg_blk > 0 ? (int64_t)blockIdx.y * H + h : unit;

    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.full_in, 1);
        mbar_init(&sm.free_in, 1);
        mbar_init(&sm.z_ready, kEpiThreads);
        mbar_init(&sm.m1a_done, 1);
        mbar_init(&sm.m1b_done, 1);
        mbar_init(&sm.p_ready, kEpiThreads);
        mbar_init(&sm.ea_done, kEpiThreads);
        mbar_init(&sm.mb_done, 1);
        mbar_init(&sm.dp_ready, kEpiThreads);
        mbar_init(&sm.eb_done, kEpiThreads);
        mbar_init(&sm.md_done, 1);
        mbar_init(&sm.do_ready, kEpiThreads);
        mbar_init(&sm.ee_done, kEpiThreads);
        mbar_init(&sm.mf_done, 1);
        mbar_init(&sm.acc_free_c1, kEpiThreads);
        mbar_init(&sm.acc_free_c2, kEpiThreads);
        mbar_init(&sm.acc_free_c3, kEpiThreads);
        mbar_init(&sm.drain, 1);
        mbar_init(&sm.full_z, 1);
        mbar_init(&sm.z_free, 1);
        mbar_init(&sm.never, 1);
        sm.abort_flag = 0;
        sm.wait_ns = wait_ns;
        for (int r = 0; r < 3; ++r)
            sm.stall_at[r] = stall == r + 1 ? stall_blk : -1;
        mbar_fence_init();
    }
    if (kpan == 1) {   // dk = 64: the second dk panel of Q and K stays zero
        for (int e = tid; e < (int)(kPanel / 16); e += kBwdThreads) {
            reinterpret_cast<uint4 *>(sm.q + kPanel)[e] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(sm.k + kPanel)[e] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t t_e = tmem, t_c1 = tmem + 128, t_c2 = tmem + 256, t_c3 = tmem + 384;
    volatile int *abort_flag = &sm.abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdo);
            const uint32_t bytes = (uint32_t)kpan * 2u * kPanel + 2u * (uint32_t)(DV / 64) * kPanel;
            const uint32_t zbytes = (uint32_t)(DV / 64) * kPanel;
            int last_z = -1;
            if (st_tma)
                tma_prefetch_desc(&tst);
            int last = -1;
            bool ok = true;
            for (int jj = 0; jj < nblk; ++jj) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                const int j = nblk - 1 - jj;
                const int t0 = (int)(d.start + (int64_t)j * BT);
                // (test hook: the stalling producer waits on `never` here instead)
                const bool sp = jj == sm.stall_at[0];
                if ((jj > 0 || sp) && !mbar_wait_lim(sp ? &sm.never : &sm.free_in, sp ? 0u : (uint32_t)((jj - 1) & 1), &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&sm.full_in, bytes);
                for (int p = 0; p < kpan; ++p) {
                    tma_load_3d(sm.q + p * kPanel, &tq, &sm.full_in, p * 64, h, t0);
                    tma_load_3d(sm.k + p * kPanel, &tk, &sm.full_in, p * 64, h, t0);
                }
                for (int p = 0; p < DV / 64; ++p) {
                    tma_load_3d(sm.v + p * kPanel, &tv, &sm.full_in, j0 + p * 64, h, t0);
                    tma_load_3d(sm.dO + p * kPanel, &tdo, &sm.full_in, j0 + p * 64, h, t0);
                }
                last = jj;
                if (st_tma) {
                    // bf16 state before the block, straight into the z tile, once the
                    // previous block's output staging has left z
                    if (jj > 0 && !mbar_wait_lim(&sm.z_free, (jj - 1) & 1, &sm.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const int64_t slot = ckpt_slot(span.doc_start, n, (int64_t)(span.blk_base + j) * BT / st_stride, st_stride);
                    mbar_arrive_expect_tx(&sm.full_z, zbytes);
                    for (int p = 0; p < DV / 64; ++p)
                        tma_load_3d(sm.z + p * kPanel, &tst, &sm.full_z, j0 + p * 64, 0,
                                    (int)((int64_t)h * n_slots + slot));
                    last_z = jj;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(st, BDLA_ERR_TIMEOUT, 11u);
                if (last >= 0)
                    mbar_wait(&sm.full_in, last & 1, kWaitNs);
                if (last_z >= 0)
                    mbar_wait(&sm.full_z, last_z & 1, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t sq = smem_u32(sm.q), sk = smem_u32(sm.k), sv = smem_u32(sm.v);
            const uint32_t sdo = smem_u32(sm.dO), sz = smem_u32(sm.z), sx = smem_u32(sm.x);
            const uint32_t id_ss = idesc_bf16_f32(128, 128, false, false);   // C1 = Q K^T, C2 = dO V^T
            const uint32_t id_dqs = idesc_bf16_f32(128, dk, false, false);   // C3 = dO S_in^T
            const uint32_t id_pdo = idesc_bf16_f32(128, DV, true, true);     // C2 = P^T dO
            const uint32_t id_ve = idesc_bf16_f32(128, dk, false, false);    // C1 = V E^T
            const uint32_t id_dpq = idesc_bf16_f32(128, dk, true, true);     // C1 += dP^T Q
            const uint32_t id_dpk = idesc_bf16_f32(128, dk, false, true);    // C3 += dP K
            const uint32_t id_ke = idesc_bf16_f32(128, DV, false, true);     // C2 += K E
            const uint32_t id_qdo = idesc_bf16_f32(128, DV, true, true);     // E += Q^T dO
            auto kmaj = [](uint32_t base, int ks) {
                return sdesc_sw128(base + (ks >> 2) * kPanel + (ks & 3) * 32, 16, 1024);
            };
            auto mnmaj = [](uint32_t base, int ks) { return sdesc_sw128(base + ks * 2048, kPanel, 1024); };
            bool ok = true;
            for (int jj = 0; jj < nblk && ok; ++jj) {
                const uint32_t par = jj & 1;
                // (test hook: the stalling MMA warp waits on `never` instead of full_in)
                const bool sm_ = jj == sm.stall_at[1];
                // M1 accumulator by accumulator, each as soon as the previous
                // block's outputs have been read out of it (dv, then dk, then dq)
                if (*abort_flag || !mbar_wait_lim(sm_ ? &sm.never : &sm.full_in, sm_ ? 0u : par, &sm.wait_ns) ||
                    (jj > 0 && !mbar_wait_lim(&sm.acc_free_c2, (jj - 1) & 1, &sm.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < DV / 16; ++ks)
                    umma_bf16(t_c2, kmaj(sdo, ks), kmaj(sv, ks), id_ss, ks > 0);
                if (jj > 0 && !mbar_wait_lim(&sm.acc_free_c1, (jj - 1) & 1, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < dk / 16; ++ks)
                    umma_bf16(t_c1, kmaj(sq, ks), kmaj(sk, ks), id_ss, ks > 0);
                umma_commit(&sm.m1a_done);
                // S_in: straight from its TMA load, or once the epilogue converted it
                if (!mbar_wait_lim(st_tma ? &sm.full_z : &sm.z_ready, par, &sm.wait_ns) ||
                    (jj > 0 && !mbar_wait_lim(&sm.acc_free_c3, (jj - 1) & 1, &sm.wait_ns))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < DV / 16; ++ks)
                    umma_bf16(t_c3, kmaj(sdo, ks), kmaj(sz, ks), id_dqs, ks > 0);
                umma_commit(&sm.m1b_done);
                // Mb: P^T dO as soon as P is in x (and C2 read), V E^T once EA is done
                if (!mbar_wait_lim(&sm.p_ready, par, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < BT / 16; ++ks)
                    umma_bf16(t_c2, mnmaj(sx, ks), mnmaj(sdo, ks), id_pdo, ks > 0);
                if (!mbar_wait_lim(&sm.ea_done, par, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < DV / 16; ++ks)
                    umma_bf16(t_c1, kmaj(sv, ks), kmaj(sz, ks), id_ve, ks > 0);
                umma_commit(&sm.mb_done);
                // Mf's first GEMM, Q^T (e^{Lam} o dO) into E, as soon as dO is rescaled
                if (!mbar_wait_lim(&sm.do_ready, par, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < BT / 16; ++ks)
                    umma_bf16(t_e, mnmaj(sq, ks), mnmaj(sdo, ks), id_qdo, 1);
                // Md: dP K as soon as dP is in x, dP^T Q once C1 has been rescaled
                if (!mbar_wait_lim(&sm.dp_ready, par, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < BT / 16; ++ks)
                    umma_bf16(t_c3, kmaj(sx, ks), mnmaj(sk, ks), id_dpk, 1);
                if (!mbar_wait_lim(&sm.eb_done, par, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < BT / 16; ++ks)
                    umma_bf16(t_c1, mnmaj(sx, ks), mnmaj(sq, ks), id_dpq, 1);
                umma_commit(&sm.md_done);
                // Mf: K o w_s E into C2 once K o w_s is written and the column
                // sums are read
                if (!mbar_wait_lim(&sm.ee_done, par, &sm.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < dk / 16; ++ks)
                    umma_bf16(t_c2, kmaj(khat_v ? sv : sk, ks), mnmaj(sz, ks), id_ke, 1);
                umma_commit(&sm.mf_done);
                umma_commit(&sm.free_in);
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(st, BDLA_ERR_TIMEOUT, 12u);
            }
            umma_commit(&sm.drain);
            mbar_wait(&sm.drain, 0, kWaitNs);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        // Thread = row r (TMEM lane); `half` takes the 32-column chunks with
        // c % 2 == half (and half of each 64-wide smem row for the in-place folds).
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        {   // E <- dhT
            uint32_t x[32];
#pragma unroll
            for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = __float_as_uint((einit != nullptr && r < dk)
                                               ? einit[einit_unit * sstride + (size_t)r * dv + j0 + c * 32 + i]
                                               : 0.0f);
                tmem_st32(t_e + lane_off + c * 32, x);
            }
            tmem_st_wait();
        }
        // the block whose outputs are still pending (written in Eg)
        int pend_j = -1;
        // the block whose decay gradient is still pending: its partial sums
        // (parity da_par), its scalars and row
        bool da_pend = false, da_valid = false;
        int da_par = 0;
        float da_fac = 0.0f, da_lend = 0.0f, pend_fac = 0.0f, pend_lend = 0.0f;
        int64_t da_t = 0;
        uint32_t pend_par = 0;

        auto finish_block = [&]() -> bool {
            // Eg: outputs of block pend_j once Mf has completed
            const int jj = nblk - 1 - pend_j;
            if (!epi_all(mbar_wait_lim(&sm.mf_done, jj & 1, &sm.wait_ns)) || *abort_flag)
                return false;
            tc_fence_after();
            const int64_t t = d.start + (int64_t)pend_j * BT + r;
            const bool valid = (int64_t)pend_j * BT + r < d.len;
            // the warp's 32 rows start at token t_w; rows past the document end are skipped
            const int64_t t_w = d.start + (int64_t)pend_j * BT + 32 * q4;
            const int n_valid = (int)(d.len - ((int64_t)pend_j * BT + 32 * q4));
            const bool full_blk = d.len - (int64_t)pend_j * BT >= BT;
            // each accumulator is released to the next block's M1 once this
            // thread has read its last panel of it (dv, dk, then dq)
            bool c2_freed = false, c1_freed = false;
            if (DV == 128 && out_tma && full_blk && blockIdx.z <= 1) {
                // fp32 panels (32 columns) written by TMA stores.  Items: dv
                // panels, then dk panels, then dq panels.  The first n_a items
                // go two per round (one per column half) staged alternately in
                // z and x; the last four one per round (each half staging 16
                // of its columns) alternately in x's two panels, so that z is
                // released early for the next block's S_in.  A round waits
                // only for the reads of the round before it; x's last round
                // is awaited before the next block writes P into x.
                const int n_items = 2 * (dk / 32) + DV / 32;
                const int n_a = n_items - 4;           // 8 (dk = 128) or 4 (dk = 64)
                const int rounds = n_a / 2 + 4;
                const int t0s = (int)(d.start + (int64_t)pend_j * BT);
                auto item_col = [&](int it, int &coord, const CUtensorMap *&map) -> uint32_t {
                    if (it < DV / 32) {
                        coord = j0 + it * 32;
                        map = &tdv;
                        return t_c2 + it * 32;
                    }
                    if (it < DV / 32 + dk / 32) {
                        coord = (it - DV / 32) * 32;
                        map = BDLA_MAP_DK;
                        return t_c1 + (it - DV / 32) * 32;
                    }
                    coord = (it - DV / 32 - dk / 32) * 32;
                    map = BDLA_MAP_DQ;
                    return t_c3 + (it - DV / 32 - dk / 32) * 32;
                };
                const int c2_last = DV / 32 - 1, c1_last = DV / 32 + dk / 32 - 1;
                const int ka = n_a / 2;                  // two-item rounds
                for (int k = 0; k < rounds; ++k) {
                    const bool pair = k < ka;
                    unsigned char *buf = pair ? ((k & 1) ? sm.x : sm.z) : sm.x + ((k - ka) & 1) * kPanel;
                    if (k == ka) {
                        // the first single-item round reuses x, which the last
                        // two-item round may still be reading
                        if (warp == 2 && lane == 0)
                            tma_store_wait_read();
                        epi_sync();
                    }
                    if (pair) {
                        int coord;
                        const CUtensorMap *map;
                        const uint32_t col = item_col(2 * k + half, coord, map);
                        uint32_t x[32];
                        tmem_ld32(col + lane_off, x);
                        tmem_ld_wait();
                        unsigned char *sp = buf + half * kPanel;
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4)
                            *reinterpret_cast<uint4 *>(sp + sw128_offset(r, k4)) =
                                make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
                    } else {
                        int coord;
                        const CUtensorMap *map;
                        const uint32_t col = item_col(n_a + (k - ka), coord, map);
                        uint32_t x[16];
                        tmem_ld16(col + 16 * half + lane_off, x);
                        tmem_ld_wait();
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
                            *reinterpret_cast<uint4 *>(buf + sw128_offset(r, 4 * half + k4)) =
                                make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
                    }
                    {   // every item up to `read` has been read out of tensor memory by its reader
                        const int read = pair ? 2 * k + 1 : n_a + (k - ka);
                        if (!c2_freed && read >= c2_last) {
                            tc_fence_before();
                            mbar_arrive(&sm.acc_free_c2);
                            c2_freed = true;
                        }
                        if (!c1_freed && read >= c1_last) {
                            tc_fence_before();
                            mbar_arrive(&sm.acc_free_c1);
                            c1_freed = true;
                        }
                    }
                    fence_proxy_async_smem();
                    epi_sync();
                    if (warp == 2 && lane == 0) {
                        const int n_st = pair ? 2 : 1;
                        for (int hh = 0; hh < n_st; ++hh) {
                            int coord;
                            const CUtensorMap *map;
                            item_col(pair ? 2 * k + hh : n_a + (k - ka), coord, map);
                            if (ADD && map != &tdv)
                                tma_reduce_add_3d(map, buf + hh * kPanel, coord, h, t0s);
                            else
                                tma_store_3d(map, buf + hh * kPanel, coord, h, t0s);
                        }
                        tma_store_commit();
                        tma_store_wait_read1();   // the round before this one is read
                        if (k == ka - 1)
                            mbar_arrive(&sm.z_free);   // z's last round (ka - 2) is read
                    }
                    epi_sync();   // that round's buffers may be staged again
                }
            } else if (out_tma && full_blk && blockIdx.z <= 1) {
                // fp32 panels (32 columns) staged in z + x and written by TMA stores:
                // item i < dk/32: dq panel i; next dk/32: dk panels; then dv panels
                constexpr int kStagePanels = DV / 64 + 2;
                const int n_items = 2 * (dk / 32) + DV / 32;
                const int t0s = (int)(d.start + (int64_t)pend_j * BT);
                for (int base = 0; base < n_items; base += kStagePanels) {
#pragma unroll
                    for (int pi = 0; pi < kStagePanels; ++pi) {
                        const int it = base + pi;
                        if (it >= n_items || (it & 1) != half)
                            continue;
                        const int kind = it < dk / 32 ? 0 : (it < 2 * (dk / 32) ? 1 : 2);
                        const int c = kind == 0 ? it : (kind == 1 ? it - dk / 32 : it - 2 * (dk / 32));
                        const uint32_t col = (kind == 0 ? t_c3 : (kind == 1 ? t_c1 : t_c2)) + c * 32;
                        uint32_t x[32];
                        tmem_ld32(col + lane_off, x);
                        tmem_ld_wait();
                        unsigned char *sp = sm.z + pi * kPanel;
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4)
                            *reinterpret_cast<uint4 *>(sp + sw128_offset(r, k4)) =
                                make_uint4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
                    }
                    fence_proxy_async_smem();
                    epi_sync();
                    if (warp == 2 && lane == 0) {
                        for (int pi = 0; pi < kStagePanels && base + pi < n_items; ++pi) {
                            const int it = base + pi;
                            if (it < dk / 32) {
                                if (ADD)
                                    tma_reduce_add_3d(BDLA_MAP_DQ, sm.z + pi * kPanel, it * 32, h, t0s);
                                else
                                    tma_store_3d(BDLA_MAP_DQ, sm.z + pi * kPanel, it * 32, h, t0s);
                            } else if (it < 2 * (dk / 32)) {
                                if (ADD)
                                    tma_reduce_add_3d(BDLA_MAP_DK, sm.z + pi * kPanel, (it - dk / 32) * 32, h, t0s);
                                else
                                    tma_store_3d(BDLA_MAP_DK, sm.z + pi * kPanel, (it - dk / 32) * 32, h, t0s);
                            }
                            else
                                tma_store_3d(&tdv, sm.z + pi * kPanel, j0 + (it - 2 * (dk / 32)) * 32, h, t0s);
                        }
                        tma_store_commit();
                        tma_store_wait_read();
                    }
                    epi_sync();   // staging panels may be reused
                }
                if (warp == 2 && lane == 0)
                    mbar_arrive(&sm.z_free);   // the producer may load the next state into z
            } else {
                if (warp == 2 && lane == 0)
                    tma_store_wait_read();   // x may still be read by earlier stores
                epi_sync();
                unsigned char *stage = sm.x + (warp - 2) * 4096;   // x is free until the next EA
#pragma unroll
                for (int c = 0; c < 4; ++c) if ((c & 1) == half && c * 32 < dk) {
                    uint32_t x[32], y[32];
                    tmem_ld32(t_c3 + lane_off + c * 32, x);
                    tmem_ld32(t_c1 + lane_off + c * 32, y);
                    tmem_ld_wait();
                    warp_store_rows_f32<ADD>(stage, x, dq + ((size_t)t_w * H + h) * dk + c * 32, (size_t)H * dk, n_valid, lane);
                    warp_store_rows_f32<ADD>(stage, y, dkk + ((size_t)t_w * H + h) * dk + c * 32, (size_t)H * dk, n_valid, lane);
                }
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                    uint32_t x[32];
                    tmem_ld32(t_c2 + lane_off + c * 32, x);
                    tmem_ld_wait();
                    warp_store_rows_f32(stage, x, dvv + ((size_t)t_w * H + h) * dv + j0 + c * 32, (size_t)H * dv, n_valid, lane);
                }
                if (warp == 2 && lane == 0)
                    mbar_arrive(&sm.z_free);   // the producer may load the next state into z
            }
            tc_fence_before();
            if (!c2_freed)
                mbar_arrive(&sm.acc_free_c2);
            if (!c1_freed)
                mbar_arrive(&sm.acc_free_c1);
            mbar_arrive(&sm.acc_free_c3);
            // its decay gradient is summed up later, off the path to the next EA
            da_pend = true;
            da_valid = valid;
            da_t = t;
            da_par = (int)pend_par;
            da_fac = pend_fac;
            da_lend = pend_lend;
            return true;
        };

        // decay gradient of the pending block (both halves compute it; half 0 stores)
        auto block_da = [&]() {
            const int bp = da_par;
            const float X = (sm.colpart[bp][0][r] + sm.colpart[bp][1][r]) -
                            (sm.rowpart[bp][0][r] + sm.rowpart[bp][1][r]) +
                            (sm.kdpart[bp][0][r] + sm.kdpart[bp][1][r]);
            const float Yv = sm.ypart[bp][0][r] + sm.ypart[bp][1][r];
            float tx, ty;
            const float px = block_exclusive_scan(X, sm.scan[0], q4, lane, tx);
            const float py = block_exclusive_scan(Yv, sm.scan[1], q4, lane, ty);
            float se = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w)
                se += sm.se[bp][w];
            const float C = expf(da_lend) * se;
            if (da_valid && half == 0) {
                if (ADD)
                    atomicAdd(&da[(size_t)da_t * H + h], (px + (ty - py) + C) * da_fac);
                else
                    da[(size_t)da_t * H + h] = (px + (ty - py) + C) * da_fac;
            }
            epi_sync();   // the scan scratch is reused by the next block
            da_pend = false;
        };

        bool ok = true;
        for (int jj = 0; jj < nblk; ++jj) {
            const int j = nblk - 1 - jj;
            const uint32_t par = jj & 1;
            const int64_t t0 = d.start + (int64_t)j * BT;
            const int Lb = (int)(d.len - (int64_t)j * BT < BT ? d.len - (int64_t)j * BT : BT);
            const bool valid = r < Lb;
            const int tau = r >> 4;
            // the decay scalars load overlaps the previous block's output stores
            const float g = valid ? gamma[(int64_t)h * tokens + t0 + r] : 0.0f;
            const float fac = valid ? dfac[(int64_t)h * tokens + t0 + r] : 0.0f;
            if (pend_j >= 0) {
                ok = finish_block();
                if (!ok)
                    break;
                pend_j = -1;
            }
            // ---- decay scalars
            const int last = min(16 * tau + 15, Lb - 1);
            const float g_last = __shfl_sync(0xffffffffu, g, last & 31);
            const float gam_tau = (16 * tau < Lb) ? g_last : 0.0f;
            if (half == 0) {
                if ((r & 15) == 0)
                    sm.gam[tau] = gam_tau;
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
            const float wsc = valid ? expf(lend - lam_r) : 0.0f;

            const int bp = (int)par;   // parity of this block's partial sums
            if (st_tma) {
                // the producer loaded S_in (bf16) into z; <S_in, E> is taken in EA
                ok = epi_all(mbar_wait_lim(&sm.full_z, par, &sm.wait_ns)) && !*abort_flag;
                if (!ok)
                    break;
            } else {
                // ---- S_in row r -> bf16 copy (z) and <S_in, E>
                float se = 0.0f;
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                    uint32_t e[32];
                    tmem_ld32(t_e + lane_off + c * 32, e);
                    unsigned char *zp = sm.z + (c >> 1) * kPanel;
                    float s_in[32];
                    if (r < dk)
                        load_state_row(states, st_bf16, st_stride, n_slots, span.doc_start, n, h, span.blk_base + j, dk, dv, j0, r, s_in, c);
                    else
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            s_in[i] = 0.0f;
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        se = fmaf(s_in[i], __uint_as_float(e[i]), se);
                    uint32_t u[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        u[i] = pack_bf16(s_in[2 * i], s_in[2 * i + 1]);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        *reinterpret_cast<uint4 *>(zp + sw128_offset(r, (c & 1) * 4 + k4)) =
                            make_uint4(u[4 * k4], u[4 * k4 + 1], u[4 * k4 + 2], u[4 * k4 + 3]);
                }
                se = warp_sum(se);
                if (lane == 0)
                    sm.se[bp][warp - 2] = se;
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&sm.z_ready);
            }

            // ---- EA (P goes into x: the previous block's output stores are done reading it)
            if (warp == 2 && lane == 0)
                tma_store_wait_read();
            {
                // (test hook: the stalling epilogue waits on `never` instead of m1a_done)
                const bool se = jj == sm.stall_at[2];
                ok = epi_all(mbar_wait_lim(se ? &sm.never : &sm.m1a_done, se ? 0u : par, &sm.wait_ns)) && !*abort_flag;
            }
            if (!ok)
                break;
            tc_fence_after();
            if (ABL) {
                // explicit position-pair path for the diagonal tile:
                // P_ts = (q_t . k_s) e^{Gamma_t - Gamma_s}, dP_ts = (dO_t . v_s) e^{Gamma_t - Gamma_s};
                // each half takes 8 of the row's 16 pairs, reading each 16-byte
                // chunk of its q and dO rows once
                const int s0 = 16 * tau + 8 * half;
                float acc[8];
                // q_t . k_s first, then dO_t . v_s, so one set of accumulators is live
#pragma unroll 1
                for (int which = 0; which < 2; ++which) {
                    const unsigned char *xa = which == 0 ? sm.q : sm.dO;
                    const unsigned char *yb = which == 0 ? sm.k : sm.v;
                    const int npan = which == 0 ? kpan : DV / 64;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[i] = 0.0f;
#pragma unroll 1
                    for (int p = 0; p < npan; ++p)
#pragma unroll 2
                        for (int c8 = 0; c8 < 8; ++c8) {
                            const uint4 xr = *reinterpret_cast<const uint4 *>(xa + p * kPanel + sw128_offset(r, c8));
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const uint4 yr = *reinterpret_cast<const uint4 *>(yb + p * kPanel + sw128_offset(s0 + i, c8));
                                acc[i] = dot_bf16x8(xr, yr, acc[i]);
                            }
                        }
                    float (*dst)[kChunk + 1] = which == 0 ? sm.dgp : sm.dgd;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int sc = s0 + i;
                        dst[r][8 * half + i] = (valid && sc <= r) ? acc[i] * expf(g - sm.gq[sc]) : 0.0f;
                    }
                }
                epi_sync();   // all raw V rows read before any row is rescaled below
            }
            float rowsum = 0.0f;
            uint32_t dpk[BT / 4];   // dP row r on this half's two chunks, bf16 pairs
            float f[BT / kChunk];
#pragma unroll
            for (int sg = 0; sg < BT / kChunk; ++sg)
                f[sg] = sg < tau ? rt * expf(Gt - G[sg + 1]) : (sg == tau ? rt : 0.0f);
#pragma unroll
            for (int c = 0; c < BT / 32; ++c) if ((c & 1) == half) {
                const int cc = c >> 1;   // this half's chunk index 0..1
                float pv[32];   // bf16-rounded: the P the GEMMs and the row sums use
                uint32_t dpu[32];
                if (c <= q4) {
                    uint32_t xs[32], xa[32];
                    tmem_ld32(t_c1 + lane_off + c * 32, xs);
                    tmem_ld32(t_c2 + lane_off + c * 32, xa);
                    tmem_ld_wait();
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
                            const float sc = __uint_as_float(xs[i]);
                            const float av = __uint_as_float(xa[i]);
                            // branch-free: rows of one warp sit in two different tiles
                            const bool diag = (sg == tau);
                            const bool live = (sg < tau) || (diag && col <= r);
                            const float w = diag ? cdv[e] * rt : cov[e] * f[sg];
                            float p = live ? sc * w : 0.0f;
                            float dp = live ? av * w : 0.0f;
                            if (ABL && diag) {
                                p = (col <= r) ? sm.dgp[r][col & 15] : 0.0f;
                                dp = (col <= r) ? sm.dgd[r][col & 15] : 0.0f;
                            }
                            pv[i] = bf16_round(p);
                            rowsum = fmaf(pv[i], av, rowsum);   // p = 0 past the diagonal
                            dpu[i] = __float_as_uint(dp);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        pv[i] = 0.0f;
                        dpu[i] = 0u;
                    }
                }
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    dpk[cc * 16 + i] = pack_bf16(__uint_as_float(dpu[2 * i]), __uint_as_float(dpu[2 * i + 1]));
                uint32_t u[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    u[i] = pack_bf16(pv[2 * i], pv[2 * i + 1]);
                unsigned char *xp = sm.x + (c >> 1) * kPanel;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    *reinterpret_cast<uint4 *>(xp + sw128_offset(r, (c & 1) * 4 + k4)) =
                        make_uint4(u[4 * k4], u[4 * k4 + 1], u[4 * k4 + 2], u[4 * k4 + 3]);
            }
            sm.rowpart[bp][half][r] = rowsum;
            // P is in x and C2 (dO V^T) has been read: Mb's P^T dO may start
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.p_ready);
            // the C3 GEMM of M1 (dO S_in^T) reads S_in from z: it has completed
            // before E overwrites z (and before C3 is scaled below)
            ok = epi_all(mbar_wait_lim(&sm.m1b_done, par, &sm.wait_ns)) && !*abort_flag;
            if (!ok)
                break;
            tc_fence_after();
            // E in one pass: <S_in, E> with the S_in row in z (bf16 checkpoints),
            // then the bf16 copy of E over it (z) and E <- e^{Lam_end} E in
            // tensor memory (read only by Mf, after ea_done)
            {
                const float el = expf(lend);
                float se = 0.0f;
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                    uint32_t e[32];
                    tmem_ld32(t_e + lane_off + c * 32, e);
                    tmem_ld_wait();
                    unsigned char *zp = sm.z + (c >> 1) * kPanel;
                    uint32_t u[16];
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        uint4 *zq = reinterpret_cast<uint4 *>(zp + sw128_offset(r, (c & 1) * 4 + k4));
                        if (st_tma) {
                            const uint4 zz = *zq;
                            const uint32_t w4[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                se = fmaf(bf16_lo(w4[i]), __uint_as_float(e[8 * k4 + 2 * i]), se);
                                se = fmaf(bf16_hi(w4[i]), __uint_as_float(e[8 * k4 + 2 * i + 1]), se);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            u[4 * k4 + i] = pack_bf16(__uint_as_float(e[8 * k4 + 2 * i]),
                                                      __uint_as_float(e[8 * k4 + 2 * i + 1]));
                        *zq = make_uint4(u[4 * k4], u[4 * k4 + 1], u[4 * k4 + 2], u[4 * k4 + 3]);
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        e[i] = __float_as_uint(__uint_as_float(e[i]) * el);
                    tmem_st32(t_e + lane_off + c * 32, e);
                }
                if (st_tma) {
                    se = warp_sum(se);
                    if (lane == 0)
                        sm.se[bp][warp - 2] = se;
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.ea_done);

            // ---- while Mb runs (it touches neither E nor C3):
            // C3 <- e^{Lam_t} C3 (the inter-block part of dq) and Y_t = q_t . dq_inter_t
            float yv = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) if ((c & 1) == half && c * 32 < dk) {
                uint32_t x[32];
                tmem_ld32(t_c3 + lane_off + c * 32, x);
                tmem_ld_wait();
                const unsigned char *qp = sm.q + (c >> 1) * kPanel;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const uint4 qq = *reinterpret_cast<const uint4 *>(qp + sw128_offset(r, (c & 1) * 4 + k4));
                    const uint32_t w[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float a0 = __uint_as_float(x[8 * k4 + 2 * i]) * qsc;
                        const float a1 = __uint_as_float(x[8 * k4 + 2 * i + 1]) * qsc;
                        yv = fmaf(bf16_lo(w[i]), a0, yv);
                        yv = fmaf(bf16_hi(w[i]), a1, yv);
                        x[8 * k4 + 2 * i] = __float_as_uint(a0);
                        x[8 * k4 + 2 * i + 1] = __float_as_uint(a1);
                    }
                }
                tmem_st32(t_c3 + lane_off + c * 32, x);
            }
            sm.ypart[bp][half][r] = yv;
            tmem_st_wait();   // visible to Md and Mf through the fence before eb_done

            // ---- Eb: dO -> e^{Lam} o dO (then Mf's Q^T dO may start: Mb has read
            //      dO), dP -> smem (then Md's dP K may start), C1 <- w_s o C1 (the
            //      inter-block part of dk) and k . dk_inter
            ok = epi_all(mbar_wait_lim(&sm.mb_done, par, &sm.wait_ns)) && !*abort_flag;
            if (!ok)
                break;
            tc_fence_after();
#pragma unroll
            for (int p = 0; p < DV / 64; ++p)
#pragma unroll
                for (int c8 = 4 * half; c8 < 4 * half + 4; ++c8) {
                    uint4 *oa = reinterpret_cast<uint4 *>(sm.dO + p * kPanel + sw128_offset(r, c8));
                    *oa = scale_bf16x8(*oa, qsc);
                }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.do_ready);
#pragma unroll
            for (int c = 0; c < BT / 32; ++c) if ((c & 1) == half) {
                const int cc = c >> 1;
                unsigned char *xp = sm.x + (c >> 1) * kPanel;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    *reinterpret_cast<uint4 *>(xp + sw128_offset(r, (c & 1) * 4 + k4)) =
                        make_uint4(dpk[cc * 16 + 4 * k4], dpk[cc * 16 + 4 * k4 + 1],
                                   dpk[cc * 16 + 4 * k4 + 2], dpk[cc * 16 + 4 * k4 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.dp_ready);
            float kd = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) if ((c & 1) == half && c * 32 < dk) {
                uint32_t x[32];
                tmem_ld32(t_c1 + lane_off + c * 32, x);
                tmem_ld_wait();
                const unsigned char *kp = sm.k + (c >> 1) * kPanel;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const uint4 kk = *reinterpret_cast<const uint4 *>(kp + sw128_offset(r, (c & 1) * 4 + k4));
                    const uint32_t w[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        kd = fmaf(bf16_lo(w[i]), __uint_as_float(x[8 * k4 + 2 * i]), kd);
                        kd = fmaf(bf16_hi(w[i]), __uint_as_float(x[8 * k4 + 2 * i + 1]), kd);
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[i] = __float_as_uint(__uint_as_float(x[i]) * wsc);
                tmem_st32(t_c1 + lane_off + c * 32, x);
            }
            sm.kdpart[bp][half][r] = kd * wsc;
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.eb_done);
            // ---- while Md runs: the column sums of W: v_s . (P^T dO)_s (C2 and V stay untouched until Mf)
            {
                float vc = 0.0f;
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                    uint32_t x[32];
                    tmem_ld32(t_c2 + lane_off + c * 32, x);
                    tmem_ld_wait();
                    const unsigned char *vp = sm.v + (c >> 1) * kPanel;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const uint4 vv = *reinterpret_cast<const uint4 *>(vp + sw128_offset(r, (c & 1) * 4 + k4));
                        const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            vc = fmaf(bf16_lo(w[i]), __uint_as_float(x[8 * k4 + 2 * i]), vc);
                            vc = fmaf(bf16_hi(w[i]), __uint_as_float(x[8 * k4 + 2 * i + 1]), vc);
                        }
                    }
                }
                sm.colpart[bp][half][r] = vc;
            }

            if (khat_v) {
                // K o w_s for Mf into V's tile: this thread has read its part of
                // V row r above and writes only that part; Md reads K, not V
#pragma unroll 1
                for (int p = 0; p < kpan; ++p)
#pragma unroll
                    for (int c8 = 4 * half; c8 < 4 * half + 4; ++c8) {
                        const uint4 kk = *reinterpret_cast<const uint4 *>(sm.k + p * kPanel + sw128_offset(r, c8));
                        *reinterpret_cast<uint4 *>(sm.v + p * kPanel + sw128_offset(r, c8)) = scale_bf16x8(kk, wsc);
                    }
            } else {
                // ---- Ee: K -> K o w_s in place once Md has read K
                ok = epi_all(mbar_wait_lim(&sm.md_done, par, &sm.wait_ns)) && !*abort_flag;
                if (!ok)
                    break;
                tc_fence_after();
#pragma unroll 1
                for (int p = 0; p < kpan; ++p)
#pragma unroll
                    for (int c8 = 4 * half; c8 < 4 * half + 4; ++c8) {
                        uint4 *ka = reinterpret_cast<uint4 *>(sm.k + p * kPanel + sw128_offset(r, c8));
                        *ka = scale_bf16x8(*ka, wsc);
                    }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&sm.ee_done);
            // the previous block's decay gradient, while Md and Mf run
            if (da_pend)
                block_da();

            pend_j = j;
            pend_fac = fac;
            pend_lend = lend;
            pend_par = par;
        }
        if (ok && pend_j >= 0)
            ok = finish_block();
        if (ok && da_pend)
            block_da();
        if (ok && dh0 != nullptr && span.s == 0 && r < dk) {
#pragma unroll
            for (int c = 0; c < DV / 32; ++c) if ((c & 1) == half) {
                uint32_t x[32];
                tmem_ld32(t_e + lane_off + c * 32, x);
                tmem_ld_wait();
                float4 *row = reinterpret_cast<float4 *>(dh0 + unit * sstride + (size_t)r * dv + j0 + c * 32);
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4)
                    row[k4] = make_float4(__uint_as_float(x[4 * k4]), __uint_as_float(x[4 * k4 + 1]),
                                          __uint_as_float(x[4 * k4 + 2]), __uint_as_float(x[4 * k4 + 3]));
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0)
                set_status(st, BDLA_ERR_TIMEOUT, 13u);
        }
    }
    if (warp == 2 && lane == 0)
        tma_store_wait_all();   // output stores complete before the CTA's shared memory goes
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem, 512);
}
#undef BDLA_MAP_DQ
#undef BDLA_MAP_DK

template <int DV, bool ABL>
cudaError_t launch_bwd_sm100_t(const Problem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                               const CUtensorMap &mv, const CUtensorMap &mdo, const CUtensorMap &mst,
                               int st_tma, const CUtensorMap &mdq, const CUtensorMap &mdk,
                               const CUtensorMap &mdvv, int out_tma, const float *gamma,
                               const float *dfac, const void *states, int st_bf16, int st_stride,
                               const float *dhT, float *dq, float *dk, float *dv, float *da, float *dh0,
                               float *part, const SegPlan &seg)
{
    auto kern0 = bwd_sm100_kernel<DV, ABL, false>;
    auto kern1 = bwd_sm100_kernel<DV, ABL, true>;
    const size_t smem = sizeof(BwdSmem<DV>);
    const int slices = p.dv / DV;
    cudaError_t err = cudaFuncSetAttribute(kern0, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err == cudaSuccess && slices > 1)
        err = cudaFuncSetAttribute(kern1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    dim3 grid(p.H, seg.seg_blk > 0 ? (unsigned)seg.n_slots : (unsigned)p.n_docs, 1);
    const WaitCfg wc = wait_cfg(BDLA_KERNEL_BWD);
    // one launch per value slice, in stream order: the first stores dq, dk, da,
    // the second (ADD) adds its partial sums to them
    for (int slice = 0; slice < slices; ++slice) {
        (slice == 0 ? kern0 : kern1)<<<grid, kBwdThreads, smem, p.stream>>>(
            mq, mk, mv, mdo, mst, st_tma, mdq, mdk, mdvv, mdq, mdk, out_tma, gamma, dfac, p.cu, p.T, p.tokens, p.H,
            p.dk, p.dv, states, st_bf16, st_stride, ckpt_slots(p, st_stride), dhT, dq, dk, dv, da, dh0, part, 0, 0,
            p.n_docs, seg.seg_blk, seg.buf, seg.order, p.st, wc.ns, wc.stall);
        if ((err = cudaGetLastError()) != cudaSuccess)
            return err;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_sm100(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const __nv_bfloat16 *dO, const float *gamma,
                             const float *dfac, const void *states, int st_bf16, int st_stride,
                             const float *dhT, float *dq, float *dk, float *dv, float *da, float *dh0,
                             float *part, const SegPlan &seg)
{
    if (p.n_docs <= 0 || p.tokens == 0)
        return cudaSuccess;
    CUtensorMap mq, mk, mv, mdo;
    if (!make_token_map(&mq, q, p.dk, p.H, p.tokens) || !make_token_map(&mk, k, p.dk, p.H, p.tokens) ||
        !make_token_map(&mv, v, p.dv, p.H, p.tokens) || !make_token_map(&mdo, dO, p.dv, p.H, p.tokens))
        return cudaErrorInvalidValue;
    // bf16 states go straight into shared memory by TMA; fp32 ones are
    // converted by the epilogue
    CUtensorMap mst = mq;
    int st_tma = 0;
    if (st_bf16) {
        if (!make_state_map(&mst, states, p.dk, p.dv, (int64_t)p.H * ckpt_slots(p, st_stride)))
            return cudaErrorInvalidValue;
        st_tma = 1;
    }
    // fp32 gradients of full blocks leave by TMA stores
    CUtensorMap mdq = mq, mdk = mq, mdvv = mq;
    const int out_tma = make_grad_map(&mdq, dq, p.dk, p.H, p.tokens) &&
                        make_grad_map(&mdk, dk, p.dk, p.H, p.tokens) &&
                        make_grad_map(&mdvv, dv, p.dv, p.H, p.tokens);
    const bool abl = p.mode == BDLA_DECAY_NEG_SOFTPLUS;
    if (p.dv == 64)
        return abl ? launch_bwd_sm100_t<64, true>(p, mq, mk, mv, mdo, mst, st_tma, mdq, mdk, mdvv, out_tma, gamma, dfac, states, st_bf16,
                                                  st_stride, dhT, dq, dk, dv, da, dh0, part, seg)
                   : launch_bwd_sm100_t<64, false>(p, mq, mk, mv, mdo, mst, st_tma, mdq, mdk, mdvv, out_tma, gamma, dfac, states, st_bf16,
                                                   st_stride, dhT, dq, dk, dv, da, dh0, part, seg);
    return abl ? launch_bwd_sm100_t<128, true>(p, mq, mk, mv, mdo, mst, st_tma, mdq, mdk, mdvv, out_tma, gamma, dfac, states, st_bf16,
                                               st_stride, dhT, dq, dk, dv, da, dh0, part, seg)
               : launch_bwd_sm100_t<128, false>(p, mq, mk, mv, mdo, mst, st_tma, mdq, mdk, mdvv, out_tma, gamma, dfac, states, st_bf16,
                                                st_stride, dhT, dq, dk, dv, da, dh0, part, seg);
}

}  // namespace bdla
