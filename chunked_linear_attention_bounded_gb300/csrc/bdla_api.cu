// C ABI of libbdla.so: argument validation, workspace carving and launches.
// Every step of the computation runs in the kernels of this library; this
// file only checks arguments and enqueues work on the caller's stream.
#include <math.h>
#include <string.h>

#include "bdla_internal.h"

using namespace bdla;

namespace bdla {
KernelEvents g_kernel_events[BDLA_KERNEL_COUNT];
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_test_stall[BDLA_KERNEL_COUNT];

bdla_status check_dims(const bdla_dims &d, bool varlen, int n_docs)
{
    if (d.T < 0 || d.H < 1 || d.B < 1)
        return BDLA_ERR_SHAPE;
    if (varlen && (d.B != 1 || n_docs < 1))
        return BDLA_ERR_SHAPE;
    if ((varlen ? n_docs : d.B) > 65535)   // documents are a grid extent
        return BDLA_ERR_UNSUPPORTED;
    if (d.dk != 64 && d.dk != 128)
        return BDLA_ERR_UNSUPPORTED;
    if (d.dv != 64 && d.dv != 128 && d.dv != 256)
        return BDLA_ERR_UNSUPPORTED;
    return BDLA_OK;
}

bdla_status check_decay(float b, int chunk, int mode)
{
    if (chunk != kChunk)
        return BDLA_ERR_UNSUPPORTED;
    if (mode != BDLA_DECAY_BOUNDED_SIGMOID && mode != BDLA_DECAY_NEG_SOFTPLUS)
        return BDLA_ERR_UNSUPPORTED;
    if (mode == BDLA_DECAY_BOUNDED_SIGMOID) {
        if (!isfinite(b) || b > 0.0f)
            return BDLA_ERR_RANGE;
        // the bound must keep e^{-Gamma} = e^{chunk |b|} representable
        if ((double)chunk * fabs((double)b) > 80.0)
            return BDLA_ERR_RANGE;
    }
    return BDLA_OK;
}
}  // namespace bdla

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
    size_t gamma = 0;    // Gamma [H, tokens] fp32 (kernels that read it from memory)
    size_t dfac = 0;     // d lambda / d a [H, tokens] fp32 (backward)
    size_t states = 0;   // recomputed bf16 states for the backward, 0 if unused
    size_t seg = 0;      // segment summaries / initial states [slots, H, dk, dv] fp32
    size_t lsum = 0;     // segment log-decay sums [slots, H] fp32
    size_t order = 0;    // documents by decreasing length, int32 [n_docs]
    size_t total = 0;
};

int64_t total_tokens(const bdla_dims &d) { return (int64_t)d.B * d.T; }

constexpr int kBlock = 128;   // tokens per block of the tensor-core kernels

// The backward reads the state before every 128-token block from checkpoints
// whose stride divides 128 (fp32 or bf16); otherwise it recomputes them.
bool bwd_ckpt_usable(int ckpt_stride) { return ckpt_stride > 0 && kBlock % ckpt_stride == 0; }

// The segment plan depends on the sizes only (never on device data).
SegPlan plan_of(const bdla_dims &d, int n_docs)
{
    Problem p{};
    p.n_docs = n_docs;
    p.T = d.T;
    p.tokens = total_tokens(d);
    p.H = d.H;
    p.dk = d.dk;
    p.dv = d.dv;
    return plan_segments(p);
}

Layout layout(int op, const bdla_dims &d, int n_docs, int ckpt_stride)
{
    Layout L;
    size_t off = round_up(kStatusBytes);
    const int64_t tokens = total_tokens(d);
    const size_t per_head = round_up((size_t)tokens * sizeof(float));
    L.gamma = off;
    off += per_head * d.H;
    if (op == BDLA_OP_BWD) {
        L.dfac = off;
        off += per_head * d.H;
        // bf16 block states: recomputed, or converted from fp32 checkpoints
        // inside the blocks (strides below 128 are fp32 only)
        if (!bwd_ckpt_usable(ckpt_stride) || ckpt_stride < kBlock) {
            L.states = off;
            const int64_t slots = (tokens + kBlock - 1) / kBlock + n_docs;
            off += round_up((size_t)d.H * slots * d.dk * d.dv * 2);
        }
    }
    const SegPlan sp = plan_of(d, n_docs);
    if (sp.seg_blk > 0) {
        L.seg = off;
        off += round_up((size_t)sp.n_slots * d.H * d.dk * d.dv * sizeof(float));
        L.lsum = off;
        off += round_up((size_t)sp.n_slots * d.H * sizeof(float));
    } else if (n_docs > 1 && n_docs <= kMaxOrderedDocs) {
        L.order = off;
        off += round_up((size_t)n_docs * sizeof(int32_t));
    }
    L.total = off;
    return L;
}

bdla_status check_ws(void *ws, size_t ws_bytes, size_t need)
{
    if (ws == nullptr || ws_bytes < need || !aligned16(ws))
        return BDLA_ERR_WORKSPACE;
    return BDLA_OK;
}

Problem make_problem(const bdla_dims &d, const int32_t *cu, int n_docs, float b, int mode,
                     void *ws, void *stream)
{
    Problem p;
    p.cu = cu;
    p.n_docs = cu ? n_docs : d.B;
    p.T = cu ? d.T : d.T;
    p.tokens = total_tokens(d);
    p.H = d.H;
    p.dk = d.dk;
    p.dv = d.dv;
    p.b = b;
    p.mode = mode;
    p.st = reinterpret_cast<DeviceStatus *>(ws);
    p.stream = reinterpret_cast<cudaStream_t>(stream);
    return p;
}

#define BDLA_TRY(expr)                                                                             \
    do {                                                                                           \
        bdla_status s_ = (expr);                                                                   \
        if (s_ != BDLA_OK)                                                                         \
            return s_;                                                                             \
    } while (0)

// Segment plan of a call with its buffers carved from the workspace.
// (The order array is filled by launch_doc_check for packed calls.)
SegPlan seg_of(const bdla_dims &d, int n_docs, bool varlen, const Layout &L, void *ws)
{
    SegPlan sp = plan_of(d, n_docs);
    if (sp.seg_blk > 0) {
        sp.buf = reinterpret_cast<float *>(static_cast<char *>(ws) + L.seg);
        sp.lsum = reinterpret_cast<float *>(static_cast<char *>(ws) + L.lsum);
    } else if (varlen && L.order != 0) {
        sp.order = reinterpret_cast<const int32_t *>(static_cast<char *>(ws) + L.order);
    }
    return sp;
}

#define BDLA_CUDA(expr)                                                                            \
    do {                                                                                           \
        if ((expr) != cudaSuccess)                                                                 \
            return BDLA_ERR_CUDA;                                                                  \
    } while (0)

bdla_status fwd_impl(const void *q, const void *k, const void *v, const float *a, float b,
                     int chunk, const int32_t *cu, int n_docs, bool varlen, const float *h0,
                     void *o, bdla_dtype o_dtype, float *hT, void *ckpt, int ckpt_stride,
                     bdla_dtype ckpt_dtype, bdla_dims d, bdla_decay_mode mode, void *ws,
                     size_t ws_bytes, void *stream)
{
    BDLA_TRY(check_dims(d, varlen, n_docs));
    BDLA_TRY(check_decay(b, chunk, mode));
    const bool any_tokens = total_tokens(d) > 0;
    if ((any_tokens && (!q || !k || !v || !a || !o)) || (varlen && !cu))
        return BDLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(h0) ||
        !aligned16(hT) || !aligned16(ckpt) || !aligned16(a))
        return BDLA_ERR_ALIGN;
    if (o_dtype != BDLA_BF16 && o_dtype != BDLA_F32)
        return BDLA_ERR_DTYPE;
    if (ckpt && (ckpt_stride <= 0 || ckpt_stride % kChunk != 0))
        return BDLA_ERR_SHAPE;
    if (ckpt && ckpt_dtype != BDLA_F32 && ckpt_dtype != BDLA_BF16)
        return BDLA_ERR_DTYPE;
    if (ckpt && ckpt_dtype == BDLA_BF16 && ckpt_stride % kBlock != 0)
        return BDLA_ERR_UNSUPPORTED;
    const Layout L = layout(BDLA_OP_FWD, d, varlen ? n_docs : d.B, 0);
    BDLA_TRY(check_ws(ws, ws_bytes, L.total));
    Problem p = make_problem(d, varlen ? cu : nullptr, n_docs, b, mode, ws, stream);
    float *gamma = reinterpret_cast<float *>(static_cast<char *>(ws) + L.gamma);
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    const auto *vb = static_cast<const __nv_bfloat16 *>(v);
    // checkpoints the forward writes itself: strides that are multiples of the
    // 128-token block, or (fp32) block starts of strides dividing it
    const bool fused_ckpt = ckpt && ckpt_stride % kBlock == 0;
    const bool split_ckpt = ckpt && !fused_ckpt && kBlock % ckpt_stride == 0 && ckpt_dtype == BDLA_F32 &&
                            (int64_t)total_tokens(d) / kBlock + (varlen ? n_docs : d.B) <= INT32_MAX;
    const SegPlan seg = seg_of(d, p.n_docs, varlen, L, ws);
    {
        // the forward kernel takes Gamma from the logits itself; the segment
        // summaries and the in-block checkpoint passes read it from memory
        KernelMark mark_(BDLA_KERNEL_DECAY, p.stream);
        BDLA_CUDA(launch_doc_check(p, const_cast<int32_t *>(seg.order)));
        if (seg.seg_blk > 0 || (ckpt && !fused_ckpt))
            BDLA_CUDA(launch_decay(p, a, gamma, nullptr));
    }
    if (seg.seg_blk > 0) {
        // the state entering every segment
        {
        KernelMark mark_(BDLA_KERNEL_SEG, p.stream);
            BDLA_CUDA(launch_seg_summary(p, kb, vb, gamma, false, seg));
            BDLA_CUDA(launch_seg_scan(p, h0, false, seg));
        }
    }
    {
        KernelMark mark_(BDLA_KERNEL_FWD, p.stream);
        BDLA_CUDA(launch_fwd_sm100(p, qb, kb, vb, a, h0, o, o_dtype == BDLA_F32, hT,
                                   (fused_ckpt || split_ckpt) ? ckpt : nullptr, ckpt_dtype == BDLA_BF16,
                                   ckpt_stride, seg));
    }
    if (split_ckpt) {
        // the states inside each block, all blocks in parallel
        {
        KernelMark mark_(BDLA_KERNEL_STATES, p.stream);
            BDLA_CUDA(launch_ckpt_expand(p, kb, vb, gamma, static_cast<float *>(ckpt), ckpt_stride));
        }
    } else if (ckpt && !fused_ckpt) {
        // checkpoints inside the 128-token blocks: tile-serial state pass (fp32)
        {
        KernelMark mark_(BDLA_KERNEL_STATES, p.stream);
            BDLA_CUDA(launch_fwd_tile(p, qb, kb, vb, gamma, h0, nullptr, 0, nullptr,
                                      static_cast<float *>(ckpt), ckpt_stride, seg));
        }
    }
    return BDLA_OK;
}

bdla_status bwd_impl(const void *q, const void *k, const void *v, const float *a, float b,
                     int chunk, const int32_t *cu, int n_docs, bool varlen, const float *h0,
                     const void *dO, const float *dhT, const void *ckpt, int ckpt_stride,
                     bdla_dtype ckpt_dtype, float *dq, float *dk, float *dv, float *da, float *dh0,
                     bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream)
{
    BDLA_TRY(check_dims(d, varlen, n_docs));
    BDLA_TRY(check_decay(b, chunk, mode));
    const bool any_tokens = total_tokens(d) > 0;
    if ((any_tokens && (!q || !k || !v || !a || !dO || !dq || !dk || !dv || !da)) ||
        (varlen && !cu))
        return BDLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) || !aligned16(da) || !aligned16(a) ||
        !aligned16(h0) || !aligned16(dhT) || !aligned16(ckpt) || !aligned16(dh0))
        return BDLA_ERR_ALIGN;
    if (ckpt && (ckpt_stride <= 0 || ckpt_stride % kChunk != 0))
        return BDLA_ERR_SHAPE;
    if (ckpt && ckpt_dtype != BDLA_F32 && ckpt_dtype != BDLA_BF16)
        return BDLA_ERR_DTYPE;
    const int stride = ckpt ? ckpt_stride : 0;
    const int ck_bf16 = ckpt && ckpt_dtype == BDLA_BF16;
    const Layout L = layout(BDLA_OP_BWD, d, varlen ? n_docs : d.B, stride);
    BDLA_TRY(check_ws(ws, ws_bytes, L.total));
    Problem p = make_problem(d, varlen ? cu : nullptr, n_docs, b, mode, ws, stream);
    char *wsb = static_cast<char *>(ws);
    float *gamma = reinterpret_cast<float *>(wsb + L.gamma);
    float *dfac = reinterpret_cast<float *>(wsb + L.dfac);
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    const auto *vb = static_cast<const __nv_bfloat16 *>(v);
    const auto *dob = static_cast<const __nv_bfloat16 *>(dO);
    const SegPlan seg = seg_of(d, p.n_docs, varlen, L, ws);
    {
        // Gamma and d lambda / d a for the backward and the segment
        // summaries (the forward of the states pass forms Gamma itself)
        KernelMark mark_(BDLA_KERNEL_DECAY, p.stream);
        BDLA_CUDA(launch_doc_check(p, const_cast<int32_t *>(seg.order)));
        BDLA_CUDA(launch_decay(p, a, gamma, dfac));
    }
    const void *states = ckpt;
    int st_bf16 = ck_bf16, st_stride = stride;
    if (!bwd_ckpt_usable(stride)) {
        void *stb = wsb + L.states;
        if (seg.seg_blk > 0) {
            {
                KernelMark mark_(BDLA_KERNEL_SEG, p.stream);
                BDLA_CUDA(launch_seg_summary(p, kb, vb, gamma, false, seg));
                BDLA_CUDA(launch_seg_scan(p, h0, false, seg));
            }
        }
        {
        KernelMark mark_(BDLA_KERNEL_STATES, p.stream);
            BDLA_CUDA(launch_fwd_sm100(p, qb, kb, vb, a, h0, nullptr, 0, nullptr, stb, 1, kBlock, seg));
        }
        states = stb;
        st_bf16 = 1;
        st_stride = kBlock;
    }
    // fp32 checkpoints inside the blocks: the backward reads bf16 copies of
    // the block-start states, converted below, by TMA
    const bool convert = bwd_ckpt_usable(stride) && !ck_bf16 && stride < kBlock;
    if (convert) {
        states = wsb + L.states;
        st_bf16 = 1;
        st_stride = kBlock;
    }
    if (seg.seg_blk > 0) {
        // the adjoint entering every segment from its end
        {
        KernelMark mark_(BDLA_KERNEL_SEG, p.stream);
            BDLA_CUDA(launch_seg_summary(p, qb, dob, gamma, true, seg));
            BDLA_CUDA(launch_seg_scan(p, dhT, true, seg));
        }
    }
    float *part = nullptr;   // the second dv slice adds into dq, dk, da directly
    {
        KernelMark mark_(BDLA_KERNEL_BWD, p.stream);
        if (convert)
            BDLA_CUDA(launch_states_bf16(p, static_cast<const float *>(ckpt), stride,
                                         reinterpret_cast<__nv_bfloat16 *>(wsb + L.states)));
        BDLA_CUDA(launch_bwd_sm100(p, qb, kb, vb, dob, gamma, dfac, states, st_bf16, st_stride, dhT, dq,
                                   dk, dv, da, dh0, part, seg));
    }
    return BDLA_OK;
}

}  // namespace

extern "C" {

size_t bdla_workspace_bytes(int op, bdla_dims d, int n_docs, bdla_decay_mode mode, int ckpt_stride)
{
    (void)mode;
    const bool varlen = n_docs > 0;
    if (check_dims(d, varlen, n_docs) != BDLA_OK)
        return 0;
    return layout(op, d, varlen ? n_docs : d.B, ckpt_stride).total;
}

bdla_status bdla_decay(const float *a, float b, int chunk, const int32_t *cu_seqlens, int n_docs,
                       float *gamma, bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes,
                       void *stream)
{
    const bool varlen = cu_seqlens != nullptr;
    if (d.T < 0 || d.H < 1 || d.B < 1 || (varlen && (d.B != 1 || n_docs < 1)))
        return BDLA_ERR_SHAPE;
    BDLA_TRY(check_decay(b, chunk, mode));
    if (!a || !gamma)
        return BDLA_ERR_NULL;
    BDLA_TRY(check_ws(ws, ws_bytes, kStatusBytes));
    bdla_dims dd = d;
    dd.dk = 64;
    dd.dv = 64;
    Problem p = make_problem(dd, cu_seqlens, n_docs, b, mode, ws, stream);
    BDLA_CUDA(launch_doc_check(p, nullptr));
    BDLA_CUDA(launch_decay(p, a, gamma, nullptr));
    return BDLA_OK;
}

bdla_status bdla_fwd(const void *q, const void *k, const void *v, const float *a, float b,
                     int chunk, const float *h0, void *o, bdla_dtype o_dtype, float *hT,
                     void *ckpt, int ckpt_stride, bdla_dtype ckpt_dtype, bdla_dims d,
                     bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream)
{
    return fwd_impl(q, k, v, a, b, chunk, nullptr, 0, false, h0, o, o_dtype, hT, ckpt,
                    ckpt_stride, ckpt_dtype, d, mode, ws, ws_bytes, stream);
}

bdla_status bdla_fwd_varlen(const void *q, const void *k, const void *v, const float *a, float b,
                            int chunk, const int32_t *cu_seqlens, int n_docs, const float *h0,
                            void *o, bdla_dtype o_dtype, float *hT, void *ckpt, int ckpt_stride,
                            bdla_dtype ckpt_dtype, bdla_dims d, bdla_decay_mode mode, void *ws,
                            size_t ws_bytes, void *stream)
{
    return fwd_impl(q, k, v, a, b, chunk, cu_seqlens, n_docs, true, h0, o, o_dtype, hT, ckpt,
                    ckpt_stride, ckpt_dtype, d, mode, ws, ws_bytes, stream);
}

bdla_status bdla_bwd(const void *q, const void *k, const void *v, const float *a, float b,
                     int chunk, const float *h0, const void *dO, const float *dhT,
                     const void *ckpt, int ckpt_stride, bdla_dtype ckpt_dtype, float *dq,
                     float *dk, float *dv, float *da, float *dh0, bdla_dims d,
                     bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream)
{
    return bwd_impl(q, k, v, a, b, chunk, nullptr, 0, false, h0, dO, dhT, ckpt, ckpt_stride,
                    ckpt_dtype, dq, dk, dv, da, dh0, d, mode, ws, ws_bytes, stream);
}

bdla_status bdla_bwd_varlen(const void *q, const void *k, const void *v, const float *a, float b,
                            int chunk, const int32_t *cu_seqlens, int n_docs, const float *h0,
                            const void *dO, const float *dhT, const void *ckpt, int ckpt_stride,
                            bdla_dtype ckpt_dtype, float *dq, float *dk, float *dv, float *da,
                            float *dh0, bdla_dims d, bdla_decay_mode mode, void *ws,
                            size_t ws_bytes, void *stream)
{
    return bwd_impl(q, k, v, a, b, chunk, cu_seqlens, n_docs, true, h0, dO, dhT, ckpt,
                    ckpt_stride, ckpt_dtype, dq, dk, dv, da, dh0, d, mode, ws, ws_bytes, stream);
}

bdla_status bdla_read_device_status(void *ws, void *stream)
{
    if (ws == nullptr)
        return BDLA_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return BDLA_ERR_CUDA;
    unsigned int code = 0;
    if (cudaMemcpy(&code, ws, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
        return BDLA_ERR_CUDA;
    if (code != 0 && cudaMemset(ws, 0, kStatusBytes) != cudaSuccess)
        return BDLA_ERR_CUDA;
    return static_cast<bdla_status>(code);
}

const char *bdla_status_string(bdla_status s)
{
    switch (s) {
    case BDLA_OK: return "ok";
    case BDLA_ERR_NULL: return "a required pointer is NULL";
    case BDLA_ERR_SHAPE: return "a size is negative or inconsistent";
    case BDLA_ERR_DTYPE: return "an output or checkpoint dtype is not BDLA_BF16 or BDLA_F32";
    case BDLA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case BDLA_ERR_RANGE: return "decay bound out of range (b > 0, not finite, or chunk*|b| > 80)";
    case BDLA_ERR_UNSUPPORTED: return "unsupported chunk, head width, decay mode or document count";
    case BDLA_ERR_WORKSPACE: return "workspace NULL, misaligned or too small";
    case BDLA_ERR_CUDA: return "a CUDA runtime call failed";
    case BDLA_ERR_TIMEOUT: return "device: a bounded wait expired";
    case BDLA_ERR_DEVICE: return "device: malformed cu_seqlens or another device-side check";
    case BDLA_ERR_TOO_LARGE: return "more tokens than bdla_fwd_noalloc addresses (2^31 - 1)";
    }
    return "unknown status";
}

bdla_status bdla_set_kernel_events(int kernel, void *start_event, void *stop_event)
{
    if (kernel < 0 || kernel >= BDLA_KERNEL_COUNT)
        return BDLA_ERR_SHAPE;
    g_kernel_events[kernel].start.store(reinterpret_cast<cudaEvent_t>(start_event));
    g_kernel_events[kernel].stop.store(reinterpret_cast<cudaEvent_t>(stop_event));
    return BDLA_OK;
}

bdla_status bdla_decode(const void *q, const void *k, const void *v, const float *a, float b,
                        float *state, void *o, bdla_dtype o_dtype, bdla_dims d,
                        bdla_decay_mode mode, void *stream)
{
    if (d.T != 1)
        return BDLA_ERR_SHAPE;
    BDLA_TRY(check_dims(d, false, 0));
    BDLA_TRY(check_decay(b, kChunk, mode));
    if (!q || !k || !v || !a || !state || !o)
        return BDLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(o) ||
        !aligned16(a))
        return BDLA_ERR_ALIGN;
    if (o_dtype != BDLA_BF16 && o_dtype != BDLA_F32)
        return BDLA_ERR_DTYPE;
    BDLA_CUDA(launch_decode(d.B, d.H, d.dk, d.dv, static_cast<const __nv_bfloat16 *>(q),
                            static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v),
                            a, b, mode, state, o, o_dtype == BDLA_F32,
                            reinterpret_cast<cudaStream_t>(stream)));
    return BDLA_OK;
}

bdla_status bdla_set_seq_split(int blocks)
{
    g_seq_split.store(blocks);
    return BDLA_OK;
}

// ---------------------------------------------------------------- per-channel decay
namespace {

bdla_status check_vec(const bdla_dims &d, const int32_t *cu, int n_docs)
{
    BDLA_TRY(check_dims(d, cu != nullptr, n_docs));
    if (d.dv != 64 && d.dv != 128)
        return BDLA_ERR_UNSUPPORTED;
    return BDLA_OK;
}

// Workspace of the per-channel and delta-rule calls: status word, the
// document order (packed calls with 2 .. kMaxOrderedDocs documents), and for
// the backward the states of its own states pass.
size_t variant_order_bytes(bool varlen, int n_docs)
{
    return (varlen && n_docs > 1 && n_docs <= kMaxOrderedDocs) ? round_up((size_t)n_docs * 4) : 0;
}

// Packed calls: cu_seqlens checked on the device, and the documents longest
// first in the workspace's order region (2 .. kMaxOrderedDocs documents),
// else nullptr: one small kernel on the stream.
cudaError_t variant_order(const Problem &p, void *ws, bool varlen, const int32_t **order)
{
    *order = nullptr;
    if (!varlen)
        return cudaSuccess;
    int32_t *o = nullptr;
    if (variant_order_bytes(varlen, p.n_docs) != 0)
        o = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + round_up(kStatusBytes));
    *order = o;
    return launch_doc_check(p, o);
}

size_t vec_layout(int op, const bdla_dims &d, int n_docs, size_t *states_off, bool varlen = false)
{
    size_t off = round_up(kStatusBytes) + variant_order_bytes(varlen, n_docs);
    *states_off = off;
    if (op == BDLA_OP_BWD) {
        Problem p{};
        p.tokens = total_tokens(d);
        p.n_docs = n_docs;
        off += round_up((size_t)d.H * vec_state_slots(p) * d.dk * d.dv * 2);
    }
    return off;
}

}  // namespace

size_t bdla_tile_states_bytes(bdla_dims d, int n_docs)
{
    const bool varlen = n_docs > 0;
    if (check_vec(d, varlen ? reinterpret_cast<const int32_t *>(1) : nullptr, n_docs) != BDLA_OK)
        return 0;
    Problem p{};
    p.tokens = total_tokens(d);
    p.n_docs = varlen ? n_docs : d.B;
    return (size_t)d.H * vec_state_slots(p) * d.dk * d.dv * 2;
}

size_t bdla_workspace_bytes_vec(int op, bdla_dims d, int n_docs)
{
    const bool varlen = n_docs > 0;
    if (check_vec(d, varlen ? reinterpret_cast<const int32_t *>(1) : nullptr, n_docs) != BDLA_OK)
        return 0;
    size_t so;
    return vec_layout(op, d, varlen ? n_docs : d.B, &so, varlen);
}

bdla_status bdla_fwd_vec(const void *q, const void *k, const void *v, const float *a, float b, int chunk,
                         const int32_t *cu_seqlens, int n_docs, const float *h0, void *o,
                         bdla_dtype o_dtype, float *hT, void *states, bdla_dims d, bdla_decay_mode mode, void *ws,
                         size_t ws_bytes, void *stream)
{
    BDLA_TRY(check_vec(d, cu_seqlens, n_docs));
    BDLA_TRY(check_decay(b, chunk, mode));
    if (total_tokens(d) > 0 && (!q || !k || !v || !a || !o))
        return BDLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(h0) ||
        !aligned16(hT) || !aligned16(a) || !aligned16(states))
        return BDLA_ERR_ALIGN;
    if (o_dtype != BDLA_BF16 && o_dtype != BDLA_F32)
        return BDLA_ERR_DTYPE;
    size_t so;
    BDLA_TRY(check_ws(ws, ws_bytes, vec_layout(BDLA_OP_FWD, d, cu_seqlens ? n_docs : d.B, &so, cu_seqlens != nullptr)));
    Problem p = make_problem(d, cu_seqlens, n_docs, b, mode, ws, stream);
    KernelMark mark_(BDLA_KERNEL_FWD, p.stream);
    const int32_t *order;
    BDLA_CUDA(variant_order(p, ws, cu_seqlens != nullptr, &order));
    BDLA_CUDA(launch_vec_fwd(p, static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
                             static_cast<const __nv_bfloat16 *>(v), a, h0, o, o_dtype == BDLA_F32, hT,
                             static_cast<__nv_bfloat16 *>(states), order));
    return BDLA_OK;
}

bdla_status bdla_bwd_vec(const void *q, const void *k, const void *v, const float *a, float b, int chunk,
                         const int32_t *cu_seqlens, int n_docs, const float *h0, const void *dO,
                         const float *dhT, const void *states, float *dq, float *dk, float *dv, float *da,
                         float *dh0, bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream)
{
    BDLA_TRY(check_vec(d, cu_seqlens, n_docs));
    BDLA_TRY(check_decay(b, chunk, mode));
    if (total_tokens(d) > 0 && (!q || !k || !v || !a || !dO || !dq || !dk || !dv || !da))
        return BDLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(a) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(da) || !aligned16(h0) ||
        !aligned16(dhT) || !aligned16(dh0) || !aligned16(states))
        return BDLA_ERR_ALIGN;
    size_t so;
    BDLA_TRY(check_ws(ws, ws_bytes, vec_layout(states ? BDLA_OP_FWD : BDLA_OP_BWD, d, cu_seqlens ? n_docs : d.B, &so, cu_seqlens != nullptr)));
    Problem p = make_problem(d, cu_seqlens, n_docs, b, mode, ws, stream);
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    const auto *vb = static_cast<const __nv_bfloat16 *>(v);
    const __nv_bfloat16 *st = static_cast<const __nv_bfloat16 *>(states);
    const int32_t *order;
    if (st == nullptr) {   // no states from the forward: a states pass into the workspace
        auto *wst = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(ws) + so);
        KernelMark mark_(BDLA_KERNEL_STATES, p.stream);
        BDLA_CUDA(variant_order(p, ws, cu_seqlens != nullptr, &order));
        BDLA_CUDA(launch_vec_fwd(p, qb, kb, vb, a, h0, nullptr, 0, nullptr, wst, order));
        st = wst;
    }
    {
        KernelMark mark_(BDLA_KERNEL_BWD, p.stream);
        BDLA_CUDA(variant_order(p, ws, cu_seqlens != nullptr, &order));
        BDLA_CUDA(launch_vec_bwd(p, qb, kb, vb, static_cast<const __nv_bfloat16 *>(dO), a, st, dhT, dq,
                                 dk, dv, da, dh0, order));
    }
    return BDLA_OK;
}

// ---------------------------------------------------------------- gated delta rule
namespace {

size_t delta_layout(int op, const bdla_dims &d, int n_docs, size_t *states_off, bool varlen = false)
{
    size_t off = round_up(kStatusBytes) + variant_order_bytes(varlen, n_docs);
    *states_off = off;
    if (op == BDLA_OP_BWD) {
        Problem p{};
        p.tokens = total_tokens(d);
        p.n_docs = n_docs;
        off += round_up((size_t)d.H * delta_state_slots(p) * d.dk * d.dv * 2);
    }
    return off;
}

}  // namespace

size_t bdla_workspace_bytes_delta(int op, bdla_dims d, int n_docs)
{
    const bool varlen = n_docs > 0;
    if (check_vec(d, varlen ? reinterpret_cast<const int32_t *>(1) : nullptr, n_docs) != BDLA_OK)
        return 0;
    size_t so;
    return delta_layout(op, d, varlen ? n_docs : d.B, &so, varlen);
}

bdla_status bdla_fwd_delta(const void *q, const void *k, const void *v, const float *a, const float *beta,
                           float b, int chunk, const int32_t *cu_seqlens, int n_docs, const float *h0, void *o,
                           bdla_dtype o_dtype, float *hT, void *states, bdla_dims d, bdla_decay_mode mode, void *ws,
                           size_t ws_bytes, void *stream)
{
    BDLA_TRY(check_vec(d, cu_seqlens, n_docs));
    BDLA_TRY(check_decay(b, chunk, mode));
    if (total_tokens(d) > 0 && (!q || !k || !v || !a || !beta || !o))
        return BDLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(h0) ||
        !aligned16(hT) || !aligned16(a) || !aligned16(beta) || !aligned16(states))
        return BDLA_ERR_ALIGN;
    if (o_dtype != BDLA_BF16 && o_dtype != BDLA_F32)
        return BDLA_ERR_DTYPE;
    size_t so;
    BDLA_TRY(check_ws(ws, ws_bytes, delta_layout(BDLA_OP_FWD, d, cu_seqlens ? n_docs : d.B, &so, cu_seqlens != nullptr)));
    Problem p = make_problem(d, cu_seqlens, n_docs, b, mode, ws, stream);
    KernelMark mark_(BDLA_KERNEL_FWD, p.stream);
    const int32_t *order;
    BDLA_CUDA(variant_order(p, ws, cu_seqlens != nullptr, &order));
    BDLA_CUDA(launch_delta_fwd(p, static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
                               static_cast<const __nv_bfloat16 *>(v), a, beta, h0, o, o_dtype == BDLA_F32, hT,
                               static_cast<__nv_bfloat16 *>(states), order));
    return BDLA_OK;
}

bdla_status bdla_bwd_delta(const void *q, const void *k, const void *v, const float *a, const float *beta,
                           float b, int chunk, const int32_t *cu_seqlens, int n_docs, const float *h0,
                           const void *dO, const float *dhT, const void *states, float *dq, float *dk, float *dv,
                           float *da, float *dbeta, float *dh0, bdla_dims d, bdla_decay_mode mode, void *ws,
                           size_t ws_bytes, void *stream)
{
    BDLA_TRY(check_vec(d, cu_seqlens, n_docs));
    BDLA_TRY(check_decay(b, chunk, mode));
    if (total_tokens(d) > 0 && (!q || !k || !v || !a || !beta || !dO || !dq || !dk || !dv || !da || !dbeta))
        return BDLA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(a) ||
        !aligned16(beta) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(da) ||
        !aligned16(dbeta) || !aligned16(h0) || !aligned16(dhT) || !aligned16(dh0) || !aligned16(states))
        return BDLA_ERR_ALIGN;
    size_t so;
    BDLA_TRY(check_ws(ws, ws_bytes, delta_layout(states ? BDLA_OP_FWD : BDLA_OP_BWD, d, cu_seqlens ? n_docs : d.B, &so, cu_seqlens != nullptr)));
    Problem p = make_problem(d, cu_seqlens, n_docs, b, mode, ws, stream);
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    const auto *vb = static_cast<const __nv_bfloat16 *>(v);
    const __nv_bfloat16 *st = static_cast<const __nv_bfloat16 *>(states);
    const int32_t *order;
    if (st == nullptr) {   // no states from the forward: a states pass into the workspace
        auto *wst = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(ws) + so);
        KernelMark mark_(BDLA_KERNEL_STATES, p.stream);
        BDLA_CUDA(variant_order(p, ws, cu_seqlens != nullptr, &order));
        BDLA_CUDA(launch_delta_fwd(p, qb, kb, vb, a, beta, h0, nullptr, 0, nullptr, wst, order));
        st = wst;
    }
    {
        KernelMark mark_(BDLA_KERNEL_BWD, p.stream);
        BDLA_CUDA(variant_order(p, ws, cu_seqlens != nullptr, &order));
        BDLA_CUDA(launch_delta_bwd(p, qb, kb, vb, static_cast<const __nv_bfloat16 *>(dO), a, beta, st, dhT,
                                   dq, dk, dv, da, dbeta, dh0, order));
    }
    return BDLA_OK;
}

bdla_status bdla_set_wait_limit_ns(uint64_t ns)
{
    g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns);
    return BDLA_OK;
}

bdla_status bdla_set_test_stall(int kernel, int role)
{
    if (kernel < 0 || kernel >= BDLA_KERNEL_COUNT || role < BDLA_STALL_NONE || role > BDLA_STALL_EPILOGUE)
        return BDLA_ERR_SHAPE;
    g_test_stall[kernel].store(role);
    return BDLA_OK;
}

int bdla_version(void) { return 300; }

}  // extern "C"
