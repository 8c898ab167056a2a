// Host-side launcher interface between the C ABI (bdla_api.cu) and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bdla_tuning.h"
#include "bdla_common.cuh"

namespace bdla {

struct Problem {
    const int32_t *cu;   // device cu_seqlens or nullptr (fixed-length)
    int n_docs;          // documents (B for fixed-length calls)
    int T;               // per-document length (fixed) or total tokens (varlen)
    int64_t tokens;      // total tokens in the tensors
    int H, dk, dv;
    float b;
    int mode;            // bdla_decay
    DeviceStatus *st;
    cudaStream_t stream;
};

// Host-side argument checks shared by the entry points: sizes (documents
// are a grid extent, so at most 65535; dk in {64, 128}; dv in {64, 128, 256})
// and the decay parameters (chunk 16; bounded mode needs b finite, b <= 0 and
// chunk * |b| <= 80).
bdla_status check_dims(const bdla_dims &d, bool varlen, int n_docs);
bdla_status check_decay(float b, int chunk, int mode);

// Slots of a checkpoint array with the given stride.
inline int64_t ckpt_slots(const Problem &p, int stride)
{
    return (p.tokens + stride - 1) / stride + p.n_docs;
}

// Sequence segments of one call (see SegSpan): seg_blk 128-token blocks per
// segment, 0 when every CTA walks a whole document.
struct SegPlan {
    int seg_blk = 0;
    int64_t n_slots = 0;     // segment slots (the grid extent that replaces n_docs)
    float *buf = nullptr;    // [n_slots][H][dk][dv] fp32: segment summaries, then initial states
    float *lsum = nullptr;   // [n_slots][H] summed log-decay of each segment
    // Without segments: documents by decreasing length (doc_order), or null
    // for index order.
    const int32_t *order = nullptr;
};

// Documents of packed calls with at most this many documents are taken
// longest first.
constexpr int kMaxOrderedDocs = 4096;
// Packed calls: checks cu_seqlens on the device (a bad offset is reported as
// BDLA_ERR_DEVICE) and, with `order` given and several documents, writes the
// documents by decreasing length into it.  Nothing for fixed-length calls.
cudaError_t launch_doc_check(const Problem &p, int32_t *order);

// Chooses the segment length for a problem: a fixed length set through
// bdla_set_seq_split, never (split < 0), or, by default, a cut into about
// four segments per SM when the (document, head, dv slice) units are fewer
// than the GPU's SMs.  Pointers are left null.
SegPlan plan_segments(const Problem &p);
extern std::atomic<int> g_seq_split;

// Events recorded around a kernel's launches (measurement hook, see
// bdla_set_kernel_events); null when unset.
struct KernelEvents {
    std::atomic<cudaEvent_t> start{nullptr}, stop{nullptr};
};
extern KernelEvents g_kernel_events[BDLA_KERNEL_COUNT];

// Every kernel's launches sit inside an NVTX range named after it, so a
// timeline tool shows the launches and the gaps between them; the caller's
// measurement events (if set) are recorded at the same two points.
inline const char *kernel_range_name(int kernel)
{
    static const char *names[BDLA_KERNEL_COUNT] = {"bdla:decay", "bdla:fwd", "bdla:bwd",
                                                   "bdla:states", "bdla:seg"};
    return names[kernel];
}
// Bounded waits (bdla_set_wait_limit_ns, bdla_set_test_stall): the limit of
// the pipeline waits and, per kernel, the role that stalls (test hook).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
extern std::atomic<uint64_t> g_wait_ns;
extern std::atomic<int> g_test_stall[BDLA_KERNEL_COUNT];
struct WaitCfg {
    uint64_t ns;   // limit of the pipeline waits
    int stall;     // BDLA_STALL_* role that waits on a barrier nothing arrives at
};
inline WaitCfg wait_cfg(int kernel) { return WaitCfg{g_wait_ns.load(), g_test_stall[kernel].load()}; }

// Scope of one kernel's launches: pushes the NVTX range and records the
// caller's start event on entry, records the stop event and pops the range on
// exit (early returns included).
class KernelMark {
  public:
    KernelMark(int kernel, cudaStream_t s) : kernel_(kernel), s_(s)
    {
        nvtxRangePushA(kernel_range_name(kernel));
        if (cudaEvent_t e = g_kernel_events[kernel].start.load())
            cudaEventRecord(e, s);
    }
    ~KernelMark()
    {
        if (cudaEvent_t e = g_kernel_events[kernel_].stop.load())
            cudaEventRecord(e, s_);
        nvtxRangePop();
    }
    KernelMark(const KernelMark &) = delete;
    KernelMark &operator=(const KernelMark &) = delete;

  private:
    int kernel_;
    cudaStream_t s_;
};

// One recurrent step per sequence: state <- e^{lambda} state + k v^T in place,
// o = state^T q.  q, k bf16 [B, H, dk]; v bf16 [B, H, dv]; a fp32 [B, H];
// state fp32 [B, H, dk, dv]; o bf16 or fp32 [B, H, dv].
cudaError_t launch_decode(int B, int H, int dk, int dv, const __nv_bfloat16 *q,
                          const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *a, float b,
                          int mode, float *state, void *o, int o_f32, cudaStream_t stream);

// gamma and dfac (d lambda / d a, may be nullptr) are head-major [H][tokens].
cudaError_t launch_decay(const Problem &p, const float *a, float *gamma, float *dfac);

// Tile-serial forward on CUDA cores.  Used with o == nullptr to write fp32
// checkpoints whose stride is below the 128-token block.
cudaError_t launch_fwd_tile(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                            const __nv_bfloat16 *v, const float *gamma, const float *h0, void *o,
                            int o_f32, float *hT, float *ckpt, int ckpt_stride, const SegPlan &seg);

// Fills fp32 checkpoints whose stride divides 128 inside each 128-token block
// from the block-start states the tensor-core forward wrote (one CTA per
// block, slice and head).
cudaError_t launch_ckpt_expand(const Problem &p, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                               const float *gamma, float *ckpt, int ckpt_stride);

// bf16 copies of the block-start states ([H][slots of stride 128][dk][dv])
// from fp32 checkpoints whose stride divides 128.
cudaError_t launch_states_bf16(const Problem &p, const float *ckpt, int ckpt_stride, __nv_bfloat16 *out);

// Tensor-core forward (tcgen05 / TMEM / TMA): o, hT and checkpoints whose
// stride is a multiple of 128 tokens, or the block-start ones of fp32
// checkpoints whose stride divides 128.
// o == nullptr runs the state chain only (checkpoints for the backward).
// With segments, seg.buf holds each segment's initial state (seg_scan).
// Gamma comes from the logits `a` ([tokens][H]) inside the kernel.
cudaError_t launch_fwd_sm100(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const float *a, const float *h0, void *o,
                             int o_f32, float *hT, void *ckpt, int ck_bf16, int ckpt_stride,
                             const SegPlan &seg);

// Segment summaries (tensor cores).  Forward (x = k, y = v): the state a
// segment adds from a zero start, sum_t e^{Lam_end - Lam_t} x_t y_t^T.
// Backward (x = q, y = dO): the adjoint a segment adds going back from a zero
// adjoint, sum_t e^{Lam_t} x_t y_t^T.  Lam is the inclusive cumulative
// log-decay from the segment start; seg.lsum receives Lam_end.
cudaError_t launch_seg_summary(const Problem &p, const __nv_bfloat16 *x, const __nv_bfloat16 *y,
                               const float *gamma, bool backward, const SegPlan &seg);
// Turns summaries into initial states in place.  Forward: S_0 = h0 (or 0),
// S_{i+1} = e^{lsum_i} S_i + sum_i.  Backward, from the document end:
// D_last = dhT (or 0), D_{i-1} = e^{lsum_i} D_i + sum_i.
cudaError_t launch_seg_scan(const Problem &p, const float *init, bool backward, const SegPlan &seg);

// Tensor-core backward.  `states` holds the state before every 128-token
// block: checkpoints whose stride divides 128, fp32 or bf16.  For dv = 256
// the value columns are split in two slices, launched one after the other:
// the first stores dq, dk, da and the second adds its partial sums to them
// (`part` is not used).  Gamma and d lambda / d a ([H][tokens]) come from the
// decay kernel.
cudaError_t launch_bwd_sm100(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const __nv_bfloat16 *dO, const float *gamma,
                             const float *dfac, const void *states, int st_bf16, int st_stride,
                             const float *dhT, float *dq, float *dk, float *dv, float *da, float *dh0,
                             float *part, const SegPlan &seg);


// Per-channel decay (a, da: [tokens][H][dk] fp32).  `order` (optional): the
// documents in launch order (longest first).  Forward: o, hT; with
// `states` non-null it runs the states pass instead (no q, no o): the bf16
// state before every 16-token tile into states [H][vec_state_slots][dk][dv].
int64_t vec_state_slots(const Problem &p);
cudaError_t launch_vec_fwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, const float *a, const float *h0, void *o, int o_f32,
                           float *hT, __nv_bfloat16 *states, const int32_t *order);
cudaError_t launch_vec_bwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, const __nv_bfloat16 *dO, const float *a,
                           const __nv_bfloat16 *states, const float *dhT, float *dq, float *dk, float *dv,
                           float *da, float *dh0, const int32_t *order);

// Gated delta rule (a, beta: [tokens][H] fp32).  Forward: o, hT; with
// `states` non-null it runs the states pass instead (no q, no o): the bf16
// state before every 16-token tile into states [H][delta_state_slots][dk][dv].
int64_t delta_state_slots(const Problem &p);
cudaError_t launch_delta_fwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const float *a, const float *beta, const float *h0, void *o,
                             int o_f32, float *hT, __nv_bfloat16 *states, const int32_t *order);
cudaError_t launch_delta_bwd(const Problem &p, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const __nv_bfloat16 *dO, const float *a, const float *beta,
                             const __nv_bfloat16 *states, const float *dhT, float *dq, float *dk, float *dv,
                             float *da, float *dbeta, float *dh0, const int32_t *order);

}  // namespace bdla
