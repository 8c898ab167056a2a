/*
 * bdla.h — C ABI of the bounded-decay chunked linear attention library
 * (libbdla.so, CUDA, sm_103a).
 *
 * The operation.  Gated linear attention with one scalar decay per (token,
 * head), evaluated in 16-token tiles ("Engineering Long-Context Training for
 * Trillion-Parameter MoE Models: Three Key Breakthroughs", sec. 3.1: matmuls
 * inside a tile, a recurrent state passed between tiles).  For every document
 * n and head h, with doc-local tokens t = 1..L:
 *     lambda_t = log g_t = b * sigmoid(a_t)        BDLA_DECAY_BOUNDED_SIGMOID
 *     lambda_t = -softplus(a_t)                    BDLA_DECAY_NEG_SOFTPLUS
 *     S_t = exp(lambda_t) S_{t-1} + k_t v_t^T,  S_0 = h0,  o_t = S_t^T q_t,
 *     hT = S_L.
 * The bounded form (same page, sec. 3.2; "Scaling Trillion-Parameter MoE and
 * Long-Context LLMs", sec. II) keeps the cumulative log-decay Gamma inside a
 * 16-token tile in [16 b, 0] = [-80, 0] for b = -5, so exp(+-Gamma) is finite
 * in bf16/fp32 and every tile, diagonal included, goes through the same
 * tensor-core GEMMs.  The -softplus form is the unbounded ablation: its
 * diagonal tiles take an explicit element-wise position-pair path.
 * No 1/sqrt(dk) scaling is applied (scale q beforehand).  b is a constant:
 * no gradient flows to it.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *    feature dimension innermost.  The library never allocates, frees or
 *    synchronises on these calls; its scratch comes from the caller's `ws`.
 *  - q, k, v, dO, o and the workspace must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream); every call is
 *    asynchronous and stream-ordered.
 *  - Host-detectable errors return a status before any launch.  Errors found
 *    on the device (a bounded wait that expired, malformed cu_seqlens) are
 *    recorded in a status word inside `ws`; read it with
 *    bdla_read_device_status.
 *
 * Shapes (bdla_dims): fixed-length calls take [B, T, H, d] tensors; the
 * _varlen calls take packed documents [1, T, H, d] with B = 1, T = total
 * tokens and device int32 cu_seqlens[n_docs + 1] (cu[0] = 0, non-decreasing,
 * cu[n_docs] = T).  Tiles restart at each document start; the last tile of a
 * document may be shorter than 16.  For fixed-length calls the documents are
 * the B rows (n_docs = B).
 *   q, k      bf16  [B, T, H, dk]          dk in {64, 128}; dk = 256 is refused
 *             (BDLA_ERR_UNSUPPORTED): the kernels hold the dk x dv state in
 *             tensor memory with dk on its 128 lanes
 *   v, dO     bf16  [B, T, H, dv]          dv in {64, 128, 256}
 *   a, da     fp32  [B, T, H]              decay logits and their gradient
 *   o         bf16 or fp32 [B, T, H, dv]
 *   dq, dk    fp32  [B, T, H, dk];  dv fp32 [B, T, H, dv]
 *   h0, hT, dh0, dhT   fp32 [n_docs, H, dk, dv]   (NULL = zero / not wanted)
 *   ckpt      fp32 or bf16 [H, n_slots, dk, dv], n_slots = ceil(B*T / stride) + n_docs;
 *             slot floor(cu[n] / stride) + n + c holds the state of document n
 *             before its doc-local token c*stride (slot c = 0 holds h0).
 *             bf16 checkpoints need a stride that is a multiple of 128; the
 *             backward uses checkpoints whose stride divides 128 (16, 32, 64,
 *             128), other strides make it recompute the states it needs.
 */
#ifndef BDLA_H
#define BDLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BDLA_OK = 0,
    BDLA_ERR_NULL = 1,         /* a required pointer is NULL */
    BDLA_ERR_SHAPE = 2,        /* a size is negative or inconsistent */
    BDLA_ERR_DTYPE = 3,        /* o_dtype / ckpt_dtype is not a bdla_dtype value */
    BDLA_ERR_ALIGN = 4,        /* a pointer is not 16-byte aligned */
    BDLA_ERR_RANGE = 5,        /* b > 0, b not finite, or chunk*|b| > 80 (bounded) */
    BDLA_ERR_UNSUPPORTED = 6,  /* chunk != 16, dk/dv outside the supported set, too many documents */
    BDLA_ERR_WORKSPACE = 7,    /* workspace NULL, misaligned or too small */
    BDLA_ERR_CUDA = 8,         /* a CUDA runtime call (launch, attribute) failed */
    BDLA_ERR_TIMEOUT = 9,      /* device: a bounded wait gave up */
    BDLA_ERR_DEVICE = 10,      /* device: malformed cu_seqlens or another device check */
    BDLA_ERR_TOO_LARGE = 11    /* bdla_fwd_noalloc: more than 2^31 - 1 tokens (B * T) */
} bdla_status;

typedef enum {
    BDLA_DECAY_BOUNDED_SIGMOID = 0,  /* lambda = b * sigmoid(a), b in [-80/chunk, 0] */
    BDLA_DECAY_NEG_SOFTPLUS = 1      /* lambda = -softplus(a); ablation, b ignored */
} bdla_decay_mode;

typedef enum { BDLA_BF16 = 0, BDLA_F32 = 1 } bdla_dtype;

typedef struct {
    int B;   /* documents (fixed-length calls) or 1 (varlen calls) */
    int T;   /* tokens per document (fixed) or total packed tokens (varlen) */
    int H;   /* heads */
    int dk;  /* key / query width */
    int dv;  /* value width */
} bdla_dims;

enum { BDLA_OP_FWD = 0, BDLA_OP_BWD = 1, BDLA_OP_DECAY = 2 };

/*
 * Bytes of device workspace an op needs.  `op` is BDLA_OP_*, `n_docs` the
 * document count of a varlen call (0 for fixed-length calls), `ckpt_stride`
 * the stride of the checkpoints the backward will be handed (0 if none).
 * The stride matters because a backward handed no usable checkpoints
 * (stride 0, or a stride that does not divide 128) recomputes the states
 * before every 128-token block into the workspace, and one handed fp32
 * checkpoints inside the blocks (a stride below 128 that divides it) writes
 * bf16 copies of the block-start states there.  `mode` does not change
 * the size.  Returns 0 on invalid dims.  The first 256 bytes of every
 * workspace are the device status word: zero them once after allocating the
 * workspace (bdla_read_device_status clears them again).
 */
size_t bdla_workspace_bytes(int op, bdla_dims d, int n_docs, bdla_decay_mode mode, int ckpt_stride);

/*
 * Decay kernel (the tile-local part of the method, sec. 3.1-3.2 of the first
 * page): gamma[h, t] = sum of lambda over the doc-local 16-token tile of t,
 * from the tile start through t (inclusive).  a: fp32 [B, T, H] (token-major);
 * gamma: fp32 [H, B*T] (head-major, the layout the attention kernels read).
 * cu_seqlens may be NULL for fixed-length inputs (then n_docs is ignored).
 */
bdla_status bdla_decay(const float *a, float b, int chunk, const int32_t *cu_seqlens,
                       int n_docs, float *gamma, bdla_dims d, bdla_decay_mode mode,
                       void *ws, size_t ws_bytes, void *stream);

/*
 * Forward pass.  Writes o (dtype o_dtype) and, when non-NULL, hT and the
 * state checkpoints ckpt (dtype ckpt_dtype) every ckpt_stride tokens
 * (ckpt_stride a multiple of 16; both ignored when ckpt is NULL).
 */
bdla_status bdla_fwd(const void *q, const void *k, const void *v, const float *a,
                     float b, int chunk, const float *h0,
                     void *o, bdla_dtype o_dtype, float *hT,
                     void *ckpt, int ckpt_stride, bdla_dtype ckpt_dtype,
                     bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream);

bdla_status bdla_fwd_varlen(const void *q, const void *k, const void *v, const float *a,
                            float b, int chunk, const int32_t *cu_seqlens, int n_docs,
                            const float *h0, void *o, bdla_dtype o_dtype, float *hT,
                            void *ckpt, int ckpt_stride, bdla_dtype ckpt_dtype,
                            bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes,
                            void *stream);

/*
 * Backward pass of the loss L with upstream gradients dO = dL/do and
 * dhT = dL/dhT (NULL = 0).  Writes dq, dk, dv, da (dL/da through the decay
 * parameterisation) and, when non-NULL, dh0.  ckpt (with its ckpt_stride) may
 * hold the forward's state checkpoints; NULL makes the backward recompute the
 * states it needs into the workspace (fp32 checkpoints with a stride below
 * 128 are converted there to bf16 block-start states first).
 */
bdla_status bdla_bwd(const void *q, const void *k, const void *v, const float *a,
                     float b, int chunk, const float *h0, const void *dO, const float *dhT,
                     const void *ckpt, int ckpt_stride, bdla_dtype ckpt_dtype,
                     float *dq, float *dk, float *dv, float *da, float *dh0,
                     bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream);

bdla_status bdla_bwd_varlen(const void *q, const void *k, const void *v, const float *a,
                            float b, int chunk, const int32_t *cu_seqlens, int n_docs,
                            const float *h0, const void *dO, const float *dhT,
                            const void *ckpt, int ckpt_stride, bdla_dtype ckpt_dtype,
                            float *dq, float *dk, float *dv, float *da, float *dh0,
                            bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes,
                            void *stream);

/*
 * Synchronises `stream`, returns the device status word recorded in `ws` by
 * earlier calls (BDLA_OK if none) and clears it.  BDLA_ERR_CUDA if the
 * synchronisation itself fails.  Only the first device-side error since the
 * last read is kept (later ones are dropped).
 */
bdla_status bdla_read_device_status(void *ws, void *stream);

/*
 * One recurrent (decode) step per sequence: the same recurrence for a single
 * new token against a resident state, e.g. after a chunked prefill whose hT
 * is the state (sec. 3.1 of the first page: the state passed between chunks;
 * its sec. 3.3: inference over long contexts).  For each sequence n and
 * head h:
 *     lambda = log_decay(a[n, h]),  state <- exp(lambda) state + k v^T,
 *     o = state^T q        (o reads the updated state, as o_t reads S_t)
 *   q, k   bf16 [B, H, dk];  v bf16 [B, H, dv];  a fp32 [B, H]
 *   state  fp32 [B, H, dk, dv], updated in place (the hT / h0 layout)
 *   o      bf16 or fp32 [B, H, dv]
 * d.T must be 1 (BDLA_ERR_SHAPE otherwise).  Same b / mode rules as
 * bdla_fwd.  No workspace, no device-side errors.  Bound by HBM: it reads and
 * writes the state once.
 */
bdla_status bdla_decode(const void *q, const void *k, const void *v, const float *a, float b,
                        float *state, void *o, bdla_dtype o_dtype, bdla_dims d,
                        bdla_decay_mode mode, void *stream);

/*
 * Forward pass for callers that cannot allocate device memory (no workspace
 * argument).  The pages have no counterpart: this is an interface for
 * callers, such as code running inside an allocator's callbacks or a runtime
 * that only hands out fixed buffers for inputs and outputs, which must not
 * call cudaMalloc.  Same operation and argument meaning as bdla_fwd for
 * fixed-length batches, without checkpoints.  The kernel forms the decay
 * cumsum from the logits itself, so the only scratch is a device status word,
 * a fixed variable inside the library that every GPU loading the library
 * holds (256 B) until exit.  It calls no cudaMalloc or cudaFree.  The first
 * call on each device looks up the word's device address; make that first
 * call before any stream capture.  Device-side errors (a bounded wait that
 * expired) are recorded in that word, which keeps the first error of any
 * call until bdla_noalloc_read_status reads and clears it.  Sizes are
 * checked as for bdla_fwd (B <= 65535), and B * T above 2^31 - 1 (the
 * kernels' 32-bit token coordinates) returns BDLA_ERR_TOO_LARGE before any
 * launch.
 */
bdla_status bdla_fwd_noalloc(const void *q, const void *k, const void *v, const float *a,
                             float b, int chunk, const float *h0, void *o, bdla_dtype o_dtype,
                             float *hT, bdla_dims d, bdla_decay_mode mode, void *stream);

/*
 * Status of the bdla_fwd_noalloc calls on the current device: synchronises
 * `stream`, returns the first device-side error recorded since the last read
 * (BDLA_OK if none) and clears it.  Allocates nothing; BDLA_ERR_CUDA if the
 * synchronisation or the copy fails.  No counterpart on the pages either.
 */
bdla_status bdla_noalloc_read_status(void *stream);

/*
 * Per-channel (vector) decay: one log-decay per (token, head, key channel),
 * the variant the first page's "per-position cumulative decay" also admits
 * ("Engineering Long-Context Training for Trillion-Parameter MoE Models:
 * Three Key Breakthroughs", sec. 3.1), with its sec. 3.2 parameterisations
 * applied channel by channel:
 *     lambda_t[i] = b * sigmoid(a_t[i])   or   -softplus(a_t[i]),
 *     S_t = diag(exp(lambda_t)) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t.
 * Row i of the dk x dv state decays by its own factor; the bound keeps each
 * channel's cumulative log-decay over a 16-token tile in [16 b, 0].
 * Arguments as for bdla_fwd / bdla_bwd except:
 *   a, da      fp32 [B, T, H, dk]   (one logit / gradient per key channel)
 *   cu_seqlens device int32 [n_docs + 1] for packed documents (B = 1), or
 *              NULL for fixed-length rows
 *   dk in {64, 128}, dv in {64, 128} (BDLA_ERR_UNSUPPORTED otherwise).
 *   states     optional device bf16 [H][slots][dk][dv], slots = tokens / 16 +
 *              n_docs (B for fixed-length rows) + 1, bdla_tile_states_bytes(d,
 *              n_docs) bytes, caller-owned: the state before every 16-token
 *              tile (tile c of document n in slot floor(doc_start / 16) + n + c).
 *              The forward writes it when non-NULL; the backward reads it when
 *              non-NULL (the forward's states of the same inputs), else runs
 *              its own states pass into the workspace.
 * Workspace: bdla_workspace_bytes_vec(op, ...) bytes, status word first; for
 * BDLA_OP_BWD it includes room for the backward's own states pass (unused
 * when the caller passes states).
 */
size_t bdla_tile_states_bytes(bdla_dims d, int n_docs);
size_t bdla_workspace_bytes_vec(int op, bdla_dims d, int n_docs);
bdla_status bdla_fwd_vec(const void *q, const void *k, const void *v, const float *a, float b,
                         int chunk, const int32_t *cu_seqlens, int n_docs, const float *h0,
                         void *o, bdla_dtype o_dtype, float *hT, void *states, bdla_dims d,
                         bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream);
bdla_status bdla_bwd_vec(const void *q, const void *k, const void *v, const float *a, float b,
                         int chunk, const int32_t *cu_seqlens, int n_docs, const float *h0,
                         const void *dO, const float *dhT, const void *states, float *dq,
                         float *dk, float *dv, float *da, float *dh0, bdla_dims d,
                         bdla_decay_mode mode, void *ws, size_t ws_bytes, void *stream);

/*
 * Gated delta rule with the bounded log-decay: the "Delta Net-style"
 * structure the first page names beside linear attention ("Engineering
 * Long-Context Training for Trillion-Parameter MoE Models: Three Key
 * Breakthroughs", sec. 3.1), with the sec. 3.2 decay in its gate.  The rule
 * is the published gated delta rule ("Gated Delta Networks: Improving Mamba2
 * with Delta Rule", 2024) for a dk x dv state read by o = S^T q:
 *     S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 *     g_t = exp(lambda_t),  o_t = S_t^T q_t.
 * Arguments as for bdla_fwd_vec / bdla_bwd_vec except:
 *   a, da        fp32 [B, T, H]   (one decay logit per token and head)
 *   beta, dbeta  fp32 [B, T, H]   write strengths beta_t (the caller maps its
 *                own logits into [0, 1]; keys are expected L2-normalised) and
 *                their gradient
 *   dk in {64, 128}, dv in {64, 128} (BDLA_ERR_UNSUPPORTED otherwise).
 *   states       optional, as for bdla_fwd_vec / bdla_bwd_vec (same layout,
 *                bdla_tile_states_bytes bytes).
 * Workspace: bdla_workspace_bytes_delta(op, ...) bytes, status word first; for
 * BDLA_OP_BWD it includes room for the backward's own states pass.
 */
size_t bdla_workspace_bytes_delta(int op, bdla_dims d, int n_docs);
bdla_status bdla_fwd_delta(const void *q, const void *k, const void *v, const float *a,
                           const float *beta, float b, int chunk, const int32_t *cu_seqlens,
                           int n_docs, const float *h0, void *o, bdla_dtype o_dtype, float *hT,
                           void *states, bdla_dims d, bdla_decay_mode mode, void *ws,
                           size_t ws_bytes, void *stream);
bdla_status bdla_bwd_delta(const void *q, const void *k, const void *v, const float *a,
                           const float *beta, float b, int chunk, const int32_t *cu_seqlens,
                           int n_docs, const float *h0, const void *dO, const float *dhT,
                           const void *states, float *dq, float *dk, float *dv, float *da,
                           float *dbeta, float *dh0,
                           bdla_dims d, bdla_decay_mode mode, void *ws, size_t ws_bytes,
                           void *stream);

/* Static English description of a status code. */
const char *bdla_status_string(bdla_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int bdla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BDLA_H */
