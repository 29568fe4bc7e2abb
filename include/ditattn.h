/*
 * ditattn.h -- C ABI of the DiT attention core on GB300 (sm_103a).
 *
 * Three operations, each one hand-written CUDA kernel launch (or a few):
 *
 *   dit_qk_norm_rope    per-head QK-RMSNorm + interleaved rotary embedding
 *   dit_attn_fwd        non-causal flash attention forward -> O and fp32 LSE,
 *                       over all keys or over one key chunk [kv_begin, kv_end)
 *   dit_attn_merge_lse  blockwise log-sum-exp merge of per-chunk (O_c, LSE_c)
 *   dit_attn_fwd_causal the attention with a causal mask (the pages' VLM path)
 *   dit_attn_fwd_update the attention of one key range LSE-merged into a running
 *                       result in its epilogue (the ring step's update_out_and_lse)
 *   dit_layer_norm_modulate, dit_rms_norm   row normalisations of the DiT block
 *   dit_quant_fp8_rows, dit_gemm_fp8        W8A8 fp8 projection
 *   dit_attention       the whole hot path on device buffers, one call
 *   dit_attention_host  the whole hot path from host buffers, copies pipelined
 *                       against the kernels
 *   dit_attention_ring_overlap  one rank's ring-attention overlap: local shard ||
 *                       gather of the remote shards, then their LSE-merged attention
 *
 * Conventions shared by every entry point
 *   - Tensors are device pointers owned by the caller.  Activations are
 *     [B, S, H, D] ("BSHD", element strides given where noted, last dim
 *     contiguous), the layout a DiT block produces before the transpose to
 *     BNSD.  LSE is fp32 [B, H, Sq], contiguous.
 *   - bf16 means IEEE bfloat16 (stored as 16-bit words); fp32 is IEEE binary32.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and allocates no device memory.  The library owns a few
 *     static device words (one per kernel family) that record a device-side
 *     wait that gave up (see dit_poll_device_error).
 *   - Argument errors return DIT_ERR_INVALID_ARG / DIT_ERR_UNSUPPORTED before
 *     anything is launched.  A launch failure returns DIT_ERR_CUDA.  Work of
 *     size zero (B, H or a sequence length 0) returns DIT_OK and launches
 *     nothing.
 *   - Head dim D must be 64 or 128.  Device pointers and every byte stride
 *     must be multiples of 16 bytes (the tensor-memory-accelerator rule) unless
 *     a function says otherwise.
 */
#ifndef DITATTN_H
#define DITATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */
struct CUevent_st;  /* cudaEvent_t is `struct CUevent_st *` */

typedef enum {
    DIT_OK = 0,
    DIT_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad range, misalignment, aliasing */
    DIT_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (e.g. D not 64/128) */
    DIT_ERR_CUDA = 3,        /* CUDA runtime/driver error at launch or tensor-map creation */
    DIT_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (reported by dit_poll_device_error) */
} dit_status;

typedef enum { DIT_BF16 = 0, DIT_F32 = 1 } dit_dtype;

/*
 * dit_qk_norm_rope -- QK-RMSNorm followed by interleaved RoPE, for Q and K in one launch.
 *
 * Defined by: "Cosmos Ascend NPU multi-card parallel optimisation notes",
 * section 3.2 (RMSNorm: x * rsqrt(mean(x^2) + eps) * weight, computed in fp32)
 * and section 3.3 (rotary embedding from precomputed cos/sin); "NPU Wan2.2-I2V
 * model inference optimisation practice", sections "NPU rms_norm operator
 * adaptation" and "NPU rotary_mul operator adaptation" (rotary_mode
 * "interleave": channels 2i and 2i+1 form one rotated pair).
 *
 * For every (b, s, h) row x of D channels of q (weights wq) and of k (wk):
 *   r      = 1 / sqrt(mean_d x_d^2 + eps)
 *   y_d    = x_d * r * w_d
 *   out_2i   = y_2i * c - y_2i+1 * s,   out_2i+1 = y_2i * s + y_2i+1 * c
 * with c = cos_tab[s, i], s = sin_tab[s, i].  fp32 arithmetic, one rounding to
 * bf16 at the end.  The norm is per head (over D), one weight vector shared by
 * all heads.
 *
 *   q, k          bf16 [B, S, H, D], contiguous.  Read only.
 *   q_out, k_out  bf16 [B, S, H, D], contiguous.  May equal q / k (in place);
 *                 any other overlap is invalid.
 *   wq, wk        fp32 [D].
 *   cos_tab, sin_tab  fp32 [S, D/2], contiguous (shared over B and H).
 *   eps           added to the mean square; must be >= 0.
 * Alignment: q, k, q_out, k_out, cos_tab, sin_tab 16-byte aligned; wq, wk 4-byte.
 */
dit_status dit_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out,
                            const float *wq, const float *wk, const float *cos_tab, const float *sin_tab,
                            int B, int S, int H, int D, float eps, struct CUstream_st *stream);

/*
 * dit_attn_fwd -- non-causal multi-head flash attention forward over a key range.
 *
 * Defined by: "NPU Wan2.2-I2V model inference optimisation practice", section
 * "NPU npu_fused_infer_attention_score operator adaptation" (bidirectional
 * attention on BNSD/BSND tensors with a softmax scale, whose second output is
 * the log-sum-exp); the key-range ("chunk") form is the per-block attention of
 * "feat: support Ascend NPU backend (torch_npu) for Qwen-Image pipelines -
 * #274", item 2 (ring attention over KV blocks) and of the Wan2.2 page,
 * section "Ring Attention Overlap".
 *
 * For every (b, h, i), over keys j in [kv_begin, kv_end):
 *   s_j = scale * q_i . k_j
 *   O_i = sum_j softmax(s)_j v_j
 *   LSE_i = ln sum_j exp(s_j)            (natural log, scale included)
 * kv_begin = 0, kv_end = Skv is full attention.
 *
 *   q            bf16 [B, Sq, H, D] with element strides q_strides = {b, s, h}
 *   k, v         bf16 [B, Skv, H, D], both with element strides kv_strides = {b, s, h}
 *   scale        softmax scale (e.g. 1/sqrt(D)); must be finite and > 0
 *   kv_begin, kv_end  0 <= kv_begin < kv_end <= Skv
 *   o            [B, Sq, H, D] of o_dtype (bf16 or fp32), element strides o_strides = {b, s, h};
 *                must not overlap q, k or v
 *   lse          fp32 [B, H, Sq], contiguous, 4-byte aligned
 * Strides are in elements; every stride times the element size must be a
 * multiple of 16 bytes, and every pointer except lse 16-byte aligned.
 * Tensor maps are built on the host per call; the kernel waits on device
 * barriers with a bound, and a wait that gives up is reported by
 * dit_poll_device_error (the results of that launch are then undefined).
 */
dit_status dit_attn_fwd(const void *q, const void *k, const void *v,
                        int B, int H, int Sq, int Skv, int D,
                        const int64_t q_strides[3], const int64_t kv_strides[3],
                        float scale, int kv_begin, int kv_end,
                        void *o, dit_dtype o_dtype, const int64_t o_strides[3], float *lse,
                        struct CUstream_st *stream);

/*
 * dit_attn_fwd_causal -- the same as dit_attn_fwd with a causal mask: query i
 * sees key j only if j <= i (absolute indices, top-left aligned, so a key
 * chunk [kv_begin, kv_end) masks by kv_begin + local index).  Rows that see no
 * key of the range get O = 0 and LSE = -inf, which dit_attn_merge_lse treats as
 * an empty block.
 *
 * Defined by: "Cosmos Ascend NPU multi-card parallel optimisation notes",
 * section 3.1 (the Qwen2.5-VL reasoner's attention: npu_fusion_attention with
 * sparse_mode=2, or scaled_dot_product_attention with is_causal=True) and "NPU
 * Wan2.2-I2V model inference optimisation practice", section "NPU
 * npu_fused_infer_attention_score operator adaptation" (next_tokens=0 when
 * causal).  Arguments, layouts and errors as for dit_attn_fwd.
 */
dit_status dit_attn_fwd_causal(const void *q, const void *k, const void *v,
                               int B, int H, int Sq, int Skv, int D,
                               const int64_t q_strides[3], const int64_t kv_strides[3],
                               float scale, int kv_begin, int kv_end,
                               void *o, dit_dtype o_dtype, const int64_t o_strides[3], float *lse,
                               struct CUstream_st *stream);

/*
 * dit_attn_fwd_update -- attention over one key range, merged into a running result.
 *
 * (o_acc, lse_acc) is the result of attention over earlier, disjoint key ranges
 * (any earlier dit_attn_fwd / dit_attn_fwd_update output).  This call computes
 * (O_c, LSE_c) over keys [kv_begin, kv_end) exactly as dit_attn_fwd (causal = 1:
 * as dit_attn_fwd_causal) and writes, per (b, h, i),
 *   L = ln(exp(lse_acc) + exp(LSE_c))
 *   o = exp(lse_acc - L) * o_acc + exp(LSE_c - L) * O_c,   lse = L
 * (both -inf: o = 0, lse = -inf).  O_c itself is never written: the merge runs
 * in the attention's epilogue, with the o_acc tile brought into shared memory
 * by the tensor-memory accelerator.
 *
 * Defined by: "feat: support Ascend NPU backend (torch_npu) for Qwen-Image
 * pipelines - #274", item 2 (ring attention: after each KV block the block's
 * output and LSE are folded into the running ones by update_out_and_lse), and
 * the Wan2.2 page, section "Ring Attention Overlap" (two attentions combined by
 * their LSEs).
 *
 *   o_acc        [B, Sq, H, D] of acc_dtype (bf16 or fp32), element strides acc_strides
 *   lse_acc      fp32 [B, H, Sq], contiguous, 4-byte aligned
 *   o, lse       as for dit_attn_fwd
 *   causal       0 or 1
 * In place is allowed: o == o_acc with the same dtype and strides, and/or
 * lse == lse_acc.  Otherwise the running result must not overlap o or lse.
 * Other arguments, layouts and errors as for dit_attn_fwd.
 */
dit_status dit_attn_fwd_update(const void *q, const void *k, const void *v,
                               int B, int H, int Sq, int Skv, int D,
                               const int64_t q_strides[3], const int64_t kv_strides[3],
                               float scale, int kv_begin, int kv_end, int causal,
                               const void *o_acc, dit_dtype acc_dtype, const int64_t acc_strides[3],
                               const float *lse_acc,
                               void *o, dit_dtype o_dtype, const int64_t o_strides[3], float *lse,
                               struct CUstream_st *stream);

/*
 * dit_attn_merge_lse -- merge C partial attention results over disjoint key blocks.
 *
 * Defined by: "feat: support Ascend NPU backend (torch_npu) for Qwen-Image
 * pipelines - #274", item 2 (the ring loop must combine block outputs with
 * update_out_and_lse; its default gather path avoids the precision loss of
 * merging bf16-rounded block outputs) and "NPU Wan2.2-I2V model inference
 * optimisation practice", section "Ring Attention Overlap" (two attention
 * outputs combined by log-sum-exp).
 *
 * For every (b, h, i):
 *   L   = m + ln sum_c exp(L_c - m),  m = max_c L_c
 *   O   = sum_c exp(L_c - L) O_c      (fp32 accumulation)
 * Blocks with L_c = -inf carry no weight; when every L_c is -inf, O = 0 and
 * L = -inf.
 *
 *   o_parts        [C, B, Sq, H, D] of in_dtype; part c starts at
 *                  o_parts + c * part_stride_o elements and is contiguous BSHD
 *   lse_parts      fp32 [C, B, H, Sq]; part c at lse_parts + c * part_stride_lse
 *   o              [B, Sq, H, D] of out_dtype, contiguous
 *   lse            fp32 [B, H, Sq], contiguous
 * C >= 1.  o must not overlap o_parts; lse must not overlap lse_parts.
 * o_parts, o and part_stride_o * element size 16-byte aligned; LSE pointers
 * 4-byte aligned.
 */
dit_status dit_attn_merge_lse(const void *o_parts, dit_dtype in_dtype, const float *lse_parts,
                              int C, int B, int H, int Sq, int D,
                              int64_t part_stride_o, int64_t part_stride_lse,
                              void *o, dit_dtype out_dtype, float *lse, struct CUstream_st *stream);

/*
 * dit_layer_norm_modulate -- LayerNorm over C with adaLN modulation, per token.
 *
 * Defined by: "NPU Wan2.2-I2V model inference optimisation practice", section
 * "NPU layer_norm_eval operator adaptation" (WanLayerNorm, eps 1e-6, no affine
 * parameters; FusedLayerNormModulate folds the modulation into one layer-norm
 * call with weight 1 + scale and bias shift).
 *
 * For every row x of C channels of sample b:
 *   y = (x - mean(x)) / sqrt(var(x) + eps) * (1 + scale[b]) + shift[b]
 * with the biased variance; fp32 arithmetic, one bf16 rounding.
 *
 *   x, y           bf16 [B, L, C], contiguous, 16-byte aligned; y may equal x
 *   scale, shift   fp32 [B, C] (one modulation vector per sample), 16-byte aligned, or NULL for 0
 *   C              a multiple of 8, at most 8192 (else DIT_ERR_UNSUPPORTED)
 */
dit_status dit_layer_norm_modulate(const void *x, const float *scale, const float *shift, void *y,
                                   int B, int L, int C, float eps, struct CUstream_st *stream);

/*
 * dit_rms_norm -- RMSNorm over all C channels of each row: y = x * w / sqrt(mean(x^2) + eps).
 *
 * Defined by: "NPU Wan2.2-I2V model inference optimisation practice", section
 * "NPU rms_norm operator adaptation" (WanRMSNorm on x of shape [B, L, C]) and
 * "Cosmos Ascend NPU multi-card parallel optimisation notes", section 3.2.
 * The QK prologue (dit_qk_norm_rope) normalises each head over D; this is the
 * whole-token variant.
 *
 *   x, y   bf16 [rows, C], contiguous, 16-byte aligned; y may equal x
 *   w      fp32 [C], 16-byte aligned
 *   C      a multiple of 8, at most 8192
 */
dit_status dit_rms_norm(const void *x, const float *w, void *y, int64_t rows, int C, float eps,
                        struct CUstream_st *stream);

/*
 * dit_quant_fp8_rows -- per-token dynamic quantisation to fp8 e4m3.
 *
 * Defined by: "feat: support Ascend NPU backend (torch_npu) for Qwen-Image
 * pipelines - #274", item 4 (npu_quant_linear: activations quantised per token
 * with a dynamic scale before the quantised matmul).
 *
 * For every row x of K values: scale = max |x| / 448 (1 for an all-zero row),
 * code = e4m3(x / scale), rounded to nearest even and saturated to +-448; the
 * scale and the quotient are fp32.  e4m3 is the OCP 8-bit format with 4
 * exponent bits (bias 7), 3 mantissa bits and no infinities.
 *
 *   x       bf16 [M, K], contiguous, 16-byte aligned
 *   codes   uint8 [M, K] e4m3 codes, contiguous, 16-byte aligned
 *   scale   fp32 [M]
 *   K       a multiple of 16, at most 8192
 */
dit_status dit_quant_fp8_rows(const void *x, void *codes, float *scale, int64_t M, int K, struct CUstream_st *stream);

/*
 * dit_gemm_fp8 -- scaled fp8 GEMM: out[m, n] = a_scale[m] * b_scale[n] * sum_k A[m, k] B[n, k].
 *
 * Defined by: the same PR, item 4 (npu_quant_matmul of per-token quantised
 * activations with per-output-channel quantised weights, output bf16).  A
 * holds activation codes (row m = token), B weight codes (row n = output
 * channel); both are e4m3, row-major with K contiguous; accumulation in fp32
 * on the tensor cores.
 *
 *   a, b          uint8 [M, K] / [N, K] with row strides lda / ldb (bytes, multiples of 16)
 *   a_scale       fp32 [M];  b_scale fp32 [N]
 *   out           bf16 [M, N] with row stride ldo (elements, multiple of 8)
 *   K             a positive multiple of 16
 */
dit_status dit_gemm_fp8(const void *a, const float *a_scale, const void *b, const float *b_scale, void *out,
                        int M, int N, int K, int64_t lda, int64_t ldb, int64_t ldo, struct CUstream_st *stream);

/*
 * dit_attention_host -- the whole hot path (prologue, attention over `chunks`
 * equal KV chunks, LSE merge) on inputs in host memory, results back in host
 * memory, with the copies pipelined against the kernels.
 *
 * Chunk c covers keys [c*S/chunks, (c+1)*S/chunks).  The copies run on two
 * streams the call creates (inputs, outputs) and releases once their work is
 * done; the kernels run on `stream`.
 *   merge_update = 1 (and chunks > 1): q and k (with the prologue also wq, wk,
 *     cos_tab, sin_tab) are copied in, then the value rows of each chunk in
 *     turn (without the prologue each chunk's key rows travel with its value
 *     rows); dit_qk_norm_rope runs in place, dit_attn_fwd over chunk 0 into a
 *     running result of partial_dtype, and dit_attn_fwd_update over every
 *     later chunk, each waiting only for its own rows; O and LSE are copied
 *     back at the end.
 *   merge_update = 0, or chunks == 1: the query rows are processed in up to 8
 *     ranges whose edges are multiples of 256 rows (fewer ranges when a range
 *     would hold fewer than 608 query tiles of 256 rows over all (b, h)); when
 *     even a sixteenth of the rows makes 608 tiles, six ranges of 3/8, 1/4,
 *     1/8, 1/8, 1/16 and 1/16 of the rows (the first range's attention then
 *     covers the copy of every chunk's keys and values, the last range's
 *     output copy is short).  Per
 *     range: dit_attn_fwd over every chunk into stacked partials of
 *     partial_dtype, dit_attn_merge_lse (chunks > 1), and the range's O and
 *     LSE copied back while the next range computes.  Without the prologue the
 *     inputs arrive as: the first range's query rows, each chunk's key and
 *     value rows, the other ranges' query rows; with it, q and k in full first.
 * Results are bit-identical to dit_attention with the same chunks,
 * merge_update and partial_dtype on device copies of the inputs.
 *
 * Defined by: the entry points it composes (see each); the chunk-by-chunk
 * combination is the ring step of "feat: support Ascend NPU backend (torch_npu)
 * for Qwen-Image pipelines - #274", item 2, the stacked merge the LSE merge of
 * its sequence-parallel paths.
 *
 *   q, k, v          host bf16 [B, S, H, D], contiguous (pinned memory lets the
 *                    copies run asynchronously); must stay valid until `stream`
 *                    has passed this call
 *   wq, wk           host fp32 [D]; cos_tab, sin_tab host fp32 [S, D/2]
 *                    (ignored, may be NULL, when prologue == 0)
 *   eps, scale       as for dit_qk_norm_rope / dit_attn_fwd
 *   chunks           1 <= chunks <= S
 *   prologue         1: QK-RMSNorm + RoPE first; 0: attention on q, k as given
 *   partial_dtype    dtype of the running result / stacked partials
 *   merge_update     1: running result merged in each later chunk's epilogue;
 *                    0: stacked partials and the merge kernel, per query range
 *   o, o_dtype       host [B, S, H, D] output; lse host fp32 [B, H, S]
 *   workspace        device memory of at least dit_attention_host_workspace(...)
 *                    bytes, 256-byte aligned, owned by the caller; it must not be
 *                    used by other work until `stream` has passed this call
 * Asynchronous on `stream`: o and lse are valid once `stream` has completed the
 * call.  Errors as for the composed entry points; a workspace that is too small
 * or misaligned is DIT_ERR_INVALID_ARG; a chunk count the merge kernel cannot
 * take (merge_update = 0) is DIT_ERR_UNSUPPORTED before anything is queued.
 */
size_t dit_attention_host_workspace(int B, int S, int H, int D, int chunks, int prologue,
                                    dit_dtype partial_dtype, int merge_update, dit_dtype o_dtype);
dit_status dit_attention_host(const void *q, const void *k, const void *v,
                              const float *wq, const float *wk, const float *cos_tab, const float *sin_tab,
                              int B, int S, int H, int D, float eps, float scale, int chunks, int prologue,
                              dit_dtype partial_dtype, int merge_update, void *o, dit_dtype o_dtype, float *lse,
                              void *workspace, size_t workspace_bytes, struct CUstream_st *stream);

/*
 * dit_attention -- the whole hot path (prologue, attention over `chunks` equal
 * KV chunks, LSE merge) on device buffers, in one call.
 *
 * Runs dit_qk_norm_rope (into the workspace), then the attention over chunk c
 * = keys [c*S/chunks, (c+1)*S/chunks) for every c, then the merge: with
 * merge_update = 1, dit_attn_fwd over chunk 0 into a running result of
 * partial_dtype and dit_attn_fwd_update over every later chunk (the last one
 * writing o); with merge_update = 0, dit_attn_fwd of every chunk into stacked
 * partials of partial_dtype and dit_attn_merge_lse.  chunks == 1 writes o and
 * lse directly.  Same operations and bit-identical results as calling those
 * entry points in that order.  Chunks after the first are launched so that
 * they start beside the previous chunk's last wave and wait for it only where
 * they read its results (update form) or before they end (stacked partials);
 * launches still complete in stream order.
 *
 * Defined by: the entry points it composes; the chunk-by-chunk combination is
 * the ring step of "feat: support Ascend NPU backend (torch_npu) for Qwen-Image
 * pipelines - #274", item 2, and the stacked merge the LSE merge of its
 * sequence-parallel paths.
 *
 *   q, k, v          device bf16 [B, S, H, D], contiguous; not modified
 *   wq, wk           device fp32 [D]; cos_tab, sin_tab device fp32 [S, D/2]
 *                    (ignored, may be NULL, when prologue == 0)
 *   eps, scale       as for dit_qk_norm_rope / dit_attn_fwd
 *   chunks           1 <= chunks <= S; merge_update 0 or 1 (ignored for 1 chunk)
 *   partial_dtype    dtype of the running result / stacked partials
 *   o, o_dtype       device [B, S, H, D] output, contiguous; lse device fp32
 *                    [B, H, S]
 *   workspace        device memory of at least dit_attention_workspace(...)
 *                    bytes, 256-byte aligned, owned by the caller and not
 *                    overlapping any argument; it must not be used by other
 *                    work until `stream` has passed this call (may be NULL when
 *                    that size is 0)
 *   attn_begin, attn_end  events recorded on `stream` before the first and
 *                    after the last attention launch (for timing the attention
 *                    alone); either may be NULL
 * Errors as for the composed entry points; a workspace that is too small,
 * misaligned or overlapping is DIT_ERR_INVALID_ARG.
 */
size_t dit_attention_workspace(int B, int S, int H, int D, int chunks, int prologue, dit_dtype partial_dtype,
                               int merge_update);
dit_status dit_attention(const void *q, const void *k, const void *v,
                         const float *wq, const float *wk, const float *cos_tab, const float *sin_tab,
                         int B, int S, int H, int D, float eps, float scale, int chunks, int prologue,
                         dit_dtype partial_dtype, int merge_update, void *o, dit_dtype o_dtype, float *lse,
                         void *workspace, size_t workspace_bytes, struct CUevent_st *attn_begin,
                         struct CUevent_st *attn_end, struct CUstream_st *stream);

/*
 * dit_attention_ring_overlap -- the ring-attention overlap of one rank, on one GPU.
 *
 * Defined by: "NPU Wan2.2-I2V model inference optimisation practice", section
 * "Ring Attention Overlap" (the attention over the local KV shard overlaps the
 * gathering of the other ranks' shards; one more attention over the gathered
 * keys, combined with the first by their LSEs), and "feat: support Ascend NPU
 * backend (torch_npu) for Qwen-Image pipelines - #274", item 2
 * (update_out_and_lse).
 *
 * Computes the attention of q over the keys local ++ remote_0 ++ ... ++
 * remote_{R-1} (non-causal, as dit_attn_fwd over their concatenation) as:
 *   - the R remote shards copied device-to-device into one contiguous
 *     [B, sum(s_remote), H, D] buffer of the workspace, on a stream the call
 *     creates (it waits for the caller's earlier work on `stream` first; on
 *     one GPU these copies stand in for the all-gather);
 *   - meanwhile, on `stream`, the attention over the local shard into a
 *     running result (partial_dtype O in the workspace, LSE in `lse`);
 *   - then, once the gather is done, the attention over the gathered keys
 *     LSE-merged into that result in its epilogue (dit_attn_fwd_update's
 *     kernel), writing o and lse.
 * The call is complete on `stream` when it returns (the side stream is
 * released by the runtime when its copies finish).  Results are bit-identical
 * to dit_attn_fwd over the local shard followed by dit_attn_fwd_update over
 * the concatenated remote shards.  R = 0 is plain attention over the local
 * shard (no workspace needed).
 *
 *   q              bf16 [B, S, H, D], contiguous
 *   k_local, v_local  bf16 [B, s_local, H, D], contiguous; s_local >= 1
 *   k_remote, v_remote  HOST arrays of R device pointers; shard r is bf16
 *                  [B, s_remote[r], H, D], contiguous, 16-byte aligned; s_remote[r] >= 1
 *   partial_dtype  dtype of the local running O in the workspace (DIT_F32 recommended)
 *   o, lse         outputs as for dit_attn_fwd (contiguous), not overlapping any input
 *   workspace      >= dit_attention_ring_overlap_workspace(B, S, H, D, sum(s_remote),
 *                  partial_dtype) bytes, 256-byte aligned, not overlapping any argument
 * Argument errors return before anything is queued.
 */
size_t dit_attention_ring_overlap_workspace(int B, int S, int H, int D, int s_remote, dit_dtype partial_dtype);
dit_status dit_attention_ring_overlap(const void *q, const void *k_local, const void *v_local, int s_local,
                                      const void *const *k_remote, const void *const *v_remote,
                                      const int *s_remote, int R, int B, int S, int H, int D, float scale,
                                      dit_dtype partial_dtype, void *o, dit_dtype o_dtype, float *lse,
                                      void *workspace, size_t workspace_bytes, struct CUstream_st *stream);

/*
 * dit_attention_noalloc -- dit_attention for callers that cannot allocate
 * device memory: the same prologue, chunked attention and merge, with the
 * workspace taken from a scratch array built into the library instead of one
 * the caller provides.  For code that may not or cannot call cudaMalloc: a
 * host callback, a plugin that a host framework hands only its input and
 * output buffers, a process whose device memory budget belongs to someone
 * else.
 *
 * The pages have no counterpart: this is a deployment convenience of this
 * library, not part of the method.
 *
 *   arguments        as for dit_attention, without workspace and events
 *   limit            the scratch holds 32 MiB: sizes whose
 *                    dit_attention_workspace(...) is larger are refused with
 *                    DIT_ERR_UNSUPPORTED before anything is launched
 * Residency: with the CUDA runtime's default lazy module loading, the first
 * call on a device brings the 32 MiB scratch onto that device, and it stays
 * reserved until the process exits; with CUDA_MODULE_LOADING=EAGER the scratch
 * is reserved on every device where the process creates a context, as soon as
 * the library is loaded, even if this entry point is never called.  Every call
 * looks the scratch's device address up afresh (cudaGetSymbolAddress with the
 * call's device current), so a context rebuilt after cudaDeviceReset gets the
 * right address.  The first call on a device may load the library's module
 * there: make it before any stream capture.  All calls share the scratch:
 * nothing in it needs to start at zero, but calls that run concurrently on
 * the GPU (other streams, other host threads) race on it.  Allocates nothing.
 * Errors as for dit_attention.
 */
dit_status dit_attention_noalloc(const void *q, const void *k, const void *v,
                                 const float *wq, const float *wk, const float *cos_tab, const float *sin_tab,
                                 int B, int S, int H, int D, float eps, float scale, int chunks, int prologue,
                                 dit_dtype partial_dtype, int merge_update, void *o, dit_dtype o_dtype, float *lse,
                                 struct CUstream_st *stream);

/*
 * dit_poll_device_error -- synchronise `stream`, then read and clear the
 * library's device error word.  Returns DIT_OK, DIT_ERR_TIMEOUT if a bounded
 * device-side wait gave up since the last poll, or DIT_ERR_CUDA if the
 * synchronisation itself failed.
 */
dit_status dit_poll_device_error(struct CUstream_st *stream);

/*
 * dit_selftest_wait_timeout -- failure-detection self-test.  Launches one thread
 * that waits, with the same bounded wait every kernel here uses, on a device
 * barrier that nothing ever completes; the wait gives up after about 2 s and
 * records the timeout.  A following dit_poll_device_error must then return
 * DIT_ERR_TIMEOUT, with the CUDA context still usable.  Not part of the
 * attention path (the pages have no counterpart); it exercises the error
 * route that a stalled pipeline would take.
 */
dit_status dit_selftest_wait_timeout(struct CUstream_st *stream);

/*
 * dit_selftest_fp8_quotients -- exhaustive check of the division inside
 * dit_quant_fp8_rows.  The quantiser forms x / scale_m by Markstein's division
 * (a correctly rounded reciprocal per row, then a product, its exact FMA
 * residual and one correction per element) instead of an IEEE division per
 * element.  This call evaluates that division and IEEE division side by side
 * for every positive finite bf16 row maximum and every bf16 element whose
 * magnitude does not exceed it (the scale being RN(max / 448) as in the
 * quantiser; rows whose scale is below 2^-100 use IEEE division there and are
 * not counted), about 2.1e9 pairs, and writes to the HOST array counts:
 *   counts[0]  pairs whose fp32 quotients differ (informational: the quotient
 *              is not an output; about 2.05e6)
 *   counts[1]  pairs whose e4m3 codes differ -- the quantiser's output; 0
 *              means its codes equal those of IEEE division on every input
 * Synchronous: returns after the counts are read back.
 */
dit_status dit_selftest_fp8_quotients(uint64_t counts[2], struct CUstream_st *stream);

/*
 * dit_set_launch_overlap -- enable (1, the default) or disable (0) programmatic
 * dependent launch for every kernel this library launches afterwards.  When
 * enabled, a kernel may be scheduled while the previous kernel on its stream is
 * still finishing; each kernel waits for that kernel's completion and memory
 * (griddepcontrol.wait) before its first global-memory access, so results are
 * the same either way and only the launch gap shrinks.  Process-wide setting.
 * Returns DIT_ERR_INVALID_ARG for any other value.
 */
dit_status dit_set_launch_overlap(int enable);

/* dit_status_string -- static, human-readable name of a status code (never NULL). */
const char *dit_status_string(dit_status s);

/* dit_last_error_detail -- static text describing the most recent argument or CUDA error
 * on the calling thread ("" if none). */
const char *dit_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* DITATTN_H */
