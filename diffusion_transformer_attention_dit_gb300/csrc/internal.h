// Internal launchers shared by the C-ABI translation unit and the kernel
// translation units.  Arguments are validated by the caller (api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ditattn.h"

namespace ditattn {

// Whether launches carry programmatic stream serialisation (each kernel calls
// griddepcontrol.wait before touching global memory, so its launch and
// preamble overlap the previous kernel's tail).  Set by dit_set_launch_overlap.
bool launch_overlap_enabled();

// Set the text dit_last_error_detail returns (for entry points outside api.cu).
void set_error_detail(const char *why);

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_overlap_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Attention forward over keys [kv_begin, kv_end) (causal: query i sees keys j <= i).
// Strides in elements {b, s, h}.  With o_acc non-null (update form) the result is
// LSE-merged with the running (o_acc, lse_acc) before it is written.  defer_wait:
// the previous launch on the stream is the previous chunk of the same attention
// (it writes only what this launch reads as o_acc / lse_acc, or nothing this
// launch touches), so the dependency wait moves to where its results are needed.
cudaError_t launch_attn_fwd(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                            const int64_t q_st[3], const int64_t kv_st[3], float scale, int kv_begin, int kv_end,
                            bool causal, void *o, bool o_f32, const int64_t o_st[3], float *lse, const void *o_acc,
                            bool acc_f32, const int64_t acc_st[3], const float *lse_acc, bool defer_wait,
                            cudaStream_t stream, const char **detail);

cudaError_t launch_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out, const float *wq,
                                const float *wk, const float *cos_tab, const float *sin_tab, int B, int S, int H,
                                int D, float eps, cudaStream_t stream);

cudaError_t launch_merge_lse(const void *o_parts, bool in_f32, const float *lse_parts, int C, int B, int H, int Sq,
                             int D, int64_t part_stride_o, int64_t part_stride_lse, void *o, bool out_f32,
                             float *lse, cudaStream_t stream);

// Row normalisations (row_kernels.cu): LayerNorm + adaLN modulation, RMSNorm over C.
// C % 8 == 0, C <= row_norm_max_channels().
int row_norm_max_channels();
cudaError_t launch_layer_norm_modulate(const void *x, const float *scale, const float *shift, void *y, int B, int L,
                                       int C, float eps, cudaStream_t stream);
cudaError_t launch_rms_norm(const void *x, const float *w, void *y, long long rows, int C, float eps,
                            cudaStream_t stream);

// W8A8 fp8 (fp8.cu): per-row dynamic quantisation (K % 8 == 0, K <= quant_fp8_max_k()) and the scaled GEMM.
int quant_fp8_max_k();
cudaError_t launch_quant_fp8_rows(const void *x, void *codes, float *scale, long long M, int K, cudaStream_t stream);
cudaError_t launch_gemm_fp8(const void *a, const float *a_scale, const void *b, const float *b_scale, void *out,
                            int M, int N, int K, long long lda, long long ldb, long long ldo, cudaStream_t stream,
                            const char **detail);
cudaError_t read_and_clear_fp8_error(unsigned int *value);
// Exhaustive check of the quantiser's division against IEEE division (synchronous on `stream`):
// counts[0] fp32 quotients, counts[1] e4m3 codes that differ.
cudaError_t run_fp8_quotient_selftest(unsigned long long counts[2], cudaStream_t stream);

// Largest C the merge kernel accepts, and whether C * H weights fit its shared-memory budget.
int merge_max_parts();
bool merge_fits(int C, int H);

// One-thread kernel whose bounded wait on a never-completed mbarrier must give up.
cudaError_t launch_wait_timeout_selftest(cudaStream_t stream);

// Read and clear the device words in which each kernel's bounded waits record that they gave up.
cudaError_t read_and_clear_attn_error(unsigned int *value);
cudaError_t read_and_clear_prologue_error(unsigned int *value);
cudaError_t read_and_clear_merge_error(unsigned int *value);

// The attention entry points' argument checks, then launch_attn_fwd (api.cu).
// o_acc == nullptr: plain form; otherwise the update form.
// sequence_chunk: the position of this launch in a sequence of attention chunk
// launches that the caller issues back to back on `stream` (-1: not part of
// one).  Only sequence_chunk >= 1 defers the dependency wait, and it is valid
// only when the launch right before it on the stream is chunk sequence_chunk - 1
// of the same sequence -- chunk 0 always waits for its predecessor (say a
// prologue or a merge) at its start, and every deferred chunk waits for its
// predecessor before it ends, so each chunk's start is ordered after whatever
// preceded chunk 0.
dit_status attn_checked(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                        const int64_t q_strides[3], const int64_t kv_strides[3], float scale, int kv_begin, int kv_end,
                        bool causal, void *o, dit_dtype o_dtype, const int64_t o_strides[3], float *lse,
                        const void *o_acc, dit_dtype acc_dtype, const int64_t acc_strides[3], const float *lse_acc,
                        int sequence_chunk, cudaStream_t stream);

// Attention over `chunks` equal KV chunks of contiguous bf16 BSHD q, k, v
// (chunk c = keys [c*S/chunks, (c+1)*S/chunks)) and their merge, on `stream`
// (attention_path.cu).  merge_update: chunk 0 writes the running result `acc`
// (partial_dtype, BSHD), every later chunk is merged into it in its epilogue
// (dit_attn_fwd_update), the last one straight into o.  Otherwise chunk c
// writes part c of the stacked `acc` [chunks, B, S, H, D] and lse_parts
// [chunks, B, H, S], and dit_attn_merge_lse combines them.  chunks == 1 writes
// o and lse directly.  Chunks after the first defer their dependency wait.
// attn_begin / attn_end (may be null) are recorded before the first and after
// the last attention launch.  before_chunk (may be null) runs on the host
// before chunk c is launched (the host path makes the stream wait there for
// that chunk's value rows).
dit_status run_attention_chunks(const void *q, const void *k, const void *v, int B, int S, int H, int D, float scale,
                                int chunks, dit_dtype partial_dtype, bool merge_update, void *acc, float *lse_parts,
                                void *o, dit_dtype o_dtype, float *lse, cudaEvent_t attn_begin, cudaEvent_t attn_end,
                                cudaError_t (*before_chunk)(void *ctx, int c), void *ctx, cudaStream_t stream);

}  // namespace ditattn
