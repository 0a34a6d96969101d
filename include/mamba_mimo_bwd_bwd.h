/*
 * mamba_mimo_bwd_bwd.h -- C ABI of the second backward stage of the Mamba-3
 * MIMO chunked state-space scan (GB300, sm_103a): the reverse scan over
 * chunks and its 12 gradients.
 *
 * The operation is the one on the page "MindSpeed-Ops PR #100":
 *   - argument order, the input and output tables, the layout of DQ / DK as
 *     [B, S*R, H, N], the output dtypes and the reverse-scan formulas for
 *     dPhiO and PsiV: the op document "mamba3_mimo_bwd_bwd 算子迁移说明";
 *   - the meaning of the caches `states` (the state entering each chunk) and
 *     `qk_dot` (the same-token R x R q.k block of the diagonal term), the
 *     state and dstates recurrences, and the padding and cropping of a
 *     partial last chunk: the practice document "mamba3_mimo_bwd_bwd
 *     Triton-Ascend 实践", sections "输入缓存的语义", "反向语义拆解" and
 *     "非整 chunk".
 * The pages name the 12 outputs without formulas; each is the exact
 * derivative of L = sum dPhiO * out, out being the first stage's chunk output
 * (page "feat: add Triton-Ascend implementation of Mamba-3 mamba_mimo_bwd_fwd
 * #125", FP32 reference, no rounding points), with these readings:
 *   gamma = dt * sigmoid(trap), factor = gamma + dt[t+1] * sigmoid(-trap[t+1])
 *   (0 at the last padded position); DGAMMA / DFACTOR are the gradients with
 *   respect to them.  DDA_CS is the gradient through exp(da_cs[t]) on the
 *   inter term, DDA the one through the chunk decay exp(da_cs[last valid
 *   token]) reported at that token (0 elsewhere); DDA + DDA_CS is the whole
 *   da_cs gradient.  DSSDA sums the R x R rank pairs of each token pair.
 *
 * Symbols as in mamba_mimo_bwd_fwd.h: B, S, H, G (H % G == 0, head h reads
 * group h / (H / G)), R, N, P, C = chunk_size, nchunks = ceil(S / C),
 * RD = N / rotary_dim_divisor.
 *
 * Memory.  Every tensor pointer is a DEVICE pointer to a dense row-major
 * tensor; the caller owns all memory (inputs, outputs, workspace); each call
 * only enqueues kernels on `stream`.
 *
 * dtype codes (act_dtype, dqkv_dtype): 0 fp32, 1 bf16, 2 fp16.  The op page
 * supports float16, bfloat16 and float32 activations; here one code,
 * act_dtype, gives the dtype of all seven activation-like inputs (marked
 * "act" below: those that are BF16 in the first stage, and its two caches).
 *
 *   input       shape                                   dtype
 *   dout        reduce-O: [B,S,H,P]; per rank: [B,S,R,H,P]  act
 *   q, k        [B,S,R,G,N]                             act
 *   v           [B,S,H,P]                               act
 *   q_bias, k_bias [H,R,N]                              fp32
 *   mimo_v      [H,R,P]                                 fp32
 *   states      [B,H,nchunks,N,P]                       act    (first stage's output)
 *   qk_dot      [B,H,S,R,R]                             act    (first stage's output)
 *   da_cs, da_cs_rev, dt  [B,H,S]                       fp32
 *   trap        [B,H,S]                                 act
 *   segsum      [B,H,nchunks,C,C]                       fp32
 *   angles      [B,S,H,RD]                              fp32
 *   mimo_o      [H,R,P] or NULL                         fp32   (NULL: dout per rank)
 *   d           [H] or NULL                             fp32
 *
 *   output (fp32; DQ, DK, DV in the dtype `dqkv_dtype` selects: the pages'
 *   output_dtype, whose default is the inputs' dtype)
 *   DQ, DK      [B,S*R,H,N]   per head (sum over a group's heads for q / k)
 *   DV          [B,S,H,P]
 *   DMIMO_V     [B,H,R,P]     per batch (sum over B for mimo_v)
 *   DANGLES     [B,S,H,RD]
 *   DFACTOR, DGAMMA, DDA, DDA_CS_REV, DDA_CS  [B,H,S]
 *   DSSDA       [B,H,nchunks,C,C]   0 on and above the diagonal and past S
 *   DD          [B,H] or NULL (NULL iff d is NULL), per batch
 *
 * Alignment: every pointer 4-byte aligned, the workspace 256-byte aligned.
 * Outputs must not overlap inputs or each other.
 *
 * Envelope (checked): the pages' constraints (B..P >= 1, H % G == 0, N even,
 * rotary_dim_divisor in {2, 4}, N % rotary_dim_divisor == 0) and this
 * build's: N <= 256, P <= 128, C*R <= 128, R <= 16 (MMBF_ERR_UNSUPPORTED
 * otherwise).  Shapes with N, P and C*R all <= 64 run the gradient kernel
 * with its tiles in shared memory, one chunk per CTA; larger ones run a
 * persistent kernel (152 CTAs) whose tiles sit in a per-CTA part of the
 * workspace, which the size query then includes.
 *
 * Numerics: every input is widened to FP32 exactly; FP32 throughout (sums,
 * the reverse scan); BF16 / FP16 outputs are the FP32 results rounded to
 * nearest even.  The tile products run on the tensor cores in TF32: each
 * FP32 operand is split into two TF32 parts by truncation and each pair
 * takes three products (two where one operand is the BF16 / FP16 states
 * cache, exact in TF32), an error below 3 * 2^-20 relative per product
 * (FP32-level accuracy).  Results are deterministic (no floating-point
 * atomics).
 */
#ifndef MAMBA_MIMO_BWD_BWD_H
#define MAMBA_MIMO_BWD_BWD_H

#include "mamba_mimo_bwd_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace mamba_mimo_bwd_bwd needs (the per-chunk dstates
 * and the per-chunk partial sums of DMIMO_V and DD).  Returns MMBF_OK and
 * writes *bytes, or the validation error the call would return. */
mmbf_status mamba_mimo_bwd_bwd_workspace_size(const mmbf_dims* dims, int64_t chunk_size,
                                              int64_t rotary_dim_divisor, size_t* bytes);

/* Enqueue the second backward stage on `stream` (a cudaStream_t; NULL for
 * the legacy default stream).  Inputs in the pages' positional order (dout
 * ... angles, mimo_o, d), then chunk_size, rotary_dim_divisor, act_dtype
 * (the activations' dtype code) and dqkv_dtype (the dtype code of DQ, DK,
 * DV; MMBF_ERR_ARG for a code outside 0..2), then the 12 outputs in the
 * pages' order, then the workspace.  Validation failures
 * enqueue nothing and return an error (message in mamba_mimo_last_error);
 * MMBF_ERR_CUDA reports a launch error.  Asynchronous; calls sharing a
 * workspace must be ordered on one stream.  Four kernels: the per-chunk
 * dstates seeds, the reverse scan, the per-chunk gradients, the per-(b,h)
 * sums of DMIMO_V and DD (mamba_mimo_last_launch_count reports them;
 * mamba_mimo_stage_name names them "bb_seed", "bb_scan", "bb_grad",
 * "bb_reduce", and mamba_mimo_set_stage_events times them). */
mmbf_status mamba_mimo_bwd_bwd(const mmbf_dims* dims, const void* dout, const void* q, const void* k,
                               const void* v, const float* q_bias, const float* k_bias,
                               const float* mimo_v, const void* states, const void* qk_dot,
                               const float* da_cs, const float* da_cs_rev, const float* dt,
                               const void* trap, const float* segsum, const float* angles,
                               const float* mimo_o, const float* d, int64_t chunk_size,
                               int64_t rotary_dim_divisor, int act_dtype, int dqkv_dtype, void* DQ, void* DK,
                               void* DV, float* DMIMO_V, float* DANGLES, float* DFACTOR, float* DGAMMA,
                               float* DDA, float* DSSDA, float* DDA_CS_REV, float* DDA_CS, float* DD,
                               void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_MIMO_BWD_BWD_H */
