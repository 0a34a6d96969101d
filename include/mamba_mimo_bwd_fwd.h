/*
 * mamba_mimo_bwd_fwd.h -- C ABI of the GB300 (sm_103a) implementation of the
 * first backward stage of the Mamba-3 MIMO chunked state-space scan.
 *
 * The operation is the one defined on the page "feat: add Triton-Ascend
 * implementation of Mamba-3 mamba_mimo_bwd_fwd #125" (MindSpeed-Ops):
 *   - argument list and optional branches: docs/triton/mamba_mimo_bwd_fwd.md,
 *     sections "使用方法" (usage) and "输入与输出" (input/output tables and
 *     constraints);
 *   - arithmetic and BF16 rounding boundaries: the BF16 PyTorch reference
 *     tests/unit_tests/triton/mamba_mimo_bwd_fwd_bf16_reference.py;
 *   - validation errors: mindspeed_ops/api/triton/mamba_mimo_bwd_fwd.py,
 *     function _validate_inputs;
 *   - meaning of `states` (state entering each chunk) and `qk_dot`
 *     (same-token R x R q.k): page "MindSpeed-Ops PR #100", section
 *     "输入缓存的语义".
 *
 * Symbols (the pages' notation): B batch, S sequence length, H value heads,
 * G query/key groups (H % G == 0; head h reads group h / (H / G)), R MIMO
 * rank, N state dimension, P value dimension, C = chunk_size,
 * nchunks = ceil(S / C).
 *
 * Memory.  Every tensor pointer is a DEVICE pointer to a dense, row-major
 * (contiguous) tensor in the layout below.  The caller owns all memory:
 * inputs, outputs and the workspace.  The library never allocates, frees or
 * synchronises; each call only enqueues kernels on `stream`.
 *
 *   input       shape                                 dtype
 *   dout        reduced: [B,S,H,P]; per-rank: [B,S,R,H,P]  bf16
 *   q, k        [B,S,R,G,N]                           bf16
 *   v           [B,S,H,P]                             bf16
 *   q_bias, k_bias [H,R,N]                            fp32
 *   mimo_v      [H,R,P]                               fp32
 *   mimo_o      [H,R,P] or NULL                       fp32   (NULL: dout is per-rank)
 *   z           [B,S,H,P] or NULL                     bf16
 *   mimo_z      [H,R,P] or NULL (NULL iff z is NULL)  fp32
 *   angles      [B,S,H,N/rotary_dim_divisor]          fp32
 *   da_cs, da_cs_rev, dt  [B,H,S]                     fp32
 *   trap        [B,H,S]                               bf16
 *   d           [H] or NULL                           fp32
 *   segsum      [B,H,nchunks,C,C]                     fp32
 *
 *   output      shape                                 dtype
 *   dmimo_o     [B,H,R,P]   (NULL iff mimo_o NULL)    fp32   per batch, not batch-reduced
 *   states      [B,H,nchunks,N,P]                     bf16   state entering chunk c
 *   dz          [B,S,H,P]   (NULL iff z NULL)         bf16
 *   dmimo_z     [B,H,R,P]   (NULL iff z NULL)         fp32
 *   qk_dot      [B,H,S,R,R]                           bf16   [r_out, r_in]
 *
 * bf16 is IEEE bfloat16 (1-8-7); fp32 is IEEE binary32.  All pointers must be
 * 4-byte aligned; the workspace 256-byte aligned.  Outputs must not overlap
 * inputs or each other.
 *
 * Envelope (checked; the pages' constraints plus this build's own):
 *   B, S, H, G, R, N, P >= 1; H % G == 0; N even; N % rotary_dim_divisor == 0;
 *   rotary_dim_divisor in {2, 4}; N <= 128; P <= 128; 1 <= C*R <= 128;
 *   this build also requires R <= 16 (MMBF_ERR_UNSUPPORTED otherwise).
 *
 * Numerics.  BF16 rounding at the boundaries of the pages' BF16 reference,
 * FP32 everywhere else (FP32 tensor-core accumulation, FP32 recurrent
 * state).  Results are deterministic for a given device and input: no
 * floating-point atomics.
 */
#ifndef MAMBA_MIMO_BWD_FWD_H
#define MAMBA_MIMO_BWD_FWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MAMBA_MIMO_BWD_FWD_ABI_VERSION 1

/* Status codes.  SHAPE/ARG/DTYPE correspond to the pages' ValueError /
 * TypeError cases; UNSUPPORTED to NotImplementedError. */
typedef enum {
  MMBF_OK = 0,
  MMBF_ERR_SHAPE = 1,       /* a dimension is non-positive or violates a constraint */
  MMBF_ERR_ARG = 2,         /* a required pointer is NULL, or optional pointers are
                               inconsistent (z vs mimo_z vs dz/dmimo_z, mimo_o vs dmimo_o) */
  MMBF_ERR_UNSUPPORTED = 3, /* allowed by the pages, outside this build's envelope */
  MMBF_ERR_ALIGN = 4,       /* a pointer is not aligned as required */
  MMBF_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than the size query says */
  MMBF_ERR_CUDA = 6,        /* a CUDA runtime error while enqueuing */
  MMBF_ERR_DEVICE_TIMEOUT = 7 /* a kernel's bounded wait ran out (see mamba_mimo_device_status) */
} mmbf_status;

/* Problem dimensions (see the symbol list above). */
typedef struct {
  int64_t B, S, H, G, R, N, P;
} mmbf_dims;

/* Bytes of device workspace mamba_mimo_bwd_fwd needs for this problem.
 * `reduced_dout` = (mimo_o != NULL), `has_z` = (z != NULL).  Depends only on
 * its arguments.  Returns MMBF_OK and writes *bytes, or the validation error
 * mamba_mimo_bwd_fwd would return for the same shape. */
mmbf_status mamba_mimo_bwd_fwd_workspace_size(const mmbf_dims* dims, int64_t chunk_size,
                                              int64_t rotary_dim_divisor, int reduced_dout,
                                              int has_z, size_t* bytes);

/* Enqueue the first backward stage on `stream` (a cudaStream_t; NULL for the
 * legacy default stream).  Arguments 2-18 follow the pages' positional order
 * (dout ... segsum), then chunk_size and rotary_dim_divisor, then the five
 * outputs in the pages' output order, then the workspace.
 *
 * Branches: mimo_o != NULL selects reduced dout and produces dmimo_o;
 * z != NULL (with mimo_z) produces dz and dmimo_z; d != NULL adds the skip
 * term d[h] * PsiV to the chunk output.
 *
 * On any validation failure nothing is enqueued and an error code is
 * returned; mamba_mimo_last_error() then describes it.  MMBF_ERR_CUDA
 * reports a launch error (the stream may hold part of the work).
 * Asynchronous: outputs are valid once `stream` reaches this point.
 * Calls that share a workspace must be ordered on one stream. */
mmbf_status mamba_mimo_bwd_fwd(const mmbf_dims* dims, const void* dout, const void* q,
                               const void* k, const void* v, const float* q_bias,
                               const float* k_bias, const float* mimo_v, const float* mimo_o,
                               const void* z, const float* mimo_z, const float* angles,
                               const float* da_cs, const float* da_cs_rev, const float* dt,
                               const void* trap, const float* d, const float* segsum,
                               int64_t chunk_size, int64_t rotary_dim_divisor, float* dmimo_o,
                               void* states, void* dz, float* dmimo_z, void* qk_dot,
                               void* workspace, size_t workspace_bytes, void* stream);

/* The same operation, also writing the layer's forward output `y` (BF16, in
 * dout's layout: [B,S,H,P] when mimo_o != NULL, [B,S,R,H,P] otherwise) to the
 * caller-owned, 4-byte aligned buffer `y` (MMBF_ERR_ARG if NULL).  y is the
 * function whose gradients the op returns (op document, gradient formulas of
 * the Z / projection branch): with the chunk output out[t,r,p] (BF16) and the
 * gate g = silu(z[t,p] * mimo_z[r,p]) (g = 1 without z),
 *   y[t,p]   = sum over r in rank order of mimo_o[r,p] * out[t,r,p] * g[t,r,p]
 *   y[t,r,p] = out[t,r,p] * g[t,r,p]                  (without mimo_o)
 * computed in FP32 and rounded to BF16 once.  The pages' op has no y
 * output; every other argument and output is as for mamba_mimo_bwd_fwd
 * (the outputs equal that call's up to FP32 summation order, since the
 * launch plan may differ). */
mmbf_status mamba_mimo_bwd_fwd_y(const mmbf_dims* dims, const void* dout, const void* q,
                                 const void* k, const void* v, const float* q_bias,
                                 const float* k_bias, const float* mimo_v, const float* mimo_o,
                                 const void* z, const float* mimo_z, const float* angles,
                                 const float* da_cs, const float* da_cs_rev, const float* dt,
                                 const void* trap, const float* d, const float* segsum,
                                 int64_t chunk_size, int64_t rotary_dim_divisor, float* dmimo_o,
                                 void* states, void* dz, float* dmimo_z, void* qk_dot, void* y,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of the built-in scratch area used by
 * mamba_mimo_bwd_fwd_fixed_scratch (one area per GPU, held until exit). */
#define MAMBA_MIMO_FIXED_SCRATCH_BYTES ((size_t)32 << 20)

/* The same operation as mamba_mimo_bwd_fwd, for callers that cannot
 * allocate device memory themselves -- for example code running under a host
 * framework that owns every device allocation through its own pool, or code
 * that must not call cudaMalloc because it can synchronise the device -- and
 * so cannot provide a workspace.  (The pages define no such call; it exists
 * for these callers.)  Arguments are those of mamba_mimo_bwd_fwd without the
 * workspace; inputs and outputs are still the caller's device buffers.
 *
 * The workspace is a built-in device array of MAMBA_MIMO_FIXED_SCRATCH_BYTES
 * bytes on each GPU.  A problem whose workspace (the size query above) is
 * larger is rejected with MMBF_ERR_WORKSPACE and nothing is enqueued.  This
 * call allocates nothing.  Its first call on a device looks up the array's
 * device address on the current device (cudaGetSymbolAddress); make that
 * first call before any stream capture.  The address is kept with the CUDA
 * context it was looked up in; after the device's context is destroyed and
 * created again (cudaDeviceReset) the next call looks it up anew, so make
 * that call before capture too.  Every call on a device shares the
 * one array and leaves its contents behind; nothing in it needs to start at
 * zero.  Calls whose kernels overlap on the GPU (different streams without
 * ordering between them) race on the array and give wrong results: order
 * them on one stream. */
mmbf_status mamba_mimo_bwd_fwd_fixed_scratch(
    const mmbf_dims* dims, const void* dout, const void* q, const void* k, const void* v,
    const float* q_bias, const float* k_bias, const float* mimo_v, const float* mimo_o,
    const void* z, const float* mimo_z, const float* angles, const float* da_cs,
    const float* da_cs_rev, const float* dt, const void* trap, const float* d,
    const float* segsum, int64_t chunk_size, int64_t rotary_dim_divisor, float* dmimo_o,
    void* states, void* dz, float* dmimo_z, void* qk_dot, void* stream);

/* Message of the last failed call on the calling thread ("" if none). */
const char* mamba_mimo_last_error(void);

/* MAMBA_MIMO_BWD_FWD_ABI_VERSION of the loaded library. */
int mamba_mimo_abi_version(void);

/* Number of kernel launches the last successful mamba_mimo_bwd_fwd call on
 * this thread enqueued. */
int mamba_mimo_last_launch_count(void);

/* Optional per-kernel timing (host-side setting of the calling thread).
 * While set, each mamba_mimo_bwd_fwd call on this thread records
 * events[2*i] just before and events[2*i+1] just after its i-th kernel
 * launch, on the call's stream, for every i < count / 2.  `events` holds
 * cudaEvent_t handles (created with timing enabled) cast to void*; the array
 * must stay valid while set.  Pass NULL, 0 to stop.  Kernel i is named by
 * mamba_mimo_stage_name(i). */
void mamba_mimo_set_stage_events(void* const* events, int count);

/* Kernel family the last successful mamba_mimo_bwd_fwd call on this thread
 * used: -1 for the generic kernels (any shape of the envelope); 0, 1, 2 for
 * the shape-specialised families R4 C16 N=P=64, R8 C16 N=P=64 and R4 C16
 * N=P=32; 3 for the warp-specialised tensor-core family (R4 C16 N=P=64 with
 * reduced dout and without y: every chunk contraction on tcgen05.mma); 4 for
 * the shape-specialised wide-state family R4 C32 N=128 P=64 with rotary
 * divisor 2. */
int mamba_mimo_last_kernel_variant(void);

/* Failure detection for the last mamba_mimo_bwd_fwd call on this thread.
 * Every wait inside the kernels (the shared-memory barriers that the TMA
 * input loads complete) is bounded to about a second; when one runs out the
 * kernel records an error word tagged with the call in the first bytes of
 * the call's workspace, lets its copies in flight land, and returns early
 * (its outputs are then incomplete).  This function synchronises `stream`,
 * reads that word, and returns MMBF_OK or MMBF_ERR_DEVICE_TIMEOUT (message
 * in mamba_mimo_last_error).  The workspace must still be valid.  MMBF_OK if
 * no call has been made on this thread. */
mmbf_status mamba_mimo_device_status(void* stream);

/* Test hooks for this thread's later calls (0 = off, the default).  Bit 0:
 * in the kernels that load their inputs by TMA, each CTA's first barrier
 * expects 16 bytes more than its loads deliver, so its bounded wait runs
 * out and the call reports MMBF_ERR_DEVICE_TIMEOUT through
 * mamba_mimo_device_status.  Nothing faults or hangs; outputs of such a
 * call are incomplete.  Bit 1: the warp-specialised family takes its two-
 * kernel form (a separate state-sum kernel) where it would run as a single
 * kernel, so tests cover both forms.  Bit 2: in its single-kernel form the
 * first segment of every (b,h) does not publish its segment sum, so the later
 * segments' bounded look-back runs out and the call reports
 * MMBF_ERR_DEVICE_TIMEOUT (after about a second).  For tests only. */
void mamba_mimo_set_test_hooks(int flags);

/* Test hook: evaluates, on the device, the approximate math the shape-
 * specialised kernels use, so tests can bound its error (the pages have no
 * counterpart: these are this library's own fast paths for the rotary
 * sin/cos, exp(segsum) and the gate sigmoid).  x: n FP32 inputs, out: 4n
 * FP32 results, both device pointers owned by the caller; enqueued on
 * `stream`.  For input i, out[4i] and out[4i+1] are the fast path's values,
 * out[4i+2] and out[4i+3] the same quantities from CUDA's accurate sinf /
 * cosf / expf:
 *   which = 0: sin(x), cos(x) (reduction by 2*pi in two FP32 parts, then the
 *              sin.approx / cos.approx instructions);
 *   which = 1: exp(x) as 2^(x log2 e) by ex2.approx (second slot 0);
 *   which = 2: sigmoid(x) = rcp.approx(ex2.approx(-x log2 e) + 1) (second
 *              slot 0).
 * Returns MMBF_ERR_ARG for a bad `which`, a NULL pointer or n < 0,
 * MMBF_ERR_ALIGN if out is not 16-byte aligned, and MMBF_ERR_CUDA if the
 * launch fails. */
mmbf_status mamba_mimo_probe_fast_math(int which, const float* x, float* out, int n, void* stream);

/* Launch plan of the last successful mamba_mimo_bwd_fwd call on this thread
 * (diagnostic): writes min(n, 7) ints to out -- chunks per segment, segments
 * per (b,h), state units per segment, chunks per unit, the resident
 * output-kernel CTAs the segment length was sized for (0 for the generic
 * kernels), 1 if the call ran as a single kernel (the warp-specialised
 * family computing each segment's state sum itself, all CTAs resident at
 * once), and the CUDA error code with which the device refused that single
 * launch when the call fell back to two kernels (else 0) -- and returns how
 * many it wrote (0 if out is NULL or n < 0).  The
 * plan is a function of the problem alone (shape and branches), so the
 * workspace size query agrees with every call on any device. */
int mamba_mimo_last_plan(int* out, int n);

/* Name of the i-th kernel the last mamba_mimo_bwd_fwd call on this thread
 * launched (0 <= i < 4), or NULL past its last kernel.  The generic kernels
 * are "segment_state", "segment_prefix", "chunk_output", "grad_reduce"; the
 * shape-specialised ones "segment_state", "segment_prefix", "chunk_output"
 * (the gradient sum is folded into the output kernel). */
const char* mamba_mimo_stage_name(int i);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_MIMO_BWD_FWD_H */
