// GB300 (sm_103a) kernels and C ABI for the first backward stage of the
// Mamba-3 MIMO chunked scan (`mamba_mimo_bwd_fwd`).
//
// What is computed is defined on the page "feat: add Triton-Ascend
// implementation of Mamba-3 mamba_mimo_bwd_fwd #125": the op document's
// input/output tables and the BF16-boundary reference
// (tests/unit_tests/triton/mamba_mimo_bwd_fwd_bf16_reference.py).  The
// decomposition below is this library's own:
//
//   segment_state_kernel   grid (p-slice, segment, b*h)
//       For a segment of L consecutive chunks, the chunk-local state
//       contributions U_c = k_state_c^T PsiV_c (BF16 tensor-core GEMM, FP32
//       accumulate) folded as  local = exp(da_cs[last_c]) * local + U_c,
//       plus the segment's total decay.  Inputs: k, k_bias, angles, dt, trap,
//       da_cs, da_cs_rev, v, mimo_v.
//   segment_prefix_kernel  grid (N*P / 256, b*h)
//       Exclusive scan over segments: the FP32 state entering each segment.
//   chunk_output_kernel    grid (p-slice, segment, b*h)
//       Walks its segment's chunks with the FP32 state resident in shared
//       memory.  Per chunk: states[c] = bf16(state); biased Q/K (BF16 add);
//       same-token qk_dot (tensor cores, diagonal tiles only); rotary;
//       trapezoid factors; the strictly causal (C*R)^2 matrix A, inter =
//       Q bf16(state) exp(da_cs), intra = A PsiV (tensor cores); the rank-
//       ordered BF16 diagonal term; out; the Z / projection-gradient branch
//       (dz, and per-thread partial sums of dmimo_o / dmimo_z); then the
//       state update.
//   grad_reduce_kernel     grid (b*h)
//       Fixed-order sum of the per-segment dmimo_o / dmimo_z partials.
//
// Shapes with specialised kernels (mmbf_fast.cuh) run three launches,
// chained by programmatic dependent launch: fast::state_kernel over state
// units of LA chunks (the units of a segment form a thread-block cluster and
// fold their sums into the segment's sum); segment_prefix_fast_kernel, the
// exclusive scan over segments with one state element per thread; and
// fast::output_kernel, whose CTAs read their entering state and whose last
// CTA per (b,h) -- found with an atomic counter -- does the fixed-order
// gradient sum.
//
// The second backward stage (mamba_mimo_bwd_bwd) has its own kernels and
// entry points in mmbb.cuh, included at the end of this file.
//
// Rows of a chunk tile are j = t*R + r (token-major), as in the reference's
// flatten of the token and rank axes.  BF16 products and sums of two BF16
// values use mul.rn.bf16x2 / add.rn.bf16x2: the exact product of two BF16
// values fits FP32, and FP32 (24 bits) >= 2*8+2 bits makes FP32-then-BF16
// rounding of a sum equal to direct BF16 rounding, so these equal the
// reference's FP32-op-then-round steps bit for bit.

#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "mamba_mimo_bwd_fwd.h"

namespace mmbf {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTargetCtas = 608;  // ~4 per SM on a 152-SM GB300; device-independent

// ---------------------------------------------------------------------------
// Number formats

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
__device__ __forceinline__ float bf_f(uint16_t u) { return __uint_as_float(((uint32_t)u) << 16); }
__device__ __forceinline__ uint16_t f_bf(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float round_bf(float x) { return bf_f(f_bf(x)); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return (uint32_t)f_bf(lo) | ((uint32_t)f_bf(hi) << 16);
}
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t badd2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// ---------------------------------------------------------------------------
// Tensor-core fragments (mma.sync m16n8k16, BF16 in, FP32 accumulate).

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// acc[2][4] += A[m0:m0+16, 0:K] * B[0:K, n0:n0+16] for one warp.
//   A_T = false: A stored row-major [M][K] (leading dim lda)
//   A_T = true : A stored as its transpose, row-major [K][M]
//   B_KN = false: B stored as its transpose, row-major [N][K]
//   B_KN = true : B stored row-major [K][N]
// All tiles are padded to multiples of 16 rows/cols with zeros, and every
// row stride is an odd multiple of 16 bytes (ldmatrix rows hit distinct banks).
template <bool A_T, bool B_KN>
__device__ __forceinline__ void warp_mma_16x16(float (&acc)[2][4], const uint16_t* A, int lda,
                                               int m0, const uint16_t* B, int ldb, int n0, int K) {
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3, li = lane & 7;
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
    if (!A_T) {
      ldsm_x4(a0, a1, a2, a3, A + (m0 + (lane & 15)) * lda + k0 + (lane >> 4) * 8);
    } else {
      ldsm_x4_t(a0, a1, a2, a3, A + (k0 + (mi >> 1) * 8 + li) * lda + m0 + (mi & 1) * 8);
    }
    if (!B_KN) {
      ldsm_x4(b0, b1, b2, b3, B + (n0 + (mi >> 1) * 8 + li) * ldb + k0 + (mi & 1) * 8);
    } else {
      ldsm_x4_t(b0, b1, b2, b3, B + (k0 + (mi & 1) * 8 + li) * ldb + n0 + (mi >> 1) * 8);
    }
    mma16816(acc[0], a0, a1, a2, a3, b0, b1);
    mma16816(acc[1], a0, a1, a2, a3, b2, b3);
  }
}

// ---------------------------------------------------------------------------
// Problem description shared by host and device.

struct Params {
  int B, S, H, G, R, N, P, C, div, w, half;
  int nc, CR, MP, NP, PS, npslice, L, nseg;
  int reduced, has_z, has_d, vec_p;  // vec_p: P even (pairs of p are 4-byte aligned)
  int fast;                          // index of the shape-specialised kernels, or -1
  int tc;                            // 1: the warp-specialised tensor-core output kernel (mmbf_tc.cuh)
  int fused;                         // 1: its single-kernel form (phase A in the kernel, cooperative launch)
  int UA, LA, nunit;                 // state units per segment, chunks per unit, units per head
  const uint16_t *dout, *q, *k, *v, *z, *trap;
  const float *q_bias, *k_bias, *mimo_v, *mimo_o, *mimo_z, *angles, *da_cs, *da_cs_rev, *dt,
      *d, *segsum;
  float *dmimo_o, *dmimo_z;
  uint16_t *states, *dz, *qk_dot;
  uint16_t* y;  // the layer's forward output (layout of dout) or NULL
  int want_y;
  float *ws_state, *ws_decay, *ws_grad;
  unsigned int* ws_count;  // per (b,h): output CTAs done (specialised kernels)
  unsigned int* ws_flag;   // per (b,h) and segment: its sum is published (single-kernel form)
  unsigned int* ws_err;    // device-side error word: (tag << 8) | code of the failing call
  unsigned int tag;        // call tag (24 bits) for ws_err
  int test_flags;          // test hooks (mamba_mimo_set_test_hooks); 0 in normal use
  // Tensor maps of the specialised kernels with 128-byte rows (TMA loads):
  // q, k [N,G,R,S,B]; v, z, reduced dout [P,H,S,B]; per-rank dout
  // [P,H,R,S,B]; angles [W,H,S,B].  Unused maps are left zero.
  CUtensorMap tm_q, tm_k, tm_v, tm_dout, tm_z, tm_ang;
  CUtensorMap tm_states;   // states as [B*H*nc*N][P] (TMA tile stores)
  CUtensorMap tm_dz;       // dz [P,H,S,B] (TMA tile stores)
  CUtensorMap tm_y;        // y in dout's layout (TMA tile stores)
};

__host__ __device__ inline int round16(int x) { return (x + 15) & ~15; }
__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// Shared-memory carve-up of chunk_output_kernel (byte offsets).
struct OutLayout {
  size_t Qt, Kt, Pt, At, Sb, X, st, qkS, eseg, qbb, kbb, mvb, mob, mzf, tok, red, total;
};
__host__ __device__ inline OutLayout out_layout(const Params& p) {
  OutLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align16(o + bytes); return at; };
  L.Qt = take((size_t)p.MP * (p.NP + 8) * 2);
  L.Kt = take((size_t)p.MP * (p.NP + 8) * 2);
  L.Pt = take((size_t)p.MP * (p.PS + 8) * 2);
  L.At = take((size_t)p.MP * (p.MP + 8) * 2);
  L.Sb = take((size_t)p.NP * (p.PS + 8) * 2);
  L.X = take((size_t)p.MP * (p.PS + 4) * 4);
  L.st = take((size_t)p.NP * (p.PS + 4) * 4);
  const size_t tiles_end = o;
  L.qkS = take((size_t)p.C * p.R * p.R * 4);
  L.eseg = take(p.C <= 64 ? (size_t)p.C * p.C * 4 : 0);
  L.qbb = take((size_t)p.R * p.NP * 2);
  L.kbb = take((size_t)p.R * p.NP * 2);
  L.mvb = take((size_t)p.R * p.PS * 2);
  L.mob = take((size_t)p.R * p.PS * 2);
  L.mzf = take((size_t)p.R * p.PS * 4);
  L.tok = take((size_t)p.C * 4 * 4);
  // End-of-segment reduction scratch: reuses the tile region when it fits.
  const size_t red_bytes = (size_t)(kThreads / (p.PS / 2)) * 2 * p.R * p.PS * 4;
  if (red_bytes <= tiles_end) {
    L.red = 0;
  } else {
    L.red = take(red_bytes);
  }
  L.total = o;
  return L;
}

struct StateLayout {
  size_t Kt, Pt, st, kbb, mvb, tok, total;
};
__host__ __device__ inline StateLayout state_layout(const Params& p) {
  StateLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align16(o + bytes); return at; };
  L.Kt = take((size_t)p.MP * (p.NP + 8) * 2);
  L.Pt = take((size_t)p.MP * (p.PS + 8) * 2);
  L.st = take((size_t)p.NP * (p.PS + 4) * 4);
  L.kbb = take((size_t)p.R * p.NP * 2);
  L.mvb = take((size_t)p.R * p.PS * 2);
  L.tok = take((size_t)p.C * 4 * 4);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------
// Per-chunk building blocks (shared by the state and output kernels).

// Per-token scalars of chunk c: gamma (FP32), factor (BF16 value), exp(da_cs),
// exp(da_cs_rev).  Trapezoid rule of the reference: gamma = bf16(dt)
// sigmoid(trap); shifted = bf16(bf16(dt[t+1]) sigmoid(-trap[t+1])) (0 past the
// padded end); factor = bf16(gamma + shifted).  Padded tokens read dt = trap =
// da_cs = da_cs_rev = 0.
__device__ void token_scalars(const Params& p, int bh, int c, float* tok) {
  const int64_t row = (int64_t)bh * p.S;
  const int Sp = p.nc * p.C;
  for (int t = threadIdx.x; t < p.C; t += blockDim.x) {
    const int tg = c * p.C + t;
    float gam = 0.f, fac, eda = 1.f, edr = 1.f;
    float dtv = 0.f, trv = 0.f;
    if (tg < p.S) {
      dtv = p.dt[row + tg];
      trv = bf_f(p.trap[row + tg]);
      eda = expf(p.da_cs[row + tg]);
      edr = expf(p.da_cs_rev[row + tg]);
    }
    gam = __fmul_rn(round_bf(dtv), sigmoid_f(trv));
    float sh = 0.f;
    if (tg + 1 < Sp) {
      float dtn = 0.f, trn = 0.f;
      if (tg + 1 < p.S) {
        dtn = p.dt[row + tg + 1];
        trn = bf_f(p.trap[row + tg + 1]);
      }
      sh = round_bf(__fmul_rn(round_bf(dtn), 1.0f / (1.0f + expf(trn))));
    }
    fac = round_bf(__fadd_rn(gam, sh));
    tok[t] = gam;
    tok[p.C + t] = fac;
    tok[2 * p.C + t] = eda;
    tok[3 * p.C + t] = edr;
  }
}

// BF16(x) of FP32 parameter rows [R][len] into a padded [R][ld] table.
__device__ void param_bf16(const float* src, int R, int len, uint16_t* dst, int ld, int col0,
                           int total_cols) {
  for (int e = threadIdx.x; e < R * ld; e += blockDim.x) {
    const int r = e / ld, x = e % ld;
    const int col = col0 + x;
    dst[e] = (x < len && col < total_cols) ? f_bf(src[r * total_cols + col]) : (uint16_t)0;
  }
}

// T[j][n] = bf16(src[b,t,r,g,n] + bf16(bias[h,r,n])) for the chunk's rows
// (pairs of n; N is even).  Padded tokens read q/k = 0.
__device__ void biased_tile(const Params& p, const uint16_t* src, const uint16_t* biasb,
                            uint16_t* T, int b, int g, int c) {
  const int ld = p.NP + 8, npairs = p.N / 2;
  for (int e = threadIdx.x; e < p.CR * npairs; e += blockDim.x) {
    const int j = e / npairs, n = 2 * (e % npairs);
    const int t = j / p.R, r = j % p.R;
    const int tg = c * p.C + t;
    uint32_t x = 0;
    if (tg < p.S)
      x = __ldg(reinterpret_cast<const uint32_t*>(
          src + ((((int64_t)b * p.S + tg) * p.R + r) * p.G + g) * p.N + n));
    const uint32_t bb = *reinterpret_cast<const uint32_t*>(biasb + r * p.NP + n);
    *reinterpret_cast<uint32_t*>(T + j * ld + n) = badd2(x, bb);
  }
}

// Rotary on the pairs (m, N/2 + m), m < N/div, in FP32 with the reference's
// operation order, each result rounded to BF16; applied to Q (if given) and K.
// Then K is scaled by the token's factor (BF16 x BF16 product, rounded):
// k_scaled = bf16(k_rot * factor).  One work item per (token, m < N/2).
__device__ void rotate_and_scale(const Params& p, uint16_t* Qt, uint16_t* Kt, const float* fac,
                                 int b, int h, int c) {
  const int ld = p.NP + 8;
  const int items = p.C * p.half;
  for (int e = threadIdx.x; e < items; e += blockDim.x) {
    const int t = e / p.half, m = e % p.half;
    const int tg = c * p.C + t;
    const uint16_t fb = f_bf(fac[t]);
    const float ff = bf_f(fb);
    float cs = 1.f, sn = 0.f;
    const bool rot = m < p.w;
    if (rot && tg < p.S) {
      const float th = p.angles[(((int64_t)b * p.S + tg) * p.H + h) * p.w + m];
      sincosf(th, &sn, &cs);
    }
    for (int r = 0; r < p.R; r++) {
      const int j = t * p.R + r;
      if (rot && Qt) {
        const float a = bf_f(Qt[j * ld + m]), x = bf_f(Qt[j * ld + p.half + m]);
        Qt[j * ld + m] = f_bf(__fsub_rn(__fmul_rn(cs, a), __fmul_rn(sn, x)));
        Qt[j * ld + p.half + m] = f_bf(__fadd_rn(__fmul_rn(sn, a), __fmul_rn(cs, x)));
      }
      float a = bf_f(Kt[j * ld + m]), x = bf_f(Kt[j * ld + p.half + m]);
      if (rot) {
        const float a2 = round_bf(__fsub_rn(__fmul_rn(cs, a), __fmul_rn(sn, x)));
        const float x2 = round_bf(__fadd_rn(__fmul_rn(sn, a), __fmul_rn(cs, x)));
        a = a2;
        x = x2;
      }
      Kt[j * ld + m] = f_bf(__fmul_rn(a, ff));
      Kt[j * ld + p.half + m] = f_bf(__fmul_rn(x, ff));
    }
  }
}

// k_state = bf16(k_scaled * exp(da_cs_rev[t])), in place.
__device__ void k_state_tile(const Params& p, uint16_t* Kt, const float* edr) {
  const int ld = p.NP + 8;
  for (int e = threadIdx.x; e < p.CR * p.N; e += blockDim.x) {
    const int j = e / p.N, n = e % p.N;
    Kt[j * ld + n] = f_bf(__fmul_rn(bf_f(Kt[j * ld + n]), edr[j / p.R]));
  }
}

// PsiV[j][pp] = bf16(v[b,t,h,p0+pp] * bf16(mimo_v[h,r,p0+pp])) for the p-slice.
__device__ void psi_tile(const Params& p, const uint16_t* mvb, uint16_t* Pt, int b, int h, int c,
                         int p0, int pw) {
  const int ld = p.PS + 8;
  if (p.vec_p) {
    const int npairs = (pw + 1) / 2;
    for (int e = threadIdx.x; e < p.CR * npairs; e += blockDim.x) {
      const int j = e / npairs, pp = 2 * (e % npairs);
      const int t = j / p.R, r = j % p.R, tg = c * p.C + t;
      uint32_t x = 0;
      if (tg < p.S)
        x = __ldg(reinterpret_cast<const uint32_t*>(
            p.v + (((int64_t)b * p.S + tg) * p.H + h) * p.P + p0 + pp));
      const uint32_t m = *reinterpret_cast<const uint32_t*>(mvb + r * p.PS + pp);
      *reinterpret_cast<uint32_t*>(Pt + j * ld + pp) = bmul2(x, m);
    }
  } else {
    for (int e = threadIdx.x; e < p.CR * pw; e += blockDim.x) {
      const int j = e / pw, pp = e % pw;
      const int t = j / p.R, r = j % p.R, tg = c * p.C + t;
      float x = 0.f;
      if (tg < p.S) x = bf_f(p.v[(((int64_t)b * p.S + tg) * p.H + h) * p.P + p0 + pp]);
      Pt[j * ld + pp] = f_bf(__fmul_rn(x, bf_f(mvb[r * p.PS + pp])));
    }
  }
}

// state <- alpha * state + Kt^T Pt  over the (NP x PS) tile (one GEMM, K = MP).
__device__ void state_update(const Params& p, float* st, const uint16_t* Kt, const uint16_t* Pt,
                             float alpha) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q4 = lane & 3;
  const int ldst = p.PS + 4;
  const int nmb = p.NP / 16, npb = p.PS / 16;
  for (int task = warp; task < nmb * npb; task += kWarps) {
    const int m0 = (task / npb) * 16, n0 = (task % npb) * 16;
    float acc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; nt++) {
      const int col = n0 + nt * 8 + 2 * q4;
      acc[nt][0] = st[(m0 + g) * ldst + col] * alpha;
      acc[nt][1] = st[(m0 + g) * ldst + col + 1] * alpha;
      acc[nt][2] = st[(m0 + g + 8) * ldst + col] * alpha;
      acc[nt][3] = st[(m0 + g + 8) * ldst + col + 1] * alpha;
    }
    warp_mma_16x16<true, true>(acc, Kt, p.NP + 8, m0, Pt, p.PS + 8, n0, p.MP);
#pragma unroll
    for (int nt = 0; nt < 2; nt++) {
      const int col = n0 + nt * 8 + 2 * q4;
      st[(m0 + g) * ldst + col] = acc[nt][0];
      st[(m0 + g) * ldst + col + 1] = acc[nt][1];
      st[(m0 + g + 8) * ldst + col] = acc[nt][2];
      st[(m0 + g + 8) * ldst + col + 1] = acc[nt][3];
    }
  }
}

__device__ void zero_smem(unsigned char* base, size_t bytes) {
  uint4* p = reinterpret_cast<uint4*>(base);
  const size_t n = bytes / 16;
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) p[i] = make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------------------
// Kernel 1: segment-local state sums.

__global__ void __launch_bounds__(kThreads) segment_state_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const StateLayout Ly = state_layout(p);
  uint16_t* Kt = reinterpret_cast<uint16_t*>(smem + Ly.Kt);
  uint16_t* Pt = reinterpret_cast<uint16_t*>(smem + Ly.Pt);
  float* st = reinterpret_cast<float*>(smem + Ly.st);
  uint16_t* kbb = reinterpret_cast<uint16_t*>(smem + Ly.kbb);
  uint16_t* mvb = reinterpret_cast<uint16_t*>(smem + Ly.mvb);
  float* tok = reinterpret_cast<float*>(smem + Ly.tok);

  const int ps = blockIdx.x, seg = blockIdx.y, bh = blockIdx.z;
  const int b = bh / p.H, h = bh % p.H, g = h / (p.H / p.G);
  const int p0 = ps * p.PS, pw = min(p.PS, p.P - p0);
  const int c0 = seg * p.L, c1 = min(p.nc, c0 + p.L);

  zero_smem(smem, Ly.total);
  __syncthreads();
  param_bf16(p.k_bias + (int64_t)h * p.R * p.N, p.R, p.N, kbb, p.NP, 0, p.N);
  param_bf16(p.mimo_v + (int64_t)h * p.R * p.P, p.R, pw, mvb, p.PS, p0, p.P);
  float decay = 1.f;
  for (int c = c0; c < c1; c++) {
    __syncthreads();
    token_scalars(p, bh, c, tok);
    __syncthreads();
    biased_tile(p, p.k, kbb, Kt, b, g, c);
    psi_tile(p, mvb, Pt, b, h, c, p0, pw);
    __syncthreads();
    rotate_and_scale(p, nullptr, Kt, tok + p.C, b, h, c);
    __syncthreads();
    k_state_tile(p, Kt, tok + 3 * p.C);
    __syncthreads();
    const int last = min(c * p.C + p.C, p.S) - 1;
    const float alpha = expf(p.da_cs[(int64_t)bh * p.S + last]);
    state_update(p, st, Kt, Pt, alpha);
    decay *= alpha;
  }
  __syncthreads();
  float* dst = p.ws_state + ((int64_t)bh * p.nseg + seg) * p.N * p.P;
  for (int e = threadIdx.x; e < p.N * pw; e += blockDim.x) {
    const int n = e / pw, pp = e % pw;
    dst[n * p.P + p0 + pp] = st[n * (p.PS + 4) + pp];
  }
  if (ps == 0 && threadIdx.x == 0) p.ws_decay[(int64_t)bh * p.nseg + seg] = decay;
}

// ---------------------------------------------------------------------------
// Kernel 2: exclusive prefix over segments (in place): entering state.

__global__ void segment_prefix_kernel(Params p) {
  const int bh = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= p.N * p.P) return;
  float acc = 0.f;
  float* base = p.ws_state + (int64_t)bh * p.nseg * p.N * p.P + e;
  const float* dec = p.ws_decay + (int64_t)bh * p.nseg;
  for (int s = 0; s < p.nseg; s++) {
    const float loc = base[(int64_t)s * p.N * p.P];
    base[(int64_t)s * p.N * p.P] = acc;
    acc = acc * dec[s] + loc;
  }
}

// ---------------------------------------------------------------------------
// Kernel 3: per-chunk outputs and gradients.

template <int RMAX>
__global__ void __launch_bounds__(kThreads) chunk_output_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const OutLayout Ly = out_layout(p);
  uint16_t* Qt = reinterpret_cast<uint16_t*>(smem + Ly.Qt);
  uint16_t* Kt = reinterpret_cast<uint16_t*>(smem + Ly.Kt);
  uint16_t* Pt = reinterpret_cast<uint16_t*>(smem + Ly.Pt);
  uint16_t* At = reinterpret_cast<uint16_t*>(smem + Ly.At);
  uint16_t* Sb = reinterpret_cast<uint16_t*>(smem + Ly.Sb);
  float* X = reinterpret_cast<float*>(smem + Ly.X);
  float* st = reinterpret_cast<float*>(smem + Ly.st);
  float* qkS = reinterpret_cast<float*>(smem + Ly.qkS);
  float* eseg = reinterpret_cast<float*>(smem + Ly.eseg);
  uint16_t* qbb = reinterpret_cast<uint16_t*>(smem + Ly.qbb);
  uint16_t* kbb = reinterpret_cast<uint16_t*>(smem + Ly.kbb);
  uint16_t* mvb = reinterpret_cast<uint16_t*>(smem + Ly.mvb);
  uint16_t* mob = reinterpret_cast<uint16_t*>(smem + Ly.mob);
  float* mzf = reinterpret_cast<float*>(smem + Ly.mzf);
  float* tok = reinterpret_cast<float*>(smem + Ly.tok);
  float* red = reinterpret_cast<float*>(smem + Ly.red);

  const int ps = blockIdx.x, seg = blockIdx.y, bh = blockIdx.z;
  const int b = bh / p.H, h = bh % p.H, g = h / (p.H / p.G);
  const int p0 = ps * p.PS, pw = min(p.PS, p.P - p0);
  const int c0 = seg * p.L, c1 = min(p.nc, c0 + p.L);
  const int R = p.R, C = p.C, CR = p.CR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lg = lane >> 2, lq = lane & 3;
  const int ldQ = p.NP + 8, ldP = p.PS + 8, ldA = p.MP + 8, ldX = p.PS + 4;
  const float dval = p.has_d ? p.d[h] : 0.f;

  zero_smem(smem, Ly.total);
  __syncthreads();
  param_bf16(p.q_bias + (int64_t)h * R * p.N, R, p.N, qbb, p.NP, 0, p.N);
  param_bf16(p.k_bias + (int64_t)h * R * p.N, R, p.N, kbb, p.NP, 0, p.N);
  param_bf16(p.mimo_v + (int64_t)h * R * p.P, R, pw, mvb, p.PS, p0, p.P);
  if (p.reduced) param_bf16(p.mimo_o + (int64_t)h * R * p.P, R, pw, mob, p.PS, p0, p.P);
  if (p.has_z)
    for (int e = threadIdx.x; e < R * p.PS; e += blockDim.x) {
      const int r = e / p.PS, x = e % p.PS;
      mzf[e] = (x < pw) ? p.mimo_z[((int64_t)h * R + r) * p.P + p0 + x] : 0.f;
    }
  {  // entering state of the segment
    const float* src = p.ws_state + ((int64_t)bh * p.nseg + seg) * p.N * p.P;
    for (int e = threadIdx.x; e < p.N * pw; e += blockDim.x) {
      const int n = e / pw, pp = e % pw;
      st[n * ldX + pp] = src[n * p.P + p0 + pp];
    }
  }

  // Epilogue work assignment: thread -> fixed pair of columns (pp, pp+1) of the
  // slice, tokens t = slot, slot + nslots, ...
  const int npairs = p.PS / 2, nslots = kThreads / npairs;
  const int my_pair = threadIdx.x % npairs, my_slot = threadIdx.x / npairs;
  const int pp = 2 * my_pair;
  const bool col0_ok = pp < pw, col1_ok = pp + 1 < pw;
  float dmo[RMAX][2], dmz[RMAX][2];
#pragma unroll
  for (int r = 0; r < RMAX; r++) dmo[r][0] = dmo[r][1] = dmz[r][0] = dmz[r][1] = 0.f;

  for (int c = c0; c < c1; c++) {
    __syncthreads();
    token_scalars(p, bh, c, tok);
    if (C <= 64) {
      const float* sg = p.segsum + (((int64_t)bh * p.nc + c) * C) * C;
      for (int e = threadIdx.x; e < C * C; e += blockDim.x) {
        const int ti = e / C, tj = e % C;
        eseg[e] = (tj < ti) ? expf(sg[e]) : 0.f;
      }
    }
    // (1) biased Q/K, PsiV, bf16(state) (+ the states output)
    biased_tile(p, p.q, qbb, Qt, b, g, c);
    biased_tile(p, p.k, kbb, Kt, b, g, c);
    psi_tile(p, mvb, Pt, b, h, c, p0, pw);
    {
      uint16_t* so = p.states + (((int64_t)bh * p.nc + c) * p.N) * p.P + p0;
      for (int e = threadIdx.x; e < p.N * pw; e += blockDim.x) {
        const int n = e / pw, x = e % pw;
        const uint16_t u = f_bf(st[n * ldX + x]);
        Sb[n * ldP + x] = u;
        so[(int64_t)n * p.P + x] = u;
      }
    }
    __syncthreads();
    // (2) same-token qk_dot on the diagonal tiles of Qh Kh^T
    for (int rb = warp; rb * 16 < CR; rb += kWarps) {
      const int tlo = (rb * 16) / R, thi = min((rb * 16 + 15) / R, C - 1);
      const int cb0 = (tlo * R) / 16, cb1 = (min((thi + 1) * R, CR) + 15) / 16;
      for (int cb = cb0; cb < cb1; cb++) {
        float acc[2][4] = {};
        warp_mma_16x16<false, false>(acc, Qt, ldQ, rb * 16, Kt, ldQ, cb * 16, p.NP);
#pragma unroll
        for (int nt = 0; nt < 2; nt++)
#pragma unroll
          for (int x = 0; x < 4; x++) {
            const int row = rb * 16 + lg + ((x >> 1) << 3);
            const int col = cb * 16 + nt * 8 + 2 * lq + (x & 1);
            if (row < CR && col < CR && row / R == col / R)
              qkS[row * R + col % R] = round_bf(acc[nt][x]);
          }
      }
    }
    __syncthreads();
    if (ps == 0) {  // qk_dot output: [B,H,S,R,R], contiguous per chunk
      const int tcount = min(C, p.S - c * C);
      uint16_t* qo = p.qk_dot + (((int64_t)bh * p.S) + (int64_t)c * C) * R * R;
      for (int e = threadIdx.x; e < tcount * R * R; e += blockDim.x) qo[e] = f_bf(qkS[e]);
    }
    // (3) rotary (Q and K), k_scaled = bf16(k_rot * factor)
    rotate_and_scale(p, Qt, Kt, tok + C, b, h, c);
    __syncthreads();
    // Without mimo_o, z and y the chunk output feeds nothing: only the state
    // update remains.
    if (!(p.reduced || p.has_z || p.want_y)) {
      k_state_tile(p, Kt, tok + 3 * C);
      __syncthreads();
      const int last = min(c * C + C, p.S) - 1;
      state_update(p, st, Kt, Pt, expf(p.da_cs[(int64_t)bh * p.S + last]));
      continue;
    }
    // (4) causal A = bf16(mask(Q Ks^T) exp(segsum)) and inter = (Q bf16(state)) exp(da_cs)
    {
      const int nrb = (CR + 15) / 16;
      // tasks: A strips (rb, cb < klim/16), then inter strips (rb, pb < PS/16)
      int ntask_a = 0;
      for (int rb = 0; rb < nrb; rb++) {
        const int thi = min((rb * 16 + 15) / R, C - 1);
        ntask_a += round16(min(thi * R, CR)) / 16;
      }
      const int npb = p.PS / 16;
      const int ntask = ntask_a + nrb * npb;
      for (int task = warp; task < ntask; task += kWarps) {
        if (task < ntask_a) {
          int rb = 0, rem = task;
          for (;; rb++) {
            const int thi = min((rb * 16 + 15) / R, C - 1);
            const int nk = round16(min(thi * R, CR)) / 16;
            if (rem < nk) break;
            rem -= nk;
          }
          const int cb = rem;
          float acc[2][4] = {};
          warp_mma_16x16<false, false>(acc, Qt, ldQ, rb * 16, Kt, ldQ, cb * 16, p.NP);
#pragma unroll
          for (int nt = 0; nt < 2; nt++)
#pragma unroll
            for (int x = 0; x < 4; x++) {
              const int row = rb * 16 + lg + ((x >> 1) << 3);
              const int col = cb * 16 + nt * 8 + 2 * lq + (x & 1);
              float val = 0.f;
              if (row < CR && col < CR) {
                const int ti = row / R, tj = col / R;
                if (ti > tj) {
                  const float e = (C <= 64)
                                      ? eseg[ti * C + tj]
                                      : expf(p.segsum[(((int64_t)bh * p.nc + c) * C + ti) * C + tj]);
                  val = __fmul_rn(acc[nt][x], e);
                }
              }
              At[row * ldA + col] = f_bf(val);
            }
        } else {
          const int t2 = task - ntask_a;
          const int rb = t2 / npb, n0 = (t2 % npb) * 16;
          float acc[2][4] = {};
          warp_mma_16x16<false, true>(acc, Qt, ldQ, rb * 16, Sb, ldP, n0, p.NP);
#pragma unroll
          for (int nt = 0; nt < 2; nt++)
#pragma unroll
            for (int x = 0; x < 4; x++) {
              const int row = rb * 16 + lg + ((x >> 1) << 3);
              const int col = n0 + nt * 8 + 2 * lq + (x & 1);
              const float e = row < CR ? tok[2 * C + row / R] : 0.f;
              X[row * ldX + col] = __fmul_rn(acc[nt][x], e);
            }
        }
      }
    }
    __syncthreads();
    // (5) intra = A PsiV added to X; k_state in place
    {
      const int nrb = (CR + 15) / 16, npb = p.PS / 16;
      for (int task = warp; task < nrb * npb; task += kWarps) {
        const int rb = task / npb, n0 = (task % npb) * 16;
        const int thi = min((rb * 16 + 15) / R, C - 1);
        const int klim = round16(min(thi * R, CR));
        if (klim == 0) continue;
        float acc[2][4] = {};
        warp_mma_16x16<false, true>(acc, At, ldA, rb * 16, Pt, ldP, n0, klim);
#pragma unroll
        for (int nt = 0; nt < 2; nt++)
#pragma unroll
          for (int x = 0; x < 4; x++) {
            const int row = rb * 16 + lg + ((x >> 1) << 3);
            const int col = n0 + nt * 8 + 2 * lq + (x & 1);
            X[row * ldX + col] = __fadd_rn(X[row * ldX + col], acc[nt][x]);
          }
      }
    }
    k_state_tile(p, Kt, tok + 3 * C);
    __syncthreads();
    // (6) state update (tensor cores) and the per-element epilogue
    {
      const int last = min(c * C + C, p.S) - 1;
      const float alpha = expf(p.da_cs[(int64_t)bh * p.S + last]);
      state_update(p, st, Kt, Pt, alpha);
    }
    for (int t = my_slot; t < C; t += nslots) {
      const int tg = c * C + t;
      const bool valid = tg < p.S;
      const float gam = tok[t];
      float zt[2] = {0.f, 0.f}, dov[2] = {0.f, 0.f};
      const int64_t rowbase = (((int64_t)b * p.S + tg) * p.H + h) * p.P + p0 + pp;
      if (valid) {
        if (p.has_z) {
          if (col0_ok) zt[0] = bf_f(p.z[rowbase]);
          if (col1_ok) zt[1] = bf_f(p.z[rowbase + 1]);
        }
        if (p.reduced) {
          if (col0_ok) dov[0] = bf_f(p.dout[rowbase]);
          if (col1_ok) dov[1] = bf_f(p.dout[rowbase + 1]);
        }
      }
      float dzacc[2] = {0.f, 0.f}, yacc[2] = {0.f, 0.f};
#pragma unroll 1
      for (int o = 0; o < R; o++) {
        const int jo = t * R + o;
        // diagonal: rank-ordered BF16 products and sums, then * gamma
        uint32_t dg2 = 0;
        for (int r = 0; r < R; r++) {
          const uint32_t qb = f_bf(qkS[jo * R + r]);
          const uint32_t q2 = qb | (qb << 16);
          const uint32_t ps2 = *reinterpret_cast<const uint32_t*>(Pt + (t * R + r) * ldP + pp);
          dg2 = badd2(dg2, bmul2(q2, ps2));
        }
        const uint32_t psi2 = *reinterpret_cast<const uint32_t*>(Pt + jo * ldP + pp);
        float outv[2];
#pragma unroll
        for (int x = 0; x < 2; x++) {
          const float dg = round_bf(__fmul_rn(x ? bf_hi(dg2) : bf_lo(dg2), gam));
          float acc = __fadd_rn(X[jo * ldX + pp + x], dg);
          if (p.has_d) acc = __fadd_rn(acc, __fmul_rn(dval, x ? bf_hi(psi2) : bf_lo(psi2)));
          outv[x] = round_bf(acc);
        }
#pragma unroll
        for (int x = 0; x < 2; x++) {
          if (!(x ? col1_ok : col0_ok)) continue;
          const float o_ = outv[x];
          float pz = 0.f, sg = 0.5f, pre = 0.f;
          if (p.has_z) {
            pz = __fmul_rn(zt[x], mzf[o * p.PS + pp + x]);
            sg = sigmoid_f(pz);
          }
          if (p.want_y) {  // y: mimo_o out silu(pz) summed over ranks, or per rank
            const float g_ = p.has_z ? __fmul_rn(pz, sg) : 1.f;
            if (p.reduced)
              yacc[x] = __fmaf_rn(__fmul_rn(p.mimo_o[((int64_t)h * R + o) * p.P + p0 + pp + x], o_), g_, yacc[x]);
            else if (valid)
              p.y[((((int64_t)b * p.S + tg) * R + o) * p.H + h) * p.P + p0 + pp + x] = f_bf(__fmul_rn(o_, g_));
          }
          if (p.reduced) {
            const float dv = dov[x];
            if (p.has_z) {
              dmo[o][x] += __fmul_rn(__fmul_rn(o_, __fmul_rn(pz, sg)), dv);
              pre = round_bf(__fmul_rn(round_bf(__fmul_rn(dv, bf_f(mob[o * p.PS + pp + x]))), o_));
            } else {
              dmo[o][x] += __fmul_rn(o_, dv);
            }
          } else if (p.has_z && valid) {
            const float dr = bf_f(p.dout[((((int64_t)b * p.S + tg) * R + o) * p.H + h) * p.P + p0 +
                                         pp + x]);
            pre = round_bf(__fmul_rn(dr, o_));
          }
          if (p.has_z) {
            const float gzp =
                __fmul_rn(__fmul_rn(pre, sg), __fadd_rn(1.f, __fmul_rn(pz, 1.0f / (1.0f + expf(pz)))));
            dzacc[x] = round_bf(__fadd_rn(dzacc[x], __fmul_rn(gzp, mzf[o * p.PS + pp + x])));
            dmz[o][x] += __fmul_rn(gzp, zt[x]);
          }
        }
      }
      if (p.has_z && valid) {
        if (col0_ok) p.dz[rowbase] = f_bf(dzacc[0]);
        if (col1_ok) p.dz[rowbase + 1] = f_bf(dzacc[1]);
      }
      if (p.want_y && p.reduced && valid) {
        if (col0_ok) p.y[rowbase] = f_bf(yacc[0]);
        if (col1_ok) p.y[rowbase + 1] = f_bf(yacc[1]);
      }
    }
  }
  // End of segment: fixed-order reduction of dmimo_o / dmimo_z partials over the
  // threads that share a column pair, into this segment's workspace slot.
  if (p.reduced || p.has_z) {
    __syncthreads();
    for (int r = 0; r < R; r++)
      for (int x = 0; x < 2; x++) {
        red[((my_slot * 2 + 0) * R + r) * p.PS + pp + x] = (r < RMAX) ? dmo[r][x] : 0.f;
        red[((my_slot * 2 + 1) * R + r) * p.PS + pp + x] = (r < RMAX) ? dmz[r][x] : 0.f;
      }
    __syncthreads();
    float* dst = p.ws_grad + ((int64_t)bh * p.nseg + seg) * 2 * R * p.P;
    for (int e = threadIdx.x; e < 2 * R * pw; e += blockDim.x) {
      const int which = e / (R * pw), r = (e / pw) % R, x = e % pw;
      float s = 0.f;
      for (int sl = 0; sl < nslots; sl++) s += red[((sl * 2 + which) * R + r) * p.PS + x];
      dst[((int64_t)which * R + r) * p.P + p0 + x] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// Kernel 4: dmimo_o / dmimo_z = sum over segments (fixed order).

__global__ void grad_reduce_kernel(Params p) {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");  // no-op unless launched as a dependent
  const int bh = blockIdx.x;
  const int RP = p.R * p.P;
  for (int e = threadIdx.x; e < 2 * RP; e += blockDim.x) {
    const int which = e / RP, x = e % RP;
    if (which == 0 && !p.reduced) continue;
    if (which == 1 && !p.has_z) continue;
    float s = 0.f;
    const float* src = p.ws_grad + (int64_t)bh * p.nseg * 2 * RP + (int64_t)which * RP + x;
    for (int sgm = 0; sgm < p.nseg; sgm++) s += src[(int64_t)sgm * 2 * RP];
    (which == 0 ? p.dmimo_o : p.dmimo_z)[(int64_t)bh * RP + x] = s;
  }
}

#include "mmbf_fast.cuh"
#include "mmbf_tc.cuh"

// ---------------------------------------------------------------------------
// Host side: planning, validation, launch.

static thread_local char g_err[512] = "";
static thread_local int g_launches = 0;
static thread_local void* const* g_stage_events = nullptr;
static thread_local int g_stage_count = 0;
static thread_local cudaError_t g_stage_error = cudaSuccess;
static thread_local int g_failed_stage = -1;  // kernel index of a failed launch
static thread_local int g_variant = -1;       // kernel family of the last call
static thread_local int g_plan[7] = {0, 0, 0, 0, 0, 0, 0};  // L, nseg, UA, LA, output slots, single kernel, refusal
static thread_local int g_fused_refused = 0;  // error code of a refused single-kernel launch (diagnostic)
static thread_local unsigned int g_last_tag = 0;           // tag of this thread's last call
static thread_local int g_test_flags = 0;                  // mamba_mimo_set_test_hooks
static thread_local const unsigned int* g_last_err_word = nullptr;
// 24-bit call tags, never 0, so a stale or uninitialised error word is
// unlikely to carry the tag of the call being checked.
static unsigned int next_call_tag() {
  static std::atomic<unsigned int> n{0};
  unsigned int t;
  do {
    t = (n.fetch_add(1, std::memory_order_relaxed) + 1) & 0xffffffu;
  } while (t == 0);
  return t;
}
static const char* const kStageNames[4] = {"segment_state", "segment_prefix", "chunk_output",
                                           "grad_reduce"};
static const char* const kFastStageNames[3] = {"segment_state", "segment_prefix", "chunk_output"};
static const char* const kTcStageNames[2] = {"segment_state", "chunk_output"};
static const char* const kTcFusedStageNames[1] = {"chunk_output"};
static thread_local const char* const* g_stage_names = kStageNames;  // kernels of the last call
static thread_local int g_stage_names_n = 4;

// Records the optional timing event around kernel `i` (before: which = 0).
static void stage_event(int i, int which, cudaStream_t s) {
  const int k = 2 * i + which;
  if (g_stage_events && k < (g_stage_count / 2) * 2 && g_stage_events[k]) {
    const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(g_stage_events[k]), s);
    if (e != cudaSuccess && g_stage_error == cudaSuccess) g_stage_error = e;
  }
}

// Function attributes are per device: caches of them are kept per device
// ordinal, the last slot standing for any device past the table (never
// cached there: its value is reset on every use).
constexpr int kMaxDevices = 16;
static int device_slot() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = 0;
  }
  return (dev >= 0 && dev < kMaxDevices) ? dev : kMaxDevices;
}

// cudaFuncSetAttribute once per kernel, size and device (kept out of stream capture).
template <typename K>
static cudaError_t ensure_smem(K kern, size_t smem, int* cached) {
  if ((int)smem <= *cached) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  // the whole unified L1 / shared array as shared memory, so occupancy
  // queries and launches both see every CTA that fits
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) *cached = (int)smem;
  return e;
}

static mmbf_status fail(mmbf_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

static size_t out_smem_bytes(Params p, int PS) {
  p.PS = PS;
  return out_layout(p).total;
}

static const size_t kSmemLimit = 227 * 1024;

// ---- shape-specialised kernels: instantiated shapes and launch plan
using FastA = fast::Cfg<4, 16, 64, 64, 4, 1>;  // R4 C16 N=P=64 (the pages' timed and unit-test shape)
using FastB = fast::Cfg<8, 16, 64, 64, 4, 2>;  // R8 C16 N=P=64
using FastC = fast::Cfg<4, 16, 32, 32, 4, 1>;  // R4 C16 N=P=32
using FastD = fast::Cfg<4, 32, 128, 64, 2, 1>;  // R4 C32 N=128 P=64, rotary on all of N (wide state)

template <class K>
static size_t fast_out_smem(const Params& p) {
  return fast::smem_layout<K>(true, p.reduced, p.has_z, p.want_y).total;
}
// The state-sum kernel always runs one warp per j-block.
template <class K>
using StateCfg = fast::Cfg<K::R, K::C, K::N, K::P, K::DIV, 1>;
template <class K>
static size_t fast_state_smem(const Params& p) {
  return fast::smem_layout<StateCfg<K>>(false, p.reduced, p.has_z).total;
}
// A family takes the shape when its tile set fits in shared memory for the
// call's branches both without and with the forward output y, so the two
// entry points run the same kernels (the wide-state tiles leave no room for
// per-rank dout).
template <class K>
static bool fast_fits(const Params& p) {
  Params py = p;
  py.want_y = 1;
  return p.R == K::R && p.C == K::C && p.N == K::N && p.P == K::P && p.div == K::DIV &&
         fast_out_smem<K>(p) <= kSmemLimit && fast_out_smem<K>(py) <= kSmemLimit &&
         fast_state_smem<K>(p) <= kSmemLimit;
}
static int fast_index(const Params& p) {
  if (fast_fits<FastA>(p)) return 0;
  if (fast_fits<FastB>(p)) return 1;
  if (fast_fits<FastC>(p)) return 2;
  if (fast_fits<FastD>(p)) return 3;
  return -1;
}

// Largest dynamic shared memory each fast kernel has been opened for on the
// current device.  The limit is only ever raised (a lower request must never
// shrink it, or a later launch with a larger layout would fail).
template <class K, int MODE = -1>
static int& fast_out_smem_set() {
  static int v[kMaxDevices + 1];
  const int d = device_slot();
  if (d == kMaxDevices) v[d] = 0;
  return v[d];
}
template <class K>
static int& fast_state_smem_set() {
  static int v[kMaxDevices + 1];
  const int d = device_slot();
  if (d == kMaxDevices) v[d] = 0;
  return v[d];
}

// The launch plan is a pure function of the problem (shape and branches):
// the workspace size query and the call agree on any device, with or without
// a device current.  It assumes a GB300's 152 SMs and each kernel's resident
// CTAs per SM as fixed by its launch bounds, shared memory (plus the 1 KB per-
// CTA reservation, 228 KB per SM) and tensor-memory columns (512 per SM).  On
// another device the plan is still correct, only its wave count may differ.
constexpr int kPlanSms = 152;
constexpr size_t kSmemPerSm = 228 * 1024, kSmemReserved = 1024;
static int per_sm(int launch_bound_ctas, size_t smem, int tmem_cols) {
  int n = launch_bound_ctas;
  n = std::min(n, (int)(kSmemPerSm / (smem + kSmemReserved)));
  if (tmem_cols > 0) n = std::min(n, 512 / tmem_cols);
  return std::max(n, 1);
}
// Resident output-kernel CTAs (all SMs) of the shape-specialised family.
template <class K>
static int fast_slots_of(const Params& p) {
  return kPlanSms * per_sm(K::OUT_CTAS, fast_out_smem<K>(p), K::TM_COLS);
}
// Resident state-kernel CTAs (all SMs).
template <class K>
static int fast_state_slots_of(const Params& p) {
  return kPlanSms * per_sm(StateCfg<K>::STATE_CTAS, fast_state_smem<K>(p), K::UMMA ? 64 : 0);
}
static int fast_state_slots(const Params& p) {
  switch (p.fast) {
    case 0: return fast_state_slots_of<FastA>(p);
    case 1: return fast_state_slots_of<FastB>(p);
    case 2: return fast_state_slots_of<FastC>(p);
    default: return fast_state_slots_of<FastD>(p);
  }
}
static int fast_slots(const Params& p) {
  if (p.tc) return kPlanSms;  // one warp-specialised CTA per SM (all of its tensor memory)
  switch (p.fast) {
    case 0: return fast_slots_of<FastA>(p);
    case 1: return fast_slots_of<FastB>(p);
    case 2: return fast_slots_of<FastC>(p);
    default: return fast_slots_of<FastD>(p);
  }
}
// Chunks per segment: the length that minimises (waves x (L + per-CTA setup)),
// with every segment a CTA of the output kernel.
static int fast_segment_length(const Params& p, int slots) {
  static thread_local int64_t key[3] = {-1, -1, -1};
  static thread_local int val = 1;
  const int64_t heads = (int64_t)p.B * p.H;
  if (key[0] == p.nc && key[1] == heads && key[2] == slots) return val;
  double best = 1e300;
  int bestL = p.nc;
  for (int L = 1; L <= p.nc; L++) {
    const int64_t nseg = (p.nc + L - 1) / L;
    if (nseg > 4096 || heads * nseg > (int64_t)1 << 30) continue;
    const int64_t waves = (heads * nseg + slots - 1) / slots;
    const double cost = (double)waves * (L + 2.0);
    if (cost < best - 1e-9) {
      best = cost;
      bestL = L;
    }
  }
  key[0] = p.nc; key[1] = heads; key[2] = slots;
  val = bestL;
  return bestL;
}

// Shape validation (the pages' checks in their order, then this build's
// envelope) and the launch plan: tile sizes, p-slices, segment length.
static mmbf_status plan(const mmbf_dims* dims, int64_t C, int64_t div, int reduced, int has_z,
                        int want_y, Params* out) {
  if (!dims) return fail(MMBF_ERR_ARG, "dims is NULL");
  const int64_t B = dims->B, S = dims->S, H = dims->H, G = dims->G, R = dims->R, N = dims->N,
                P = dims->P;
  if (B < 1 || S < 1 || R < 1 || G < 1)
    return fail(MMBF_ERR_SHAPE, "B, S, R and G must be positive");
  if (C < 1 || C * R > 128) return fail(MMBF_ERR_SHAPE, "chunk_size * R must be in [1, 128]");
  if (div != 2 && div != 4) return fail(MMBF_ERR_SHAPE, "rotary_dim_divisor must be 2 or 4");
  if (N < 1 || N % div || N % 2)
    return fail(MMBF_ERR_SHAPE, "N must be even and divisible by rotary_dim_divisor");
  if (N > 128) return fail(MMBF_ERR_SHAPE, "N greater than 128 is not supported");
  if (H < 1 || P < 1) return fail(MMBF_ERR_SHAPE, "H and P must be positive");
  if (H % G) return fail(MMBF_ERR_SHAPE, "H must be divisible by G");
  if (P > 128) return fail(MMBF_ERR_SHAPE, "P greater than 128 is not supported");
  if (R > 16) return fail(MMBF_ERR_UNSUPPORTED, "R > 16 is outside this build's envelope");
  if (S > (int64_t)1 << 30 || B * H > 65535)
    return fail(MMBF_ERR_UNSUPPORTED, "S > 2^30 or B*H > 65535 is outside this build's envelope");
  Params p;
  memset(&p, 0, sizeof p);
  p.B = (int)B; p.S = (int)S; p.H = (int)H; p.G = (int)G; p.R = (int)R; p.N = (int)N;
  p.P = (int)P; p.C = (int)C; p.div = (int)div;
  p.w = p.N / p.div;
  p.half = p.N / 2;
  p.nc = (int)((S + C - 1) / C);
  p.CR = (int)(C * R);
  p.MP = round16(p.CR);
  p.NP = round16(p.N);
  p.reduced = reduced ? 1 : 0;
  p.has_z = has_z ? 1 : 0;
  p.vec_p = (P % 2 == 0);
  int PS = std::min(round16(p.P), 64);
  while (PS > 16 && out_smem_bytes(p, PS) > kSmemLimit) PS /= 2;
  if (out_smem_bytes(p, PS) > kSmemLimit)
    return fail(MMBF_ERR_UNSUPPORTED, "tile does not fit in shared memory");
  p.PS = PS;
  p.npslice = (p.P + PS - 1) / PS;
  const int64_t per_seg = (int64_t)B * H * p.npslice;
  int nseg = (int)std::min<int64_t>(p.nc, std::max<int64_t>(1, (kTargetCtas + per_seg - 1) / per_seg));
  p.L = (p.nc + nseg - 1) / nseg;
  p.nseg = (p.nc + p.L - 1) / p.L;
  p.UA = 1;
  p.LA = p.L;
  p.nunit = p.nseg;
  p.want_y = want_y ? 1 : 0;
  p.fast = fast_index(p);
  // the warp-specialised tensor-core output kernel: R4 C16 N=P=64, reduced
  // dout (mimo_o given), without the forward output y
  p.tc = (p.fast == 0 && p.reduced && !p.want_y) ? 1 : 0;
  p.fused = 0;
  if (p.fast >= 0) {
    p.L = fast_segment_length(p, fast_slots(p));
    if (p.tc) {
      // the single-kernel form: one wave of one CTA per SM (every CTA resident
      // at once), the shortest segments that allow it
      const int64_t per_head = kPlanSms / ((int64_t)p.B * p.H);
      if (per_head >= 1) {
        const int64_t L1 = (p.nc + per_head - 1) / per_head;
        if (L1 <= tc::TCfg<4>::LMAX) p.L = (int)L1;
      }
    }
    p.nseg = (p.nc + p.L - 1) / p.L;
    // The state-sum kernel works on units of about L/UA chunks, the UA units
    // of a segment one thread-block cluster: more CTAs in flight, shorter
    // chains.  UA minimises (waves x (chunks per unit + setup)) over the
    // resident state CTAs; clusters of more than two CTAs measured slower
    // (co-scheduling of the whole cluster leaves slots idle).
    // Only the sums of segments 0 .. nseg-2 are computed: no segment reads
    // the last one's.
    const int64_t heads = (int64_t)p.B * p.H;
    const int64_t sslots = fast_state_slots(p);
    const int64_t nsum = std::max(1, p.nseg - 1);
    int ua = 1;
    double best = 1e300;
    // (the tensor-core output kernel runs one long segment per SM: its state
    // units come in clusters of up to eight)
    for (int u = 1; u <= std::min(p.tc ? 8 : 2, p.L); u++) {
      const int la = (p.L + u - 1) / u;
      const int64_t ctas = heads * nsum * ((p.L + la - 1) / la);
      const double cost = (double)((ctas + sslots - 1) / sslots) * (la + 2.0);
      if (cost < best - 1e-9) {
        best = cost;
        ua = u;
      }
    }
    p.LA = (p.L + ua - 1) / ua;
    p.UA = (p.L + p.LA - 1) / p.LA;
    p.nunit = p.nseg * p.UA;
    // single-kernel form: every CTA resident at once (one per SM) and the
    // segment's token scalars in shared memory
    p.fused = (p.tc && (int64_t)p.B * p.H * p.nseg <= kPlanSms && p.L <= tc::TCfg<4>::LMAX) ? 1 : 0;
  }
  *out = p;
  return MMBF_OK;
}

// Workspace: per (b,h) and segment, the FP32 [N][P] state sum, the decay
// product and the [2][R][P] gradient partials.  Sized for the larger of the
// generic and the specialised plan, so one size serves both.
static int ws_units(const Params& p) {
  int n = std::max(p.nunit, p.nseg);
  const int64_t per_seg = (int64_t)p.B * p.H * p.npslice;
  const int ng = (int)std::min<int64_t>(p.nc, std::max<int64_t>(1, (kTargetCtas + per_seg - 1) / per_seg));
  const int Lg = (p.nc + ng - 1) / ng;
  return std::max(n, (p.nc + Lg - 1) / Lg);
}
// Workspace header: the device error word (first 4 bytes of 256).
constexpr size_t kWsHeader = 256;

static size_t workspace_bytes_of(const Params& p) {
  const int n = ws_units(p);
  const size_t st = align16((size_t)p.B * p.H * n * p.N * p.P * 4);
  const size_t dec = align16((size_t)p.B * p.H * n * 4);
  const size_t gr = align16((size_t)p.B * p.H * n * 2 * p.R * p.P * 4);
  const size_t cnt = align16((size_t)p.B * p.H * 4);
  const size_t flg = align16((size_t)p.B * p.H * n * 4);
  return kWsHeader + st + dec + gr + cnt + flg + 256;
}

// ---- tensor maps of the TMA kernels (cuTensorMapEncodeTiled through the
// runtime's driver entry point; no link against the driver library)
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  });
  return fn;
}
// dims[0] innermost; strides[i] (bytes) of dims[i+1]; box[rank].
static bool encode_map(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box, bool swizzle128) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint32_t ones[5] = {1, 1, 1, 1, 1};
  return enc(m, type, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, ones,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// The maps the TMA stage loads read (layouts as in Params); false if any
// cannot be encoded (the call then takes the generic kernels).
template <class K>
static bool encode_stage_maps(Params& p) {
  if (!K::TMA) return true;
  const cuuint64_t B = p.B, S = p.S, H = p.H, G = p.G, R = p.R, N = p.N, P = p.P, W = p.w;
  const cuuint32_t C = (cuuint32_t)K::C, Rb = (cuuint32_t)K::R;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  {  // q, k [B,S,R,G,N]
    const cuuint64_t d[5] = {N, G, R, S, B};
    const cuuint64_t st[4] = {N * 2, G * N * 2, R * G * N * 2, S * R * G * N * 2};
    const cuuint32_t box[5] = {(cuuint32_t)N, 1, Rb, C, 1};
    if (!encode_map(&p.tm_q, bf, 5, p.q, d, st, box, true)) return false;
    if (!encode_map(&p.tm_k, bf, 5, p.k, d, st, box, true)) return false;
  }
  {  // v, z, reduced dout [B,S,H,P]
    const cuuint64_t d[4] = {P, H, S, B};
    const cuuint64_t st[3] = {P * 2, H * P * 2, S * H * P * 2};
    const cuuint32_t box[4] = {(cuuint32_t)P, 1, C, 1};
    if (!encode_map(&p.tm_v, bf, 4, p.v, d, st, box, true)) return false;
    if (p.has_z && !encode_map(&p.tm_z, bf, 4, p.z, d, st, box, true)) return false;
    if (p.has_z && !encode_map(&p.tm_dz, bf, 4, p.dz, d, st, box, true)) return false;
    if (p.dout && p.reduced && !encode_map(&p.tm_dout, bf, 4, p.dout, d, st, box, true)) return false;
    if (p.want_y && p.reduced && !encode_map(&p.tm_y, bf, 4, p.y, d, st, box, true)) return false;
  }
  if (p.dout && !p.reduced) {  // per-rank dout [B,S,R,H,P]
    const cuuint64_t d[5] = {P, H, R, S, B};
    const cuuint64_t st[4] = {P * 2, H * P * 2, R * H * P * 2, S * R * H * P * 2};
    const cuuint32_t box[5] = {(cuuint32_t)P, 1, Rb, C, 1};
    if (!encode_map(&p.tm_dout, bf, 5, p.dout, d, st, box, true)) return false;
    if (p.want_y && !encode_map(&p.tm_y, bf, 5, p.y, d, st, box, true)) return false;
  }
  {  // states [B,H,nc,N,P] as rows of P
    const cuuint64_t d[2] = {P, (cuuint64_t)p.B * p.H * p.nc * N};
    const cuuint64_t st[1] = {P * 2};
    const cuuint32_t box[2] = {(cuuint32_t)P, (cuuint32_t)N};
    if (!encode_map(&p.tm_states, bf, 2, p.states, d, st, box, true)) return false;
  }
  {  // angles [B,S,H,W] fp32
    const cuuint64_t d[4] = {W, H, S, B};
    const cuuint64_t st[3] = {W * 4, H * W * 4, S * H * W * 4};
    const cuuint32_t box[4] = {(cuuint32_t)W, 1, C, 1};
    if (!encode_map(&p.tm_ang, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.angles, d, st, box, false)) return false;
  }
  return true;
}

template <int RMAX>
static cudaError_t launch_output(const Params& p, size_t smem, cudaStream_t s) {
  static int cached = 48 * 1024;
  auto kern = chunk_output_kernel<RMAX>;
  cudaError_t e = ensure_smem(kern, smem, &cached);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.npslice, p.nseg, p.B * p.H), kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

// Launch with programmatic dependent launch (the kernel waits with
// griddepcontrol.wait before it reads its predecessor's results).
// cluster_y > 1 groups consecutive blockIdx.y into thread-block clusters.
template <typename Kern>
static cudaError_t launch_ex(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                             const Params& p, int cluster_y = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    n++;
  }
  if (cluster_y > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = (unsigned)cluster_y;
    attr[n].val.clusterDim.z = 1;
    n++;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// State-sum units launched: those of segments 0 .. nseg-2 (the last segment's
// sum is read by no one); with one segment, one cluster that only resets the
// gradient counter.
static int state_units(const Params& p) { return std::max(1, p.nseg - 1) * p.UA; }

static bool aligned16(const void* x) { return x == nullptr || (reinterpret_cast<uintptr_t>(x) & 15) == 0; }

template <class K>
static cudaError_t launch_fast(const Params& p, cudaStream_t st, int* launches) {
  const size_t ss = fast_state_smem<K>(p), so = fast_out_smem<K>(p);
  // All branches on (the benchmarked combination), without and with the
  // forward output y, have their own instantiations with the branches
  // resolved at compile time; other combinations read them at run time.
  const int mode = (p.reduced && p.has_z && p.has_d) ? (p.want_y ? 15 : 7) : -1;
  cudaError_t e = ensure_smem(fast::state_kernel<StateCfg<K>>, ss, &fast_state_smem_set<K>());
  if (e == cudaSuccess)
    e = mode == 7    ? ensure_smem(fast::output_kernel<K, 7>, so, &fast_out_smem_set<K, 7>())
        : mode == 15 ? ensure_smem(fast::output_kernel<K, 15>, so, &fast_out_smem_set<K, 15>())
                     : ensure_smem(fast::output_kernel<K, -1>, so, &fast_out_smem_set<K, -1>());
  if (e != cudaSuccess) return e;
  g_stage_names = kFastStageNames;
  g_stage_names_n = 3;
  g_failed_stage = 0;
  stage_event(0, 0, st);
  // the UA units of a segment form one cluster (UA <= 8)
  e = launch_ex(fast::state_kernel<StateCfg<K>>, dim3(p.B * p.H, state_units(p)), dim3(StateCfg<K>::NT), ss,
                st, false, p, p.UA);
  stage_event(0, 1, st);
  (*launches)++;
  if (e != cudaSuccess) return e;
  // exclusive prefix over the segment sums: the state entering each segment
  g_failed_stage = 1;
  stage_event(1, 0, st);
  e = launch_ex(segment_prefix_fast_kernel, dim3((unsigned)((p.N * p.P + 127) / 128), p.B * p.H), dim3(128), 0,
                st, true, p);
  stage_event(1, 1, st);
  (*launches)++;
  if (e != cudaSuccess) return e;
  g_failed_stage = 2;
  stage_event(2, 0, st);
  const dim3 og(p.B * p.H, p.nseg);
  e = mode == 7    ? launch_ex(fast::output_kernel<K, 7>, og, dim3(K::NT), so, st, true, p)
      : mode == 15 ? launch_ex(fast::output_kernel<K, 15>, og, dim3(K::NT), so, st, true, p)
                   : launch_ex(fast::output_kernel<K, -1>, og, dim3(K::NT), so, st, true, p);
  stage_event(2, 1, st);
  (*launches)++;
  return e;  // the output kernel's last CTA per (b,h) also sums the dmimo partials
}

// Device-side evaluation of the specialised kernels' approximate math next to
// CUDA's accurate functions (mamba_mimo_probe_fast_math).
__global__ void probe_fast_math_kernel(int which, const float* x, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float v = x[i];
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  if (which == 0) {
    fast::sincos_fast(v, &r.x, &r.y);
    r.z = sinf(v);
    r.w = cosf(v);
  } else if (which == 1) {
    r.x = fast::exp_fast(v);
    r.z = expf(v);
  } else {
    r.x = fast::rcp_approx(fast::ex2_approx(v * -fast::kLog2e) + 1.f);
    r.z = 1.f / (1.f + expf(-v));
  }
  reinterpret_cast<float4*>(out)[i] = r;
}

// The timed shape family with reduced dout: the state-sum kernel (clusters of
// up to eight units per segment), then the warp-specialised tensor-core output
// kernel, which folds the earlier segments' sums itself (no prefix kernel).
template <int MODE>
static int& tc_smem_set() {
  static int v[kMaxDevices + 1];
  const int d = device_slot();
  if (d == kMaxDevices) v[d] = 0;
  return v[d];
}
static cudaError_t launch_tc(Params& p, cudaStream_t st, int* launches) {
  using T = tc::TCfg<4>;
  using KS = StateCfg<FastA>;
  const size_t ss = fast_state_smem<FastA>(p);
  const int mode = (p.has_z && p.has_d) ? 7 : -1;
  cudaError_t e = mode == 7 ? ensure_smem(tc::out_kernel<T, 7>, T::SMEM, &tc_smem_set<7>())
                            : ensure_smem(tc::out_kernel<T, -1>, T::SMEM, &tc_smem_set<-1>());
  if (e != cudaSuccess) return e;
  if (p.fused && !(p.test_flags & 2)) {
    // single kernel, all CTAs resident at once (they wait for their head's
    // earlier segments); a device that cannot hold the grid takes the two-
    // kernel form below
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B * p.H, p.nseg);
    cfg.blockDim = dim3(T::NT);
    cfg.dynamicSmemBytes = T::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    g_stage_names = kTcFusedStageNames;
    g_stage_names_n = 1;
    g_failed_stage = 0;
    stage_event(0, 0, st);
    e = mode == 7 ? cudaLaunchKernelEx(&cfg, tc::out_kernel<T, 7>, p) : cudaLaunchKernelEx(&cfg, tc::out_kernel<T, -1>, p);
    stage_event(0, 1, st);
    if (e == cudaSuccess) {
      (*launches)++;
      return e;
    }
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    cudaGetLastError();
    g_fused_refused = (int)e;
  }
  p.fused = 0;
  e = ensure_smem(fast::state_kernel<KS>, ss, &fast_state_smem_set<FastA>());
  if (e != cudaSuccess) return e;
  g_stage_names = kTcStageNames;
  g_stage_names_n = 2;
  g_failed_stage = 0;
  stage_event(0, 0, st);
  e = launch_ex(fast::state_kernel<KS>, dim3(p.B * p.H, state_units(p)), dim3(KS::NT), ss, st, false, p, p.UA);
  stage_event(0, 1, st);
  (*launches)++;
  if (e != cudaSuccess) return e;
  g_failed_stage = 1;
  stage_event(1, 0, st);
  const dim3 og(p.B * p.H, p.nseg);
  e = mode == 7 ? launch_ex(tc::out_kernel<T, 7>, og, dim3(T::NT), T::SMEM, st, true, p)
                : launch_ex(tc::out_kernel<T, -1>, og, dim3(T::NT), T::SMEM, st, true, p);
  stage_event(1, 1, st);
  (*launches)++;
  return e;
}

// Built-in scratch area of mamba_mimo_bwd_fwd_fixed_scratch: a file-scope
// device array (every GPU that loads the library holds it until exit).  Host
// code must not use the name as an address; the device address is looked up
// with the device current, once per device and CUDA context: a context torn
// down and created again (cudaDeviceReset) maps the array at a new address,
// so the cached address is kept with the context it belongs to and looked up
// again when the current context differs.
static __device__ __align__(256) unsigned char g_fixed_scratch[MAMBA_MIMO_FIXED_SCRATCH_BYTES];
static std::mutex g_fixed_scratch_mu;
struct FixedScratchSlot {
  CUcontext ctx;
  void* addr;
};
static FixedScratchSlot g_fixed_scratch_slot[256];

// The calling thread's current CUDA context (NULL if none is current yet or
// the driver entry point is unavailable); no stream work, no allocation.
static CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(f);
    else
      cudaGetLastError();
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

static mmbf_status fixed_scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MMBF_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 256) return fail(MMBF_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
  FixedScratchSlot& slot = g_fixed_scratch_slot[dev];
  const CUcontext ctx = current_context();
  if (!slot.addr || !ctx || slot.ctx != ctx) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_fixed_scratch);
    if (e != cudaSuccess || addr == nullptr)
      return fail(MMBF_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch area: %s",
                  cudaGetErrorString(e));
    slot.addr = addr;
    slot.ctx = current_context();  // the symbol lookup made the device's context current
  }
  *out = slot.addr;
  return MMBF_OK;
}

}  // namespace mmbf

using namespace mmbf;

extern "C" {

mmbf_status mamba_mimo_bwd_fwd_workspace_size(const mmbf_dims* dims, int64_t chunk_size,
                                              int64_t rotary_dim_divisor, int reduced_dout,
                                              int has_z, size_t* bytes) {
  // one size serves the op with and without the forward output y (their
  // plans may differ)
  size_t need = 0;
  for (int want_y = 0; want_y < 2; want_y++) {
    Params p;
    mmbf_status s = plan(dims, chunk_size, rotary_dim_divisor, reduced_dout, has_z, want_y, &p);
    if (s != MMBF_OK) return s;
    need = std::max(need, workspace_bytes_of(p));
  }
  if (!bytes) return fail(MMBF_ERR_ARG, "bytes is NULL");
  *bytes = need;
  return MMBF_OK;
}

}  // extern "C"

// The op, with the optional forward output y (NULL: not computed).
static mmbf_status run_op(const mmbf_dims* dims, const void* dout, const void* q, const void* k,
                          const void* v, const float* q_bias, const float* k_bias,
                          const float* mimo_v, const float* mimo_o, const void* z,
                          const float* mimo_z, const float* angles, const float* da_cs,
                          const float* da_cs_rev, const float* dt, const void* trap, const float* d,
                          const float* segsum, int64_t chunk_size, int64_t rotary_dim_divisor,
                          float* dmimo_o, void* states, void* dz, float* dmimo_z, void* qk_dot,
                          void* y, void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = '\0';
  Params p;
  mmbf_status s = plan(dims, chunk_size, rotary_dim_divisor, mimo_o != nullptr, z != nullptr, y != nullptr, &p);
  if (s != MMBF_OK) return s;
  if (!dout || !q || !k || !v || !q_bias || !k_bias || !mimo_v || !angles || !da_cs ||
      !da_cs_rev || !dt || !trap || !segsum)
    return fail(MMBF_ERR_ARG, "a required input pointer is NULL");
  if (!states || !qk_dot) return fail(MMBF_ERR_ARG, "states and qk_dot must not be NULL");
  if ((z == nullptr) != (mimo_z == nullptr))
    return fail(MMBF_ERR_ARG, z ? "mimo_z is required when z is present"
                                : "mimo_z must be None when z is None");
  if ((mimo_o == nullptr) != (dmimo_o == nullptr))
    return fail(MMBF_ERR_ARG, "dmimo_o must be given exactly when mimo_o is given");
  if ((z == nullptr) != (dz == nullptr) || (z == nullptr) != (dmimo_z == nullptr))
    return fail(MMBF_ERR_ARG, "dz and dmimo_z must be given exactly when z is given");
  const void* ptrs[] = {dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs,
                        da_cs_rev, dt, trap, d, segsum, dmimo_o, states, dz, dmimo_z, qk_dot, y};
  for (const void* x : ptrs)
    if (x && (reinterpret_cast<uintptr_t>(x) & 3))
      return fail(MMBF_ERR_ALIGN, "tensor pointers must be 4-byte aligned");
  size_t need = 0;
  s = mamba_mimo_bwd_fwd_workspace_size(dims, chunk_size, rotary_dim_divisor, mimo_o != nullptr, z != nullptr,
                                        &need);
  if (s != MMBF_OK) return s;
  if (!workspace || workspace_bytes < need)
    return fail(MMBF_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return fail(MMBF_ERR_ALIGN, "workspace must be 256-byte aligned");

  p.has_d = d != nullptr;
  p.y = static_cast<uint16_t*>(y);
  p.dout = static_cast<const uint16_t*>(dout);
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.z = static_cast<const uint16_t*>(z);
  p.trap = static_cast<const uint16_t*>(trap);
  p.q_bias = q_bias; p.k_bias = k_bias; p.mimo_v = mimo_v; p.mimo_o = mimo_o; p.mimo_z = mimo_z;
  p.angles = angles; p.da_cs = da_cs; p.da_cs_rev = da_cs_rev; p.dt = dt; p.d = d;
  p.segsum = segsum;
  p.dmimo_o = dmimo_o; p.dmimo_z = dmimo_z;
  p.states = static_cast<uint16_t*>(states);
  p.dz = static_cast<uint16_t*>(dz);
  p.qk_dot = static_cast<uint16_t*>(qk_dot);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const int wsn = ws_units(p);
  p.ws_err = reinterpret_cast<unsigned int*>(ws);
  ws += kWsHeader;
  p.ws_state = reinterpret_cast<float*>(ws);
  ws += align16((size_t)p.B * p.H * wsn * p.N * p.P * 4);
  p.ws_decay = reinterpret_cast<float*>(ws);
  ws += align16((size_t)p.B * p.H * wsn * 4);
  p.ws_grad = reinterpret_cast<float*>(ws);
  ws += align16((size_t)p.B * p.H * wsn * 2 * p.R * p.P * 4);
  p.ws_count = reinterpret_cast<unsigned int*>(ws);
  ws += align16((size_t)p.B * p.H * 4);
  p.ws_flag = reinterpret_cast<unsigned int*>(ws);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int launches = 0;
  cudaError_t e;
  cudaGetLastError();  // a stale error from elsewhere must not be reported as ours
  p.tag = next_call_tag();
  p.test_flags = g_test_flags;
  g_last_tag = p.tag;
  g_last_err_word = p.ws_err;
  bool fast_ok = p.fast >= 0 && aligned16(q) && aligned16(k) && aligned16(v) && aligned16(dout) &&
                 aligned16(z) && aligned16(angles) && aligned16(segsum) && aligned16(states) && aligned16(dz);
  if (fast_ok) {
    switch (p.fast) {
      case 0: fast_ok = encode_stage_maps<FastA>(p); break;
      case 1: fast_ok = encode_stage_maps<FastB>(p); break;
      case 2: fast_ok = encode_stage_maps<FastC>(p); break;
      default: fast_ok = encode_stage_maps<FastD>(p); break;
    }
  }
  if (fast_ok) {
    if (p.tc) {
      e = launch_tc(p, st, &launches);  // (clears p.fused if it takes the two-kernel form)
    } else {
      switch (p.fast) {
        case 0: e = launch_fast<FastA>(p, st, &launches); break;
        case 1: e = launch_fast<FastB>(p, st, &launches); break;
        case 2: e = launch_fast<FastC>(p, st, &launches); break;
        default: e = launch_fast<FastD>(p, st, &launches); break;
      }
    }
    if (e == cudaSuccess && g_stage_error != cudaSuccess) {
      e = g_stage_error;
      g_stage_error = cudaSuccess;
    }
    g_variant = p.tc ? 3 : (p.fast == 3 ? 4 : p.fast);  // (the wide-state family reports 4)
    g_plan[0] = p.L; g_plan[1] = p.nseg; g_plan[2] = p.UA; g_plan[3] = p.LA; g_plan[4] = fast_slots(p);
    g_plan[5] = p.fused;
    g_plan[6] = g_fused_refused;
    g_fused_refused = 0;
    if (e != cudaSuccess)
      return fail(MMBF_ERR_CUDA, "CUDA error in %s (fast %d, grid %d x %d/%d): %s",
                  g_failed_stage >= 0 ? g_stage_names[g_failed_stage] : "setup", p.fast, p.B * p.H,
                  p.nseg, p.nunit, cudaGetErrorString(e));
    g_launches = launches;
    return MMBF_OK;
  }
  // Generic kernels (any shape of the envelope).  Their segmentation is the
  // generic one, one state unit per segment.
  g_stage_names = kStageNames;
  g_stage_names_n = 4;
  {
    const int64_t per_seg = (int64_t)p.B * p.H * p.npslice;
    const int ng = (int)std::min<int64_t>(p.nc, std::max<int64_t>(1, (kTargetCtas + per_seg - 1) / per_seg));
    p.L = (p.nc + ng - 1) / ng;
    p.nseg = (p.nc + p.L - 1) / p.L;
    p.UA = 1;
    p.LA = p.L;
    p.nunit = p.nseg;
  }
  {
    static int cached = 48 * 1024;
    const size_t smem = state_layout(p).total;
    e = ensure_smem(segment_state_kernel, smem, &cached);
    if (e == cudaSuccess) {
      stage_event(0, 0, st);
      segment_state_kernel<<<dim3(p.npslice, p.nseg, p.B * p.H), kThreads, smem, st>>>(p);
      e = cudaGetLastError();
      stage_event(0, 1, st);
      launches++;
    }
  }
  if (e == cudaSuccess) {
    stage_event(1, 0, st);
    if ((p.N * p.P) % 4 == 0)
      segment_prefix_vec_kernel<4><<<dim3((p.N * p.P / 4 + 127) / 128, p.B * p.H), 128, 0, st>>>(p);
    else
      segment_prefix_vec_kernel<1><<<dim3((p.N * p.P + 127) / 128, p.B * p.H), 128, 0, st>>>(p);
    e = cudaGetLastError();
    stage_event(1, 1, st);
    launches++;
  }
  if (e == cudaSuccess) {
    const size_t smem = out_layout(p).total;
    stage_event(2, 0, st);
    if (p.R <= 4)
      e = launch_output<4>(p, smem, st);
    else if (p.R <= 8)
      e = launch_output<8>(p, smem, st);
    else
      e = launch_output<16>(p, smem, st);
    stage_event(2, 1, st);
    launches++;
  }
  if (e == cudaSuccess && (p.reduced || p.has_z)) {
    stage_event(3, 0, st);
    grad_reduce_kernel<<<p.B * p.H, 256, 0, st>>>(p);
    e = cudaGetLastError();
    stage_event(3, 1, st);
    launches++;
  }
  if (e == cudaSuccess && g_stage_error != cudaSuccess) {
    e = g_stage_error;
    g_stage_error = cudaSuccess;
  }
  if (e != cudaSuccess)
    return fail(MMBF_ERR_CUDA,
                "CUDA error in generic kernel %d (fast=%d, grid %d/%d/%d, smem state %zu out %zu): %s",
                launches, p.fast, p.npslice, p.nseg, p.B * p.H, state_layout(p).total,
                out_layout(p).total, cudaGetErrorString(e));
  g_launches = launches;
  g_variant = -1;
  g_plan[0] = p.L; g_plan[1] = p.nseg; g_plan[2] = 1; g_plan[3] = p.L; g_plan[4] = 0; g_plan[5] = 0; g_plan[6] = 0;
  return MMBF_OK;
}

extern "C" {

mmbf_status mamba_mimo_bwd_fwd(const mmbf_dims* dims, const void* dout, const void* q,
                               const void* k, const void* v, const float* q_bias,
                               const float* k_bias, const float* mimo_v, const float* mimo_o,
                               const void* z, const float* mimo_z, const float* angles,
                               const float* da_cs, const float* da_cs_rev, const float* dt,
                               const void* trap, const float* d, const float* segsum,
                               int64_t chunk_size, int64_t rotary_dim_divisor, float* dmimo_o,
                               void* states, void* dz, float* dmimo_z, void* qk_dot,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return run_op(dims, dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs,
                da_cs_rev, dt, trap, d, segsum, chunk_size, rotary_dim_divisor, dmimo_o, states, dz,
                dmimo_z, qk_dot, nullptr, workspace, workspace_bytes, stream);
}

mmbf_status mamba_mimo_bwd_fwd_y(const mmbf_dims* dims, const void* dout, const void* q,
                                 const void* k, const void* v, const float* q_bias,
                                 const float* k_bias, const float* mimo_v, const float* mimo_o,
                                 const void* z, const float* mimo_z, const float* angles,
                                 const float* da_cs, const float* da_cs_rev, const float* dt,
                                 const void* trap, const float* d, const float* segsum,
                                 int64_t chunk_size, int64_t rotary_dim_divisor, float* dmimo_o,
                                 void* states, void* dz, float* dmimo_z, void* qk_dot, void* y,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!y) {
    g_err[0] = '\0';
    return fail(MMBF_ERR_ARG, "y must not be NULL");
  }
  return run_op(dims, dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs,
                da_cs_rev, dt, trap, d, segsum, chunk_size, rotary_dim_divisor, dmimo_o, states, dz,
                dmimo_z, qk_dot, y, workspace, workspace_bytes, stream);
}

mmbf_status mamba_mimo_bwd_fwd_fixed_scratch(
    const mmbf_dims* dims, const void* dout, const void* q, const void* k, const void* v,
    const float* q_bias, const float* k_bias, const float* mimo_v, const float* mimo_o,
    const void* z, const float* mimo_z, const float* angles, const float* da_cs,
    const float* da_cs_rev, const float* dt, const void* trap, const float* d,
    const float* segsum, int64_t chunk_size, int64_t rotary_dim_divisor, float* dmimo_o,
    void* states, void* dz, float* dmimo_z, void* qk_dot, void* stream) {
  g_err[0] = '\0';
  size_t need = 0;
  mmbf_status s = mamba_mimo_bwd_fwd_workspace_size(dims, chunk_size, rotary_dim_divisor,
                                                    mimo_o != nullptr, z != nullptr, &need);
  if (s != MMBF_OK) return s;
  if (need > MAMBA_MIMO_FIXED_SCRATCH_BYTES)
    return fail(MMBF_ERR_WORKSPACE,
                "this problem needs %zu bytes of workspace; the built-in scratch area holds %zu "
                "(use mamba_mimo_bwd_fwd with a caller-provided workspace)",
                need, (size_t)MAMBA_MIMO_FIXED_SCRATCH_BYTES);
  void* scratch = nullptr;
  s = fixed_scratch_address(&scratch);
  if (s != MMBF_OK) return s;
  return mamba_mimo_bwd_fwd(dims, dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles,
                            da_cs, da_cs_rev, dt, trap, d, segsum, chunk_size, rotary_dim_divisor,
                            dmimo_o, states, dz, dmimo_z, qk_dot, scratch,
                            (size_t)MAMBA_MIMO_FIXED_SCRATCH_BYTES, stream);
}

const char* mamba_mimo_last_error(void) { return g_err; }
int mamba_mimo_abi_version(void) { return MAMBA_MIMO_BWD_FWD_ABI_VERSION; }
int mamba_mimo_last_launch_count(void) { return g_launches; }
int mamba_mimo_last_kernel_variant(void) { return g_variant; }

void mamba_mimo_set_test_hooks(int flags) { g_test_flags = flags; }

mmbf_status mamba_mimo_probe_fast_math(int which, const float* x, float* out, int n, void* stream) {
  g_err[0] = '\0';
  if (which < 0 || which > 2) return fail(MMBF_ERR_ARG, "which must be 0, 1 or 2");
  if (n < 0 || (n > 0 && (!x || !out))) return fail(MMBF_ERR_ARG, "x and out must be device pointers, n >= 0");
  if (n == 0) return MMBF_OK;
  if (reinterpret_cast<uintptr_t>(out) & 15) return fail(MMBF_ERR_ALIGN, "out must be 16-byte aligned");
  probe_fast_math_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(which, x, out, n);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MMBF_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return MMBF_OK;
}

mmbf_status mamba_mimo_device_status(void* stream) {
  if (!g_last_err_word) return MMBF_OK;
  unsigned int w = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&w, g_last_err_word, sizeof w, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(MMBF_ERR_CUDA, "reading the device status: %s", cudaGetErrorString(e));
  if ((w >> 8) == g_last_tag && (w & 0xffu) != 0)
    return fail(MMBF_ERR_DEVICE_TIMEOUT, "a kernel of the last call stopped: a bounded wait ran out (code %u: %s)",
                w & 0xffu,
                (w & 0xffu) == 5u ? "the look-back on an earlier segment's published sum" : "a shared-memory barrier");
  return MMBF_OK;
}

int mamba_mimo_last_plan(int* out, int n) {
  if (!out || n < 0) return 0;
  const int k = n < 7 ? n : 7;
  for (int i = 0; i < k; i++) out[i] = g_plan[i];
  return k;
}

void mamba_mimo_set_stage_events(void* const* events, int count) {
  g_stage_events = (events && count > 0) ? events : nullptr;
  g_stage_count = g_stage_events ? count : 0;
}

const char* mamba_mimo_stage_name(int i) {
  return (i >= 0 && i < g_stage_names_n) ? g_stage_names[i] : nullptr;
}

}  // extern "C"

// The second backward stage (its own kernels and C entry points).
#include "mmbb.cuh"
