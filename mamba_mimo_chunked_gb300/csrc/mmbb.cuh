// Second backward stage of the Mamba-3 MIMO chunked scan (mamba_mimo_bwd_bwd):
// the reverse scan over chunks and its 12 gradients.  Definition: the page
// "MindSpeed-Ops PR #100" (op document "mamba3_mimo_bwd_bwd 算子迁移说明" for
// the interface, dPhiO and PsiV; practice document, sections "输入缓存的语义"
// for the state and dstates recurrences and the caches, "非整 chunk" for the
// padding of a partial last chunk); each output is the exact derivative of
// L = sum dPhiO * out of the first stage's chunk output (readings in
// include/mamba_mimo_bwd_bwd.h).
//
// Four launches per call:
//   seed_kernel   (chunk, b*h)  G_c = sum_i exp(da_cs[t_i]) q_rot[i]^T dPhiO[i]
//                               and the chunk decay alpha_c = exp(da_cs[last]);
//   scan_kernel   (N*P slice, b*h)  D_c = alpha_c D_{c+1} + G_c in reverse
//                               chunk order; chunk c's slot then holds
//                               D_{c+1}, the gradient of the state leaving it;
//   grad_kernel   (chunk, b*h)  every gradient of the chunk from its inputs,
//                               the state entering it (the states cache) and
//                               D_{c+1}: 9 products of FP32 tiles on the
//                               tensor cores (TF32, three passes per FP32
//                               product).  N, P, C*R <= 64: tiles in shared
//                               memory, one chunk per CTA; larger shapes:
//                               grad_kernel_wide, a persistent grid whose
//                               tiles sit in a per-CTA slice of the workspace;
//   reduce_kernel (b*h)         DMIMO_V and DD: the chunks' partial sums in a
//                               fixed order.
// The kernels that read activations are instantiated per activation dtype
// (FP32, BF16, FP16) and per shape policy: run-time extents, or compile-time
// extents for BF16 on N = P = 64, R = 4, C = 16 (shifts instead of the
// divisions that split flat element indices).
// FP32-level accuracy throughout, deterministic (no floating-point atomics).

#include <cuda_fp16.h>

#include "mamba_mimo_bwd_bwd.h"

namespace mmbf {
namespace bb {

struct BBParams {
  int B, S, H, G, R, N, P, C, w, nc, CR, reduced, has_d;
  int act;   // dtype of dout, q, k, v, states, qk_dot, trap: kF32, kBF16 or kF16
  int dqkv;  // dtype of DQ, DK, DV (same codes)
  const void *dout, *q, *k, *v, *states, *qk, *trap;
  const float *q_bias, *k_bias, *mimo_v, *mimo_o, *d, *da_cs, *da_cs_rev, *dt, *segsum, *angles;
  void *DQ, *DK, *DV;  // in the dtype dqkv selects
  float *DMIMO_V, *DANGLES, *DFACTOR, *DGAMMA, *DDA, *DSSDA, *DDA_CS_REV, *DDA_CS, *DD;
  float* ws_D;      // [BH][nc][N][P]: seeds G_c, then D_{c+1}
  float* ws_alpha;  // [BH][nc]
  float* ws_mv;     // [BH][nc][R][P]: DMIMO_V partials
  float* ws_dd;     // [BH][nc]: DD partials
  // wide path (N, P or C*R above 64): tiles in a per-CTA FP32 scratch
  int wide;
  int LN, LP, LC, CR16, N16;  // tile strides (extents rounded up to 16) and padded row counts
  int sLN, sLP;               // seed kernel strides (N, P rounded up to 64)
  int64_t m1sz, m2sz, scr_floats;
  float* ws_scr;              // [grid][scr_floats]
};

constexpr int kT = 256;             // threads per CTA of the seed and reduce kernels' thread groups
constexpr int kTG = 512;            // threads per CTA of the gradient kernel (16 warps, 16 x 16 output tiles)
constexpr int kMax = 64;            // N, P and C*R limit of the 64-wide path (tiles in shared memory)
constexpr int kLD = kMax + 4;       // FP32 tile row stride: 4 (mod 32) puts the 32 lanes of every m16n8k8 fragment load on distinct banks
constexpr int kTile = kMax * kLD;   // floats per tile
constexpr int kSmall = 4224;        // segsum [C][C], qk [C][R][R], dqk (C*R <= 64, R <= 16)
constexpr int kMaxW = 128;          // wide path: C*R and P limit (N up to 2 * kMaxW)
constexpr int kSmallW = 16640;      // segsum, qk, dqk for C*R <= 128, R <= 16
constexpr int kWideGrid = 152;      // persistent CTAs of the wide gradient kernel
constexpr int kRedCols = 16;        // per-row partial sums, one per column block

// dtype codes of the ABI (dqkv_dtype / act_dtype)
constexpr int kF32 = 0, kBF16 = 1, kF16 = 2;

__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }
// Element i of an activation tensor of dtype code A, widened to FP32 (exact
// for all three).  The kernels that read activations are instantiated per A.
template <int A>
__device__ __forceinline__ float ld_act(const void* base, int64_t i) {
  if constexpr (A == kBF16) return bf_f(static_cast<const uint16_t*>(base)[i]);
  else if constexpr (A == kF16) return __half2float(static_cast<const __half*>(base)[i]);
  else return static_cast<const float*>(base)[i];
}
// Element i of DQ / DK / DV in the requested dtype (FP32, or BF16 / FP16
// rounded to nearest even).
__device__ __forceinline__ void store_dqkv(void* base, int64_t i, float x, int dt) {
  if (dt == kBF16)
    static_cast<uint16_t*>(base)[i] = f_bf(x);
  else if (dt == kF16)
    static_cast<__half*>(base)[i] = __float2half_rn(x);
  else
    static_cast<float*>(base)[i] = x;
}

// acc[u][v] += sum_k a(i0+u, k) * b(k, j0+v): a 4 x 4 block of a product of
// shared-memory tiles (rows and columns past the operands' extents are
// computed on whatever the tile holds there and never used).
template <int TM, int TN, class FA, class FB>
__device__ __forceinline__ void mm4(float (&acc)[TM][TN], int i0, int j0, int K, FA a, FB b) {
#pragma unroll 4
  for (int kk = 0; kk < K; kk++) {
    float av[TM], bv[TN];
#pragma unroll
    for (int u = 0; u < TM; u++) av[u] = a(i0 + u, kk);
#pragma unroll
    for (int v = 0; v < TN; v++) bv[v] = b(kk, j0 + v);
#pragma unroll
    for (int u = 0; u < TM; u++)
#pragma unroll
      for (int v = 0; v < TN; v++) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
  }
}
// FP32 products on the tensor cores with FP32-level accuracy: each operand
// x = hi + lo + e with hi = x truncated to TF32 (the low 13 mantissa bits
// cleared), lo = (x - hi) truncated the same way (x - hi is exact), so
// |e| < 2^-20 |x|; a b = hi_a hi_b + hi_a lo_b + lo_a hi_b, whose error
// (the dropped lo_a lo_b and the two truncations) is below 3 * 2^-20
// relative; FP32 accumulation.  Bit operations only (finite inputs).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  constexpr uint32_t kTf32 = 0xffffe000u;
  hi = __float_as_uint(x) & kTf32;
  lo = __float_as_uint(x - __uint_as_float(hi)) & kTf32;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// acc += a b over k < K for this warp's 16 x 16 output tile at (r0, c0):
// m16n8k8 fragments (A: rows g, g+8 at k = c, c+4; B: column g at k = c,
// c+4; accumulator nb: rows g, g+8, columns nb*8 + 2c, +1; g = lane / 4,
// c = lane % 4).  k past K reads as zero.
// BEXACT: every b value is exactly a TF32 number (a widened BF16 or FP16
// value), so b needs no split and a b = hi_a b + lo_a b takes two products.
template <bool BEXACT = false, class FA, class FB>
__device__ __forceinline__ void mm_tc(float (&acc)[2][4], int r0, int c0, int K, FA a, FB b) {
  const int lane = threadIdx.x & 31, g = lane >> 2, cq = lane & 3;
  for (int k0 = 0; k0 < K; k0 += 8) {
    const int ka = k0 + cq, kb = ka + 4;
    const bool va = ka < K, vb = kb < K;
    float af[4];
    af[0] = va ? a(r0 + g, ka) : 0.f;
    af[1] = va ? a(r0 + g + 8, ka) : 0.f;
    af[2] = vb ? a(r0 + g, kb) : 0.f;
    af[3] = vb ? a(r0 + g + 8, kb) : 0.f;
    uint32_t ah[4], al[4];
#pragma unroll
    for (int q = 0; q < 4; q++) split_tf32(af[q], ah[q], al[q]);
#pragma unroll
    for (int nb = 0; nb < 2; nb++) {
      if constexpr (BEXACT) {
        const uint32_t b0 = __float_as_uint(va ? b(ka, c0 + nb * 8 + g) : 0.f);
        const uint32_t b1 = __float_as_uint(vb ? b(kb, c0 + nb * 8 + g) : 0.f);
        mma_tf32(acc[nb], al, b0, b1);
        mma_tf32(acc[nb], ah, b0, b1);
      } else {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(va ? b(ka, c0 + nb * 8 + g) : 0.f, bh0, bl0);
        split_tf32(vb ? b(kb, c0 + nb * 8 + g) : 0.f, bh1, bl1);
        mma_tf32(acc[nb], ah, bl0, bl1);
        mma_tf32(acc[nb], al, bh0, bh1);
        mma_tf32(acc[nb], ah, bh0, bh1);
      }
    }
  }
}
__device__ __forceinline__ void zero_tc(float (&acc)[2][4]) {
#pragma unroll
  for (int nb = 0; nb < 2; nb++) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
}
// Row and column of element e of accumulator nb of this lane's fragments.
#define TC_ROW(r0, e) ((r0) + ((threadIdx.x & 31) >> 2) + 8 * ((e) >> 1))
#define TC_COL(c0, nb, e) ((c0) + (nb) * 8 + 2 * (threadIdx.x & 3) + ((e) & 1))
// Per-row sums of this warp's tile: each lane adds its values of rows g and
// g+8 (rs[0], rs[1]); the four lanes of a row group combine, and lane c = 0
// writes the tile's partial to red[row * kRedCols + wc].
__device__ __forceinline__ void tc_row_sums(float (&rs)[2], float* red, int r0, int wc) {
#pragma unroll
  for (int h2 = 0; h2 < 2; h2++) {
    rs[h2] += __shfl_xor_sync(0xffffffffu, rs[h2], 1);
    rs[h2] += __shfl_xor_sync(0xffffffffu, rs[h2], 2);
  }
  if ((threadIdx.x & 3) == 0) {
    const int g = (threadIdx.x & 31) >> 2;
    red[(r0 + g) * kRedCols + wc] = rs[0];
    red[(r0 + g + 8) * kRedCols + wc] = rs[1];
  }
}
template <int TM, int TN>
__device__ __forceinline__ void zero4(float (&acc)[TM][TN]) {
#pragma unroll
  for (int u = 0; u < TM; u++)
#pragma unroll
    for (int v = 0; v < TN; v++) acc[u][v] = 0.f;
}

// Problem extents, read from the parameters (ShapeRT) or fixed at compile
// time for one shape (ShapeCT: the divisions and remainders of the element
// loops by them become shifts and masks).
struct ShapeRT {
  static constexpr bool kVec = false;  // element-wise loads
  static __device__ __forceinline__ int N(const BBParams& p) { return p.N; }
  static __device__ __forceinline__ int P(const BBParams& p) { return p.P; }
  static __device__ __forceinline__ int R(const BBParams& p) { return p.R; }
  static __device__ __forceinline__ int C(const BBParams& p) { return p.C; }
  static __device__ __forceinline__ int CR(const BBParams& p) { return p.CR; }
  static __device__ __forceinline__ int w(const BBParams& p) { return p.w; }
};
template <int N_, int P_, int R_, int C_, int W_, bool VEC_>
struct ShapeCT {
  // VEC_: BF16 activations with every activation, bias and mimo pointer
  // 16-byte aligned; rows of 8 elements move with one 16-byte load
  static constexpr bool kVec = VEC_;
  static_assert(!VEC_ || (N_ % 8 == 0 && P_ % 8 == 0), "vector loads take rows of 8 elements");
  static __device__ __forceinline__ int N(const BBParams&) { return N_; }
  static __device__ __forceinline__ int P(const BBParams&) { return P_; }
  static __device__ __forceinline__ int R(const BBParams&) { return R_; }
  static __device__ __forceinline__ int C(const BBParams&) { return C_; }
  static __device__ __forceinline__ int CR(const BBParams&) { return C_ * R_; }
  static __device__ __forceinline__ int w(const BBParams&) { return W_; }
  static bool matches(const BBParams& p) { return p.N == N_ && p.P == P_ && p.R == R_ && p.C == C_ && p.w == W_; }
};
// the shape with its own instantiation: N = P = 64, R = 4, C = 16, rotary
// width 16, BF16 activations on 16-byte aligned pointers
using ShapeFast = ShapeCT<64, 64, 4, 16, 16, true>;

// 8 BF16 values at element i of `base` (16-byte aligned) widened to FP32, and
// 8 FP32 values to / from 16-byte aligned memory.
__device__ __forceinline__ void ld8_bf16(const void* base, int64_t i, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; q++) {
    f[2 * q] = bf_lo(w[q]);
    f[2 * q + 1] = bf_hi(w[q]);
  }
}
__device__ __forceinline__ void ld8_f32(const float* base, int64_t i, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(base + i), b = *reinterpret_cast<const float4*>(base + i + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void st8_f32(float* dst, const float (&f)[8]) {
  *reinterpret_cast<float4*>(dst) = make_float4(f[0], f[1], f[2], f[3]);
  *reinterpret_cast<float4*>(dst + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

// Token scalars of chunk c (reading of the op header): gamma, factor,
// exp(da_cs), exp(da_cs_rev), and whether the token is inside S.
template <int A, class SH, int NT>
__device__ __forceinline__ void load_tokens(const BBParams& p, int bh, int c, float* gam, float* fac, float* ea, float* er,
                            float* valid) {
  #pragma unroll
  for (int t = threadIdx.x; t < SH::C(p); t += NT) {
    const int tg = c * SH::C(p) + t;
    const int64_t i = (int64_t)bh * p.S + tg;
    const bool in = tg < p.S, in1 = tg + 1 < p.S;
    const float dtv = in ? p.dt[i] : 0.f, trv = in ? ld_act<A>(p.trap, i) : 0.f;
    const float dtn = in1 ? p.dt[i + 1] : 0.f, trn = in1 ? ld_act<A>(p.trap, i + 1) : 0.f;
    const float g = dtv * sigm(trv);
    gam[t] = g;
    fac[t] = g + dtn * sigm(-trn);  // 0 shifted part past S and at the last padded position
    ea[t] = expf(in ? p.da_cs[i] : 0.f);
    er[t] = expf(in ? p.da_cs_rev[i] : 0.f);
    valid[t] = in ? 1.f : 0.f;
  }
}

// Biased rows of q (or k) of chunk c, then the rotary on the pairs (m, N/2+m),
// m < w, in place: rows j = t*R + r of a [C*R][N] tile (zero input past S,
// plus the bias, as the padded reference).
template <int A, class SH, int NT>
__device__ __forceinline__ void load_rotated(const BBParams& p, int b, int h, int c, const void* src, const float* bias,
                             float* T, int ld) {
  const int g = h / (p.H / p.G);
  if constexpr (SH::kVec) {  // 8 consecutive n of one row per step
#pragma unroll
    for (int e8 = threadIdx.x; e8 < SH::CR(p) * SH::N(p) / 8; e8 += NT) {
      const int e = e8 * 8, j = e / SH::N(p), n = e % SH::N(p), t = j / SH::R(p), r = j % SH::R(p),
                tg = c * SH::C(p) + t;
      float x[8], y[8];
      ld8_f32(bias, ((int64_t)h * SH::R(p) + r) * SH::N(p) + n, x);
      if (tg < p.S) {
        ld8_bf16(src, ((((int64_t)b * p.S + tg) * SH::R(p) + r) * p.G + g) * SH::N(p) + n, y);
#pragma unroll
        for (int q = 0; q < 8; q++) x[q] += y[q];
      }
      st8_f32(T + j * ld + n, x);
    }
  } else {
#pragma unroll
    for (int e = threadIdx.x; e < SH::CR(p) * SH::N(p); e += NT) {
      const int j = e / SH::N(p), n = e % SH::N(p), t = j / SH::R(p), r = j % SH::R(p), tg = c * SH::C(p) + t;
      float x = bias[((int64_t)h * SH::R(p) + r) * SH::N(p) + n];
      if (tg < p.S) x += ld_act<A>(src, ((((int64_t)b * p.S + tg) * SH::R(p) + r) * p.G + g) * SH::N(p) + n);
      T[j * ld + n] = x;
    }
  }
  __syncthreads();
  const int half = SH::N(p) / 2;
  // one angle per (token, pair), applied to the token's R rank rows
  #pragma unroll
  for (int e = threadIdx.x; e < SH::C(p) * SH::w(p); e += NT) {
    const int t = e / SH::w(p), m = e % SH::w(p), tg = c * SH::C(p) + t;
    const float th = tg < p.S ? p.angles[(((int64_t)b * p.S + tg) * p.H + h) * SH::w(p) + m] : 0.f;
    float sn, cs;
    sincosf(th, &sn, &cs);
    for (int r = 0; r < SH::R(p); r++) {
      const int j = t * SH::R(p) + r;
      const float lo = T[j * ld + m], hi = T[j * ld + half + m];
      T[j * ld + m] = cs * lo - sn * hi;
      T[j * ld + half + m] = sn * lo + cs * hi;
    }
  }
}

// dPhiO rows [C*R][P] (zero past S) [op document: reduce-O or per rank].
template <int A, class SH, int NT>
__device__ __forceinline__ void load_dphio(const BBParams& p, int b, int h, int c, float* T, int ld) {
  if constexpr (SH::kVec) {  // 8 consecutive p of one row per step
#pragma unroll
    for (int e8 = threadIdx.x; e8 < SH::CR(p) * SH::P(p) / 8; e8 += NT) {
      const int e = e8 * 8, j = e / SH::P(p), pp = e % SH::P(p), t = j / SH::R(p), r = j % SH::R(p),
                tg = c * SH::C(p) + t;
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (tg < p.S) {
        if (p.reduced) {
          float m[8];
          ld8_bf16(p.dout, (((int64_t)b * p.S + tg) * p.H + h) * SH::P(p) + pp, x);
          ld8_f32(p.mimo_o, ((int64_t)h * SH::R(p) + r) * SH::P(p) + pp, m);
#pragma unroll
          for (int q = 0; q < 8; q++) x[q] *= m[q];
        } else {
          ld8_bf16(p.dout, ((((int64_t)b * p.S + tg) * SH::R(p) + r) * p.H + h) * SH::P(p) + pp, x);
        }
      }
      st8_f32(T + j * ld + pp, x);
    }
  } else {
#pragma unroll
    for (int e = threadIdx.x; e < SH::CR(p) * SH::P(p); e += NT) {
      const int j = e / SH::P(p), pp = e % SH::P(p), t = j / SH::R(p), r = j % SH::R(p), tg = c * SH::C(p) + t;
      float x = 0.f;
      if (tg < p.S) {
        if (p.reduced)
          x = ld_act<A>(p.dout, (((int64_t)b * p.S + tg) * p.H + h) * SH::P(p) + pp) * p.mimo_o[((int64_t)h * SH::R(p) + r) * SH::P(p) + pp];
        else
          x = ld_act<A>(p.dout, ((((int64_t)b * p.S + tg) * SH::R(p) + r) * p.H + h) * SH::P(p) + pp);
      }
      T[j * ld + pp] = x;
    }
  }
}

// PsiV rows [C*R][P] = v[t,p] * mimo_v[r,p] (zero past S).
template <int A, class SH, int NT>
__device__ __forceinline__ void load_psi(const BBParams& p, int b, int h, int c, float* T, int ld) {
  if constexpr (SH::kVec) {  // 8 consecutive p of one row per step
#pragma unroll
    for (int e8 = threadIdx.x; e8 < SH::CR(p) * SH::P(p) / 8; e8 += NT) {
      const int e = e8 * 8, j = e / SH::P(p), pp = e % SH::P(p), t = j / SH::R(p), r = j % SH::R(p),
                tg = c * SH::C(p) + t;
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (tg < p.S) {
        float m[8];
        ld8_bf16(p.v, (((int64_t)b * p.S + tg) * p.H + h) * SH::P(p) + pp, x);
        ld8_f32(p.mimo_v, ((int64_t)h * SH::R(p) + r) * SH::P(p) + pp, m);
#pragma unroll
        for (int q = 0; q < 8; q++) x[q] *= m[q];
      }
      st8_f32(T + j * ld + pp, x);
    }
  } else {
#pragma unroll
    for (int e = threadIdx.x; e < SH::CR(p) * SH::P(p); e += NT) {
      const int j = e / SH::P(p), pp = e % SH::P(p), t = j / SH::R(p), r = j % SH::R(p), tg = c * SH::C(p) + t;
      float x = 0.f;
      if (tg < p.S)
        x = ld_act<A>(p.v, (((int64_t)b * p.S + tg) * p.H + h) * SH::P(p) + pp) * p.mimo_v[((int64_t)h * SH::R(p) + r) * SH::P(p) + pp];
      T[j * ld + pp] = x;
    }
  }
}

// ---- 1. seeds: G_c[n][p] = sum_i exp(da_cs[t_i]) q_rot[i][n] dPhiO[i][p]
// The 64-wide path (W = false) keeps [64][kLD] tiles and one 64 x 64 output
// block; the wide path strides its rows by N and P rounded up to 64 (every
// 4 x 4 read of a block stays inside its row) and walks the output blocks.
template <int A, bool W, class SH>
__global__ void __launch_bounds__(kT, W ? 1 : 4) seed_kernel(const BBParams p) {  // 64-wide: 4 CTAs per SM
  extern __shared__ float smf[];
  const int LN = W ? p.sLN : kLD, LP = W ? p.sLP : kLD, rows = W ? SH::CR(p) : kMax, TC = W ? kMaxW : kMax;
  float* Qr = smf;
  float* Gp = Qr + rows * LN;
  float* tk = Gp + rows * LP;  // gam, fac, ea, er, valid: 5 x TC
  float* ear = tk + 5 * TC;    // exp(da_cs) per row j = t*R + r
  const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  load_tokens<A, SH, kT>(p, bh, c, tk, tk + TC, tk + 2 * TC, tk + 3 * TC, tk + 4 * TC);
  load_dphio<A, SH, kT>(p, b, h, c, Gp, LP);
  load_rotated<A, SH, kT>(p, b, h, c, p.q, p.q_bias, Qr, LN);
  __syncthreads();
  const float* ea = tk + 2 * TC;
  for (int j = threadIdx.x; j < SH::CR(p); j += blockDim.x) ear[j] = ea[j / SH::R(p)];
  __syncthreads();
  float* dst = p.ws_D + ((int64_t)bh * p.nc + c) * SH::N(p) * SH::P(p);
  if constexpr (!W) {  // the 64 x 64 block as 16 x 16 tiles on the tensor cores, two per warp
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int t = warp; t < 16; t += kT / 32) {
      const int r0 = (t >> 2) * 16, c0 = (t & 3) * 16;
      float acc[2][4];
      zero_tc(acc);
      mm_tc(acc, r0, c0, SH::CR(p), [=](int n, int i) { return Qr[i * LN + n] * ear[i]; },
            [=](int i, int pp) { return Gp[i * LP + pp]; });
#pragma unroll
      for (int nb = 0; nb < 2; nb++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int n = TC_ROW(r0, e), pp = TC_COL(c0, nb, e);
          if (n < SH::N(p) && pp < SH::P(p)) dst[n * SH::P(p) + pp] = acc[nb][e];
        }
    }
  } else {  // FP32 FMAs, 4 x 4 outputs per thread, over the 64 x 64 output blocks
    for (int n0 = 0; n0 < SH::N(p); n0 += 64)
      for (int p0 = 0; p0 < SH::P(p); p0 += 64) {
        const int i0 = n0 + (threadIdx.x >> 4) * 4, j0 = p0 + (threadIdx.x & 15) * 4;
        float acc[4][4];
        zero4(acc);
        mm4(acc, i0, j0, SH::CR(p), [=](int n, int i) { return Qr[i * LN + n] * ear[i]; },
            [=](int i, int pp) { return Gp[i * LP + pp]; });
#pragma unroll
        for (int u = 0; u < 4; u++)
#pragma unroll
          for (int v = 0; v < 4; v++)
            if (i0 + u < SH::N(p) && j0 + v < SH::P(p)) dst[(i0 + u) * SH::P(p) + j0 + v] = acc[u][v];
      }
  }
  if (threadIdx.x == 0) {
    const int last = min(c * SH::C(p) + SH::C(p), p.S) - 1;
    p.ws_alpha[(int64_t)bh * p.nc + c] = expf(p.da_cs[(int64_t)bh * p.S + last]);
  }
}

// ---- 2. reverse scan, one state element per thread: slot c becomes D_{c+1}
__global__ void __launch_bounds__(128) scan_kernel(const BBParams p) {
  const int bh = blockIdx.y;
  const int64_t NP = (int64_t)p.N * p.P;
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= NP) return;
  float* base = p.ws_D + (int64_t)bh * p.nc * NP + e;
  const float* al = p.ws_alpha + (int64_t)bh * p.nc;
  constexpr int GRP = 32;  // chunks whose loads are in flight at once
  float acc = 0.f;
  for (int c1 = p.nc - 1; c1 >= 0; c1 -= GRP) {
    float x[GRP], a[GRP];
#pragma unroll
    for (int q = 0; q < GRP; q++) {
      const int c = c1 - q;
      x[q] = c >= 0 ? base[(int64_t)c * NP] : 0.f;
      a[q] = c >= 0 ? al[c] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < GRP; q++) {
      const int c = c1 - q;
      if (c >= 0) {
        base[(int64_t)c * NP] = acc;
        acc = fmaf(a[q], acc, x[q]);
      }
    }
  }
}

// ---- 3. every gradient of one chunk
// This warp's 16 x 16 output tiles of a rows x cols product, f(r0, c0, tile
// column): on the 64-wide path one tile of the 4 x 4 grid per warp (16
// warps), on the wide path a strided walk over the grid.
template <bool W, class F>
__device__ __forceinline__ void for_tiles(int rows, int cols, F f) {
  const int wid = threadIdx.x >> 5;
  if constexpr (!W) {
    f((wid >> 2) * 16, (wid & 3) * 16, wid & 3);
  } else {
    const int nr = (rows + 15) >> 4, ncol = (cols + 15) >> 4;
    for (int t = wid; t < nr * ncol; t += kTG / 32) f((t / ncol) * 16, (t % ncol) * 16, t % ncol);
  }
}

// Tiles: on the 64-wide path eleven [64][kLD] FP32 tiles in shared memory;
// on the wide path the same tiles in this CTA's global scratch (rows padded
// to 16 and strides rounded up to 16, so that every fragment read of a
// 16 x 16 tile stays inside its tile), the small tables in shared memory.
template <int A, bool WIDE, class SH>
__device__ __forceinline__ void grad_chunk(const BBParams& p, int c, int bh, float* smf, float* scr) {
  const int LN = WIDE ? p.LN : kLD, LP = WIDE ? p.LP : kLD, LC = WIDE ? p.LC : kLD;
  const int TC = WIDE ? kMaxW : kMax;
  float *Qr, *Kr, *Ps, *Gp, *Hc, *Dn, *M1, *M2, *dQ, *dK, *dP, *sm;
  if constexpr (!WIDE) {
    Qr = smf;              // rotated q rows
    Kr = Qr + kTile;       // rotated k rows
    Ps = Kr + kTile;       // PsiV
    Gp = Ps + kTile;       // dPhiO
    Hc = Gp + kTile;       // state entering the chunk [N][P]
    Dn = Hc + kTile;       // gradient of the state leaving it [N][P]
    M1 = Dn + kTile;       // A, then (kept) for the segsum gradient
    M2 = M1 + kTile;       // dA, then dS
    dQ = M2 + kTile;       // gradient of q_rot
    dK = dQ + kTile;       // gradient of k_scaled
    dP = dK + kTile;       // gradient of PsiV
    sm = dP + kTile;       // segsum [C][C] | qk [C][R][R] | dqk [C][R][R]
  } else {
    const int64_t tq = (int64_t)p.CR16 * LN, tp = (int64_t)p.CR16 * LP, th = (int64_t)p.N16 * LP;
    Qr = scr;
    Kr = Qr + tq;
    dQ = Kr + tq;
    dK = dQ + tq;
    Ps = dK + tq;
    Gp = Ps + tp;
    dP = Gp + tp;
    Hc = dP + tp;
    Dn = Hc + th;
    M1 = Dn + th;
    M2 = M1 + p.m1sz;
    sm = smf;
  }
  float* tk = sm + (WIDE ? kSmallW : kSmall);  // gam | fac | ea | er | valid, TC each
  float* red = tk + 5 * TC;                 // three [TC][kRedCols] row-partial buffers
  float* red2 = red + TC * kRedCols;
  float* red3 = red2 + TC * kRedCols;
  float* wsum = red3 + TC * kRedCols;       // [2][kTG / 32] per-warp sums
  float* facr = wsum + 2 * (kTG / 32);      // factor, exp(da_cs), exp(da_cs_rev) per row j = t*R + r
  float* ear = facr + TC;
  float* err = ear + TC;
  float* gam = tk;
  float* fac = tk + TC;
  float* ea = tk + 2 * TC;
  float* er = tk + 3 * TC;
  float* valid = tk + 4 * TC;
  const int C = SH::C(p), R = SH::R(p), N = SH::N(p), P = SH::P(p), CR = SH::CR(p);
  float* seg = sm;  // exp(segsum) below the diagonal, 0 elsewhere
  float* qk = sm + C * C;
  float* dqk = qk + C * R * R;
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x;
  // column tiles of the N-wide and P-wide row sums
  const int ctn = WIDE ? (N + 15) >> 4 : 4, ctp = WIDE ? (P + 15) >> 4 : 4;

  // ---- inputs of the chunk
  load_tokens<A, SH, kTG>(p, bh, c, gam, fac, ea, er, valid);
  #pragma unroll
  for (int e = tid; e < C * C; e += kTG) {  // exp(segsum) below the diagonal, once per chunk
    const float x = p.segsum[((int64_t)bh * p.nc + c) * C * C + e];
    seg[e] = (e / C > e % C) ? expf(x) : 0.f;
  }
  #pragma unroll
  for (int e = tid; e < C * R * R; e += kTG) {
    const int tg = c * C + e / (R * R);
    qk[e] = tg < p.S ? ld_act<A>(p.qk, ((int64_t)bh * p.S + tg) * R * R + e % (R * R)) : 0.f;
  }
  if constexpr (SH::kVec) {  // 8 consecutive p of one state row per step
#pragma unroll
    for (int e8 = tid; e8 < N * P / 8; e8 += kTG) {
      const int e = e8 * 8;
      float x[8];
      ld8_bf16(p.states, ((int64_t)bh * p.nc + c) * N * P + e, x);
      st8_f32(Hc + (e / P) * LP + e % P, x);
      ld8_f32(p.ws_D, ((int64_t)bh * p.nc + c) * N * P + e, x);
      st8_f32(Dn + (e / P) * LP + e % P, x);
    }
  } else {
#pragma unroll
    for (int e = tid; e < N * P; e += kTG) {
      Hc[(e / P) * LP + e % P] = ld_act<A>(p.states, ((int64_t)bh * p.nc + c) * N * P + e);
      Dn[(e / P) * LP + e % P] = p.ws_D[((int64_t)bh * p.nc + c) * N * P + e];
    }
  }
  load_psi<A, SH, kTG>(p, b, h, c, Ps, LP);
  load_dphio<A, SH, kTG>(p, b, h, c, Gp, LP);
  load_rotated<A, SH, kTG>(p, b, h, c, p.q, p.q_bias, Qr, LN);
  load_rotated<A, SH, kTG>(p, b, h, c, p.k, p.k_bias, Kr, LN);
  __syncthreads();
  for (int j = tid; j < CR; j += kTG) {
    facr[j] = fac[j / R];
    ear[j] = ea[j / R];
    err[j] = er[j / R];
  }
  __syncthreads();

  // ---- A = mask(q_rot k_scaled^T) exp(segsum): selected, never multiplied by
  //      a mask (padded rows and the upper triangle never reach a product)
  auto tok_ok = [=](int i, int j) { return (i / R) > (j / R) && valid[i / R] != 0.f; };
  for_tiles<WIDE>(CR, CR, [&](int fr0, int fc0, int) {
    float acc[2][4];
    zero_tc(acc);
    mm_tc(acc, fr0, fc0, N, [=](int i, int n) { return Qr[i * LN + n]; }, [=](int n, int j) { return Kr[j * LN + n]; });
#pragma unroll
    for (int nb = 0; nb < 2; nb++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int i = TC_ROW(fr0, e), j = TC_COL(fc0, nb, e);
        if (i < CR && j < CR)
          M1[i * LC + j] = tok_ok(i, j) ? acc[nb][e] * facr[j] * seg[(i / R) * C + j / R] : 0.f;
      }
  });
  __syncthreads();

  // ---- dPsiV = A^T dPhiO + k_state D_{c+1} + d dPhiO + gamma qk^T dPhiO (diagonal);
  //      dA = dPhiO PsiV^T
  const float dv = p.has_d ? p.d[h] : 0.f;
  for_tiles<WIDE>(CR, P, [&](int fr0, int fc0, int) {
    float acc[2][4], acc2[2][4];
    zero_tc(acc);
    mm_tc(acc, fr0, fc0, CR, [=](int j, int i) { return M1[i * LC + j]; }, [=](int i, int pp) { return Gp[i * LP + pp]; });
    zero_tc(acc2);
    mm_tc(acc2, fr0, fc0, N, [=](int j, int n) { return Kr[j * LN + n]; }, [=](int n, int pp) { return Dn[n * LP + pp]; });
#pragma unroll
    for (int nb = 0; nb < 2; nb++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int j = TC_ROW(fr0, e), pp = TC_COL(fc0, nb, e);
        if (j < CR && pp < P) {
          const int t = j / R, r = j % R;
          float x = acc[nb][e] + acc2[nb][e] * facr[j] * err[j] + dv * Gp[j * LP + pp];
          float dg = 0.f;
          for (int o = 0; o < R; o++) dg = fmaf(qk[(t * R + o) * R + r], Gp[(t * R + o) * LP + pp], dg);
          dP[j * LP + pp] = fmaf(gam[t], dg, x);
        }
      }
  });
  for_tiles<WIDE>(CR, CR, [&](int fr0, int fc0, int) {
    float acc[2][4];
    zero_tc(acc);
    mm_tc(acc, fr0, fc0, P, [=](int i, int pp) { return Gp[i * LP + pp]; }, [=](int pp, int j) { return Ps[j * LP + pp]; });
#pragma unroll
    for (int nb = 0; nb < 2; nb++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int i = TC_ROW(fr0, e), j = TC_COL(fc0, nb, e);
        if (i < CR && j < CR) M2[i * LC + j] = acc[nb][e];
      }
  });
  __syncthreads();

  // ---- DSSDA[ti][tj] = sum over the token pair's rank pairs of dA * A
  #pragma unroll
  for (int e = tid; e < C * C; e += kTG) {
    const int ti = e / C, tj = e % C;
    float s = 0.f;
    if (ti > tj && valid[ti] != 0.f)
      for (int o = 0; o < R; o++)
        for (int r = 0; r < R; r++) s = fmaf(M2[(ti * R + o) * LC + tj * R + r], M1[(ti * R + o) * LC + tj * R + r], s);
    p.DSSDA[((int64_t)bh * p.nc + c) * C * C + e] = (valid[tj] != 0.f) ? s : 0.f;
  }
  __syncthreads();
  // dS = dA exp(segsum) on the causal entries (in place)
  #pragma unroll
  for (int e = tid; e < CR * CR; e += kTG) {
    const int i = e / CR, j = e % CR;
    M2[i * LC + j] = tok_ok(i, j) ? M2[i * LC + j] * seg[(i / R) * C + j / R] : 0.f;
  }
  __syncthreads();

  // ---- dq_rot = dS k_scaled + exp(da_cs) dPhiO Hc^T;
  //      dk_scaled = dS^T q_rot + exp(da_cs_rev) dk_state, dk_state = PsiV Dn^T;
  //      row sums for DDA_CS_REV (dk_state * k_state), DFACTOR (dk_scaled *
  //      k_rot) and DDA_CS (inter * dPhiO)
  for_tiles<WIDE>(CR, N, [&](int fr0, int fc0, int) {
    float acc[2][4], acc2[2][4];
    zero_tc(acc);
    mm_tc(acc, fr0, fc0, CR, [=](int i, int j) { return M2[i * LC + j] * facr[j]; },
          [=](int j, int n) { return Kr[j * LN + n]; });
    zero_tc(acc2);
    // Hc holds widened BF16 / FP16 cache values: exact TF32 operands
    mm_tc<A != kF32>(acc2, fr0, fc0, P, [=](int i, int pp) { return Gp[i * LP + pp]; },
                     [=](int pp, int n) { return Hc[n * LP + pp]; });
#pragma unroll
    for (int nb = 0; nb < 2; nb++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int i = TC_ROW(fr0, e), n = TC_COL(fc0, nb, e);
        if (i < CR && n < N) dQ[i * LN + n] = fmaf(ear[i], acc2[nb][e], acc[nb][e]);
      }
  });
  for_tiles<WIDE>(CR, N, [&](int fr0, int fc0, int wc) {
    float acc[2][4], acc2[2][4];
    zero_tc(acc);
    mm_tc(acc, fr0, fc0, P, [=](int j, int pp) { return Ps[j * LP + pp]; }, [=](int pp, int n) { return Dn[n * LP + pp]; });
    zero_tc(acc2);
    mm_tc(acc2, fr0, fc0, CR, [=](int j, int i) { return M2[i * LC + j]; }, [=](int i, int n) { return Qr[i * LN + n]; });
    float r1[2] = {0.f, 0.f}, r2[2] = {0.f, 0.f};
#pragma unroll
    for (int nb = 0; nb < 2; nb++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int j = TC_ROW(fr0, e), n = TC_COL(fc0, nb, e);
        if (j < CR && n < N) {
          const float kr = Kr[j * LN + n];
          r1[e >> 1] = fmaf(acc[nb][e], kr * facr[j] * err[j], r1[e >> 1]);
          const float dks = fmaf(err[j], acc[nb][e], acc2[nb][e]);
          r2[e >> 1] = fmaf(dks, kr, r2[e >> 1]);
          dK[j * LN + n] = dks;
        }
      }
    tc_row_sums(r1, red, fr0, wc);
    tc_row_sums(r2, red2, fr0, wc);
  });
  // inter = exp(da_cs) q_rot Hc
  for_tiles<WIDE>(CR, P, [&](int fr0, int fc0, int wc) {
    float acc[2][4];
    zero_tc(acc);
    mm_tc<A != kF32>(acc, fr0, fc0, N, [=](int i, int n) { return Qr[i * LN + n]; },
                     [=](int n, int pp) { return Hc[n * LP + pp]; });
    float r3[2] = {0.f, 0.f};
#pragma unroll
    for (int nb = 0; nb < 2; nb++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int i = TC_ROW(fr0, e), pp = TC_COL(fc0, nb, e);
        if (i < CR && pp < P) r3[e >> 1] = fmaf(acc[nb][e] * ear[i], Gp[i * LP + pp], r3[e >> 1]);
      }
    tc_row_sums(r3, red3, fr0, wc);
  });
  // same-token terms: dot[t,o,r] = dPhiO[(t,o)] . PsiV[(t,r)]; dqk = gamma dot,
  // DGAMMA = sum qk * dot
  #pragma unroll
  for (int e = tid; e < C * R * R; e += kTG) {
    const int t = e / (R * R), o = (e / R) % R, r = e % R;
    float s = 0.f;
    for (int pp = 0; pp < P; pp++) s = fmaf(Gp[(t * R + o) * LP + pp], Ps[(t * R + r) * LP + pp], s);
    dqk[e] = s;  // gamma applied below
  }
  // DDA (alpha_c <Hc, D_{c+1}> at the chunk's last valid token) and the DD
  // partial (sum dPhiO * PsiV): block sums in a fixed order
  {
    float s = 0.f, dd = 0.f;
    #pragma unroll
    for (int e = tid; e < N * P; e += kTG) s = fmaf(Hc[(e / P) * LP + e % P], Dn[(e / P) * LP + e % P], s);
    #pragma unroll
    for (int e = tid; e < CR * P; e += kTG) dd = fmaf(Gp[(e / P) * LP + e % P], Ps[(e / P) * LP + e % P], dd);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      dd += __shfl_xor_sync(0xffffffffu, dd, o);
    }
    if ((tid & 31) == 0) {
      wsum[tid >> 5] = s;
      wsum[kTG / 32 + (tid >> 5)] = dd;
    }
  }
  __syncthreads();
  #pragma unroll
  for (int t = tid; t < C; t += kTG) {  // per-token sums
    float s1 = 0.f, s2 = 0.f, s3 = 0.f, g = 0.f;
    for (int r = 0; r < R; r++) {  // the column tiles of the row
      for (int q = 0; q < ctn; q++) {
        s1 += red[(t * R + r) * kRedCols + q];
        s2 += red2[(t * R + r) * kRedCols + q];
      }
      for (int q = 0; q < ctp; q++) s3 += red3[(t * R + r) * kRedCols + q];
    }
    for (int e = 0; e < R * R; e++) g = fmaf(qk[t * R * R + e], dqk[t * R * R + e], g);
    const int tg = c * C + t;
    if (tg < p.S) {
      const int64_t o = (int64_t)bh * p.S + tg;
      p.DDA_CS_REV[o] = s1;
      p.DFACTOR[o] = s2;
      p.DDA_CS[o] = s3;
      p.DGAMMA[o] = g;
      float hd = 0.f;
      for (int w8 = 0; w8 < kTG / 32; w8++) hd += wsum[w8];
      p.DDA[o] = (tg == min(c * C + C, p.S) - 1) ? p.ws_alpha[(int64_t)bh * p.nc + c] * hd : 0.f;
    }
  }
  if (tid == 0) {
    float dd = 0.f;
    for (int w8 = 0; w8 < kTG / 32; w8++) dd += wsum[kTG / 32 + w8];
    p.ws_dd[(int64_t)bh * p.nc + c] = dd;
  }
  __syncthreads();
  #pragma unroll
  for (int e = tid; e < C * R * R; e += kTG) dqk[e] *= gam[e / (R * R)];

  // ---- rotary post-pass.  Stage the rotary cos / sin of the chunk and
  //      mimo_v in M1, v in M2 (both free now); DANGLES from the rotated rows.
  const int half = N / 2, W = SH::w(p);
  float* cst = M1;                // cos [C][W]
  float* snt = M1 + C * W;        // sin [C][W]
  float* mvs = M1 + 2 * C * W;    // mimo_v [R][P]
  float* vs = M2;                 // v [C][P]
  #pragma unroll
  for (int e = tid; e < C * W; e += kTG) {
    const int t = e / W, m = e % W, tg = c * C + t;
    float sn = 0.f, cs = 1.f;
    if (tg < p.S) sincosf(p.angles[(((int64_t)b * p.S + tg) * p.H + h) * W + m], &sn, &cs);
    cst[e] = cs;
    snt[e] = sn;
  }
  #pragma unroll
  for (int e = tid; e < R * P; e += kTG) mvs[e] = p.mimo_v[(int64_t)h * R * P + e];
  #pragma unroll
  for (int e = tid; e < C * P; e += kTG) {
    const int t = e / P, pp = e % P, tg = c * C + t;
    vs[e] = tg < p.S ? ld_act<A>(p.v, (((int64_t)b * p.S + tg) * p.H + h) * P + pp) : 0.f;
  }
  #pragma unroll
  for (int e = tid; e < C * W; e += kTG) {
    const int t = e / W, m = e % W, tg = c * C + t;
    if (tg >= p.S) continue;
    float s = 0.f;
    for (int r = 0; r < R; r++) {
      const int j = t * R + r;
      s += dQ[j * LN + m] * (-Qr[j * LN + half + m]) + dQ[j * LN + half + m] * Qr[j * LN + m];
      s += fac[t] * (dK[j * LN + m] * (-Kr[j * LN + half + m]) + dK[j * LN + half + m] * Kr[j * LN + m]);
    }
    p.DANGLES[(((int64_t)b * p.S + tg) * p.H + h) * W + m] = s;
  }
  __syncthreads();
  // q_rot, k_rot -> the un-rotated biased rows (transposed rotation, in place)
  #pragma unroll
  for (int e = tid; e < CR * W; e += kTG) {
    const int j = e / W, m = e % W, t = j / R;
    const float cs = cst[t * W + m], sn = snt[t * W + m];
    float lo = Qr[j * LN + m], hi = Qr[j * LN + half + m];
    Qr[j * LN + m] = cs * lo + sn * hi;
    Qr[j * LN + half + m] = -sn * lo + cs * hi;
    lo = Kr[j * LN + m];
    hi = Kr[j * LN + half + m];
    Kr[j * LN + m] = cs * lo + sn * hi;
    Kr[j * LN + half + m] = -sn * lo + cs * hi;
  }
  // DV and the DMIMO_V partial of the chunk
  #pragma unroll
  for (int e = tid; e < C * P; e += kTG) {
    const int t = e / P, pp = e % P, tg = c * C + t;
    if (tg >= p.S) continue;
    float s = 0.f;
    for (int r = 0; r < R; r++) s = fmaf(dP[(t * R + r) * LP + pp], mvs[r * P + pp], s);
    store_dqkv(p.DV, (((int64_t)b * p.S + tg) * p.H + h) * P + pp, s, p.dqkv);
  }
  #pragma unroll
  for (int e = tid; e < R * P; e += kTG) {
    const int r = e / P, pp = e % P;
    float s = 0.f;
    for (int t = 0; t < C; t++) s = fmaf(dP[(t * R + r) * LP + pp], vs[t * P + pp], s);
    p.ws_mv[((int64_t)bh * p.nc + c) * R * P + e] = s;
  }
  __syncthreads();
  // DQ / DK: the transposed rotation of the rotated-domain gradients plus the
  // diagonal's same-token terms, qk[t,o,x] = qh[(t,o)] . kh[(t,x)]
  #pragma unroll
  for (int e = tid; e < CR * N; e += kTG) {
    const int j = e / N, n = e % N, t = j / R, r = j % R, tg = c * C + t;
    if (tg >= p.S) continue;
    float dq = dQ[j * LN + n], dk = dK[j * LN + n] * fac[t];
    const int m = n < W ? n : (n >= half && n < half + W ? n - half : -1);
    if (m >= 0) {
      const float cs = cst[t * W + m], sn = snt[t * W + m];
      const float qlo = dQ[j * LN + m], qhi = dQ[j * LN + half + m];
      const float klo = dK[j * LN + m] * fac[t], khi = dK[j * LN + half + m] * fac[t];
      dq = n < W ? cs * qlo + sn * qhi : -sn * qlo + cs * qhi;
      dk = n < W ? cs * klo + sn * khi : -sn * klo + cs * khi;
    }
    for (int x = 0; x < R; x++) {
      dq = fmaf(dqk[(t * R + r) * R + x], Kr[(t * R + x) * LN + n], dq);  // row (t, o = r) of q
      dk = fmaf(dqk[(t * R + x) * R + r], Qr[(t * R + x) * LN + n], dk);  // row (t, r) of k
    }
    const int64_t o = (((int64_t)b * p.S + tg) * R + r) * p.H + h;
    store_dqkv(p.DQ, o * N + n, dq, p.dqkv);
    store_dqkv(p.DK, o * N + n, dk, p.dqkv);
  }
}

// One chunk per CTA (N, P, C*R <= 64).
template <int A, class SH>
__global__ void __launch_bounds__(kTG, 1) grad_kernel(const BBParams p) {
  extern __shared__ float smf[];
  grad_chunk<A, false, SH>(p, blockIdx.x, blockIdx.y, smf, nullptr);
}

// Wide shapes: a persistent grid walks the (b*h, chunk) items, each CTA
// reusing its own scratch.
template <int A>
__global__ void __launch_bounds__(kTG, 1) grad_kernel_wide(const BBParams p) {
  extern __shared__ float smf[];
  float* scr = p.ws_scr + (int64_t)blockIdx.x * p.scr_floats;
  const int64_t items = (int64_t)p.nc * p.B * p.H;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    grad_chunk<A, true, ShapeRT>(p, (int)(it % p.nc), (int)(it / p.nc), smf, scr);
    __syncthreads();  // every read of this item's tiles precedes the next item's loads
  }
}

// ---- 4. DMIMO_V and DD: the chunks' partials in a fixed order (each of
//      kRG thread groups sums the chunks c = g (mod kRG) in chunk order, then
//      the group sums are added in group order: deterministic)
constexpr int kRG = 4;              // thread groups of the reduce kernel
constexpr int kTR = kRG * kT;       // its threads
__global__ void __launch_bounds__(kTR) reduce_kernel(const BBParams p) {
  __shared__ float part[kRG][kT];
  __shared__ float dpart[kTR / 32];
  const int bh = blockIdx.x, grp = threadIdx.x / kT, lt = threadIdx.x % kT;
  for (int e0 = 0; e0 < p.R * p.P; e0 += kT) {
    const int e = e0 + lt;
    float s = 0.f;
    if (e < p.R * p.P) {
#pragma unroll 8
      for (int c = grp; c < p.nc; c += kRG) s += p.ws_mv[((int64_t)bh * p.nc + c) * p.R * p.P + e];
    }
    part[grp][lt] = s;
    __syncthreads();
    if (grp == 0 && e < p.R * p.P) {
      float t = part[0][lt];
#pragma unroll
      for (int g = 1; g < kRG; g++) t += part[g][lt];
      p.DMIMO_V[(int64_t)bh * p.R * p.P + e] = t;
    }
    __syncthreads();
  }
  if (p.has_d) {  // each thread a strided share of the chunks, then warp and block sums in a fixed order
    float s = 0.f;
    for (int c = threadIdx.x; c < p.nc; c += kTR) s += p.ws_dd[(int64_t)bh * p.nc + c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) dpart[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int w = 0; w < kTR / 32; w++) t += dpart[w];
      p.DD[bh] = t;
    }
  }
}

static const char* const kBBStageNames[4] = {"bb_seed", "bb_scan", "bb_grad", "bb_reduce"};

constexpr size_t kSeedSmem = (2 * kTile + 6 * kMax) * sizeof(float);
constexpr size_t kGradSmem = (11 * kTile + kSmall + 8 * kMax + 3 * kMax * kRedCols + 2 * (kTG / 32)) * sizeof(float);
// wide path: the seed tiles at their largest (C*R = 128 rows, N = 256, P = 128)
constexpr size_t kSeedSmemW = (kMaxW * 2 * kMaxW + kMaxW * kMaxW + 6 * kMaxW) * sizeof(float);
constexpr size_t kGradSmemW = (kSmallW + 8 * kMaxW + 3 * kMaxW * kRedCols + 2 * (kTG / 32)) * sizeof(float);
static size_t seed_smem_wide(const BBParams& p) {
  return ((size_t)p.CR * (p.sLN + p.sLP) + 6 * kMaxW) * sizeof(float);
}
static int grad_grid_wide(const BBParams& p) {
  return (int)std::min<int64_t>((int64_t)p.nc * p.B * p.H, kWideGrid);
}

static size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace carve-up (bytes): D, alpha, DMIMO_V partials, DD partials and,
// on the wide path, the gradient kernel's per-CTA tile scratch.
static size_t bb_workspace(const BBParams& p, size_t* off) {
  const size_t BH = (size_t)p.B * p.H, nc = (size_t)p.nc;
  size_t o = 0;
  off[0] = o; o += a256(BH * nc * p.N * p.P * 4);
  off[1] = o; o += a256(BH * nc * 4);
  off[2] = o; o += a256(BH * nc * p.R * p.P * 4);
  off[3] = o; o += a256(BH * nc * 4);
  off[4] = o; o += p.wide ? a256((size_t)grad_grid_wide(p) * p.scr_floats * 4) : 0;
  return o;
}

static mmbf_status bb_plan(const mmbf_dims* dims, int64_t chunk_size, int64_t div, BBParams* out) {
  if (!dims) return fail(MMBF_ERR_ARG, "dims is NULL");
  const mmbf_dims& d = *dims;
  if (d.B < 1 || d.S < 1 || d.H < 1 || d.G < 1 || d.R < 1 || d.N < 1 || d.P < 1 || chunk_size < 1)
    return fail(MMBF_ERR_SHAPE, "every dimension and chunk_size must be positive");
  if (d.H % d.G) return fail(MMBF_ERR_SHAPE, "H (%lld) must be a multiple of G (%lld)", (long long)d.H, (long long)d.G);
  if (div != 2 && div != 4) return fail(MMBF_ERR_SHAPE, "rotary_dim_divisor must be 2 or 4");
  if (d.N % 2 || d.N % div) return fail(MMBF_ERR_SHAPE, "N must be even and a multiple of rotary_dim_divisor");
  if (d.N > 2 * kMaxW || d.P > kMaxW || chunk_size * d.R > kMaxW || d.R > 16)
    return fail(MMBF_ERR_UNSUPPORTED, "this build of the second stage needs N <= %d, P, C*R <= %d and R <= 16",
                2 * kMaxW, kMaxW);
  if (d.S > (1 << 30) || d.B * d.H > 65535) return fail(MMBF_ERR_UNSUPPORTED, "S > 2^30 or B*H > 65535");
  BBParams p = {};
  p.B = (int)d.B; p.S = (int)d.S; p.H = (int)d.H; p.G = (int)d.G; p.R = (int)d.R; p.N = (int)d.N; p.P = (int)d.P;
  p.C = (int)chunk_size;
  p.w = (int)(d.N / div);
  p.nc = (int)((d.S + chunk_size - 1) / chunk_size);
  p.CR = p.C * p.R;
  p.wide = (p.N > kMax || p.P > kMax || p.CR > kMax) ? 1 : 0;
  if (p.wide) {
    auto up = [](int x, int m) { return (x + m - 1) / m * m; };
    p.LN = up(p.N, 16); p.LP = up(p.P, 16); p.LC = up(p.CR, 16);
    p.CR16 = p.LC; p.N16 = p.LN;
    p.sLN = up(p.N, 64); p.sLP = up(p.P, 64);
    const int64_t cc = (int64_t)p.CR16 * p.LC;
    p.m1sz = std::max<int64_t>(cc, 2 * (int64_t)p.C * p.w + (int64_t)p.R * p.P);  // A; rotary cos / sin, mimo_v
    p.m2sz = std::max<int64_t>(cc, (int64_t)p.C * p.P);                              // dA, dS; v
    auto a64 = [](int64_t x) { return (x + 63) / 64 * 64; };
    p.m1sz = a64(p.m1sz);
    p.m2sz = a64(p.m2sz);
    p.scr_floats = 4 * (int64_t)p.CR16 * p.LN + 3 * (int64_t)p.CR16 * p.LP + 2 * (int64_t)p.N16 * p.LP + p.m1sz + p.m2sz;
    p.scr_floats = a64(p.scr_floats);
  }
  *out = p;
  return MMBF_OK;
}

// The four launches of one call for activation dtype A (the kernels' shared
// memory limits are raised once per instantiation).
template <int A>
cudaError_t launch_bb(const BBParams& p, cudaStream_t st) {
  // the compile-time shape for BF16 activations on its own shape; run-time extents otherwise
  auto a16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  const bool fast = A == kBF16 && !p.wide && ShapeFast::matches(p) && a16(p.q) && a16(p.k) && a16(p.v) &&
                    a16(p.dout) && a16(p.states) && a16(p.q_bias) && a16(p.k_bias) && a16(p.mimo_v) &&
                    (!p.reduced || a16(p.mimo_o));
  using SF = ShapeFast;
  static bool smem_set[kMaxDevices + 1];  // per device: function attributes are
  const int dev = device_slot();
  if (!smem_set[dev] || dev == kMaxDevices) {
    cudaError_t e = cudaFuncSetAttribute(seed_kernel<A, false, ShapeRT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSeedSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grad_kernel<A, ShapeRT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmem);
    if constexpr (A == kBF16) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(seed_kernel<A, false, SF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSeedSmem);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(grad_kernel<A, SF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmem);
    }
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(seed_kernel<A, true, ShapeRT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSeedSmemW);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grad_kernel_wide<A>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmemW);
    if (e != cudaSuccess) return e;
    smem_set[dev] = true;
  }
  const int BH = p.B * p.H;
  g_stage_names = kBBStageNames;
  g_stage_names_n = 4;
  stage_event(0, 0, st);
  if (p.wide)
    seed_kernel<A, true, ShapeRT><<<dim3(p.nc, BH), kT, seed_smem_wide(p), st>>>(p);
  else if constexpr (A == kBF16) {
    if (fast)
      seed_kernel<A, false, SF><<<dim3(p.nc, BH), kT, kSeedSmem, st>>>(p);
    else
      seed_kernel<A, false, ShapeRT><<<dim3(p.nc, BH), kT, kSeedSmem, st>>>(p);
  } else
    seed_kernel<A, false, ShapeRT><<<dim3(p.nc, BH), kT, kSeedSmem, st>>>(p);
  stage_event(0, 1, st);
  stage_event(1, 0, st);
  scan_kernel<<<dim3((p.N * p.P + 127) / 128, BH), 128, 0, st>>>(p);
  stage_event(1, 1, st);
  stage_event(2, 0, st);
  if (p.wide)
    grad_kernel_wide<A><<<grad_grid_wide(p), kTG, kGradSmemW, st>>>(p);
  else if constexpr (A == kBF16) {
    if (fast)
      grad_kernel<A, SF><<<dim3(p.nc, BH), kTG, kGradSmem, st>>>(p);
    else
      grad_kernel<A, ShapeRT><<<dim3(p.nc, BH), kTG, kGradSmem, st>>>(p);
  } else
    grad_kernel<A, ShapeRT><<<dim3(p.nc, BH), kTG, kGradSmem, st>>>(p);
  stage_event(2, 1, st);
  stage_event(3, 0, st);
  reduce_kernel<<<BH, kTR, 0, st>>>(p);
  stage_event(3, 1, st);
  return cudaSuccess;
}

}  // namespace bb
}  // namespace mmbf

extern "C" {

mmbf_status mamba_mimo_bwd_bwd_workspace_size(const mmbf_dims* dims, int64_t chunk_size, int64_t rotary_dim_divisor,
                                              size_t* bytes) {
  using namespace mmbf::bb;
  BBParams p;
  mmbf_status s = bb_plan(dims, chunk_size, rotary_dim_divisor, &p);
  if (s != MMBF_OK) return s;
  if (!bytes) return fail(MMBF_ERR_ARG, "bytes is NULL");
  size_t off[5];
  *bytes = bb_workspace(p, off);
  return MMBF_OK;
}

mmbf_status mamba_mimo_bwd_bwd(const mmbf_dims* dims, const void* dout, const void* q, const void* k, const void* v,
                               const float* q_bias, const float* k_bias, const float* mimo_v, const void* states,
                               const void* qk_dot, const float* da_cs, const float* da_cs_rev, const float* dt,
                               const void* trap, const float* segsum, const float* angles, const float* mimo_o,
                               const float* d, int64_t chunk_size, int64_t rotary_dim_divisor, int act_dtype, int dqkv_dtype,
                               void* DQ, void* DK, void* DV, float* DMIMO_V, float* DANGLES, float* DFACTOR, float* DGAMMA, float* DDA,
                               float* DSSDA, float* DDA_CS_REV, float* DDA_CS, float* DD, void* workspace,
                               size_t workspace_bytes, void* stream) {
  using namespace mmbf::bb;
  BBParams p;
  mmbf_status s = bb_plan(dims, chunk_size, rotary_dim_divisor, &p);
  if (s != MMBF_OK) return s;
  const void* req[] = {dout, q, k, v, q_bias, k_bias, mimo_v, states, qk_dot, da_cs, da_cs_rev, dt, trap, segsum, angles,
                       DQ, DK, DV, DMIMO_V, DANGLES, DFACTOR, DGAMMA, DDA, DSSDA, DDA_CS_REV, DDA_CS};
  for (const void* x : req)
    if (!x) return fail(MMBF_ERR_ARG, "a required pointer is NULL");
  if ((d == nullptr) != (DD == nullptr)) return fail(MMBF_ERR_ARG, "DD must be given exactly when d is");
  if (act_dtype < kF32 || act_dtype > kF16) return fail(MMBF_ERR_ARG, "act_dtype must be 0 (fp32), 1 (bf16) or 2 (fp16)");
  if (dqkv_dtype < kF32 || dqkv_dtype > kF16)
    return fail(MMBF_ERR_ARG, "dqkv_dtype must be 0 (fp32), 1 (bf16) or 2 (fp16)");
  const void* all[] = {dout, q, k, v, q_bias, k_bias, mimo_v, states, qk_dot, da_cs, da_cs_rev, dt, trap, segsum,
                       angles, mimo_o, d, DQ, DK, DV, DMIMO_V, DANGLES, DFACTOR, DGAMMA, DDA, DSSDA, DDA_CS_REV, DDA_CS, DD};
  for (const void* x : all)
    if (x && (reinterpret_cast<uintptr_t>(x) & 3)) return fail(MMBF_ERR_ALIGN, "tensor pointers must be 4-byte aligned");
  size_t off[5];
  const size_t need = bb_workspace(p, off);
  if (!workspace || workspace_bytes < need)
    return fail(MMBF_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(MMBF_ERR_ALIGN, "workspace must be 256-byte aligned");
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.dout = dout; p.q = q; p.k = k; p.v = v; p.states = states; p.qk = qk_dot; p.trap = trap;
  p.act = act_dtype;
  p.q_bias = q_bias; p.k_bias = k_bias; p.mimo_v = mimo_v; p.mimo_o = mimo_o; p.d = d;
  p.da_cs = da_cs; p.da_cs_rev = da_cs_rev; p.dt = dt; p.segsum = segsum; p.angles = angles;
  p.reduced = mimo_o != nullptr;
  p.has_d = d != nullptr;
  p.DQ = DQ; p.DK = DK; p.DV = DV;
  p.dqkv = dqkv_dtype; p.DMIMO_V = DMIMO_V; p.DANGLES = DANGLES; p.DFACTOR = DFACTOR;
  p.DGAMMA = DGAMMA; p.DDA = DDA; p.DSSDA = DSSDA; p.DDA_CS_REV = DDA_CS_REV; p.DDA_CS = DDA_CS; p.DD = DD;
  p.ws_D = reinterpret_cast<float*>(ws + off[0]);
  p.ws_alpha = reinterpret_cast<float*>(ws + off[1]);
  p.ws_mv = reinterpret_cast<float*>(ws + off[2]);
  p.ws_dd = reinterpret_cast<float*>(ws + off[3]);
  p.ws_scr = p.wide ? reinterpret_cast<float*>(ws + off[4]) : nullptr;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = p.act == kBF16 ? launch_bb<kBF16>(p, st) : p.act == kF16 ? launch_bb<kF16>(p, st)
                                                                           : launch_bb<kF32>(p, st);
  if (e != cudaSuccess) return fail(MMBF_ERR_CUDA, "shared-memory attribute: %s", cudaGetErrorString(e));
  e = cudaGetLastError();
  g_launches = 4;
  if (e != cudaSuccess) return fail(MMBF_ERR_CUDA, "launching the second stage: %s", cudaGetErrorString(e));
  return MMBF_OK;
}

}  // extern "C"
