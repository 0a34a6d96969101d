/*
 * CPU oracle for the first backward stage of the Mamba-3 MIMO chunked scan
 * (`mamba_mimo_bwd_fwd`).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Source of the definition (all on the page "feat: add Triton-Ascend
 * implementation of Mamba-3 mamba_mimo_bwd_fwd #125", MindSpeed-Ops):
 *   [doc]     docs/triton/mamba_mimo_bwd_fwd.md, tables "输入与输出"
 *             (inputs / outputs, shapes, dtypes, constraints) and the
 *             paragraph after "Triton 实现" on the BF16 boundaries.
 *   [review]  docs/triton/mamba_mimo_bwd_fwd_review_validation.md, section
 *             "NPU 实现修改" (which fragments are rounded to BF16, and that
 *             the diagonal term is rounded rank by rank).
 *   [bf16ref] tests/unit_tests/triton/mamba_mimo_bwd_fwd_bf16_reference.py,
 *             the BF16-boundary reference: padding, GQA expansion, biased
 *             Q/K, same-token QK, rotary, PsiV, trapezoid factors, the chunk
 *             loop, and the Z / projection-gradient branch.
 *   [fp32ref] tests/unit_tests/triton/mamba_mimo_bwd_fwd_reference.py, the
 *             same algorithm with no BF16 boundaries.
 *   On the page "MindSpeed-Ops PR #100" (second stage), section
 *   "输入缓存的语义": states[c] is the state *entering* chunk c, and
 *   qk_dot[b,h,s,r_out,r_in] is the same-token R x R q.k block.
 *
 * Arithmetic.  Every value between two rounding points is carried in IEEE
 * double.  With `round_bf16 = 1` each rounding point that [bf16ref] and
 * [review] name rounds that double to the nearest BF16 value, ties to even
 * (the rounding of torch's float -> bfloat16 conversion); with
 * `round_bf16 = 0` no rounding point is applied at all (the [fp32ref]
 * algorithm, evaluated in double).  Input tensors are read at their own
 * precision in both modes.  sin, cos and exp are libm's double functions.
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes too):
 *   - BF16 rounding is round-to-nearest-even with the FP32 exponent range;
 *     the oracle rounds its double intermediate directly to BF16 (the pages
 *     round an FP32 intermediate; the two agree except within 2^-24 of a
 *     BF16 tie).
 *   - In exact mode, dt enters gamma unrounded and sigma(-trap) is the
 *     sigmoid of -trap, as in [fp32ref]; in BF16 mode bf16(dt) is used, as
 *     in [bf16ref].
 *   - The state decay of the last (possibly partial) chunk uses da_cs at the
 *     last valid token, as [bf16ref] does; the state after the last chunk is
 *     never an output, so the choice is not observable.
 *   - Sums over t of dmimo_o and dmimo_z run over the padded sequence in
 *     token order, accumulated in double.
 *
 * Parity pins of this file live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int64_t B, S, H, G, R, N, P, C; /* pages' symbols; C is chunk_size        */
  int64_t div;                    /* rotary_dim_divisor (2 or 4)            */
  int64_t reduced;                /* 1: mimo_o given, dout is [B,S,H,P]     */
                                  /* 0: dout is [B,S,R,H,P]                  */
  int64_t has_z;                  /* z and mimo_z given                     */
  int64_t has_d;                  /* d given                                */
  int64_t round_bf16;             /* 1: BF16 rounding points; 0: exact      */
} oracle_dims;

/* ------------------------------------------------------------------------ */
/* Number formats.                                                           */

/* A BF16 input element (its 16 bits) as the exact value it holds. */
static double from_bf16_bits(uint16_t u) {
  uint32_t w = ((uint32_t)u) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* Nearest BF16 value to x, ties to even: 8 significant bits, the exponent
 * range of FP32 (normal numbers down to 2^-126, subnormal quantum 2^-133),
 * overflow to infinity.  NaN and infinities pass through. */
static double bf16_nearest(double x) {
  if (x == 0.0 || isnan(x) || isinf(x)) return x;
  int e;
  frexp(x, &e); /* |x| in [2^(e-1), 2^e) */
  int quantum_exp = (e - 1 >= -126) ? (e - 8) : -133;
  double q = rint(ldexp(x, -quantum_exp)); /* rint: nearest, ties to even */
  double y = ldexp(q, quantum_exp);
  const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  if (fabs(y) > bf16_max) return copysign(INFINITY, x);
  return y;
}

/* A rounding point of [bf16ref]: active only in BF16 mode. */
static double bf(const oracle_dims* d, double x) {
  return d->round_bf16 ? bf16_nearest(x) : x;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Exposed for the rounding pin tests. */
double oracle_bf16_nearest(double x) { return bf16_nearest(x); }

/* ------------------------------------------------------------------------ */
/* Input access with the zero padding of [bf16ref] (positions t >= S read 0). */

typedef struct {
  const oracle_dims* d;
  const uint16_t *dout, *q, *k, *v, *z, *trap;                  /* BF16 */
  const float *q_bias, *k_bias, *mimo_v, *mimo_o, *mimo_z;       /* FP32 */
  const float *angles, *da_cs, *da_cs_rev, *dt, *dd, *segsum;    /* FP32 */
} oracle_inputs;

/* q[b,t,r,g,n], k likewise: [B,S,R,G,N] */
static double in_qk(const oracle_inputs* I, const uint16_t* x, int64_t b, int64_t t,
                    int64_t r, int64_t g, int64_t n) {
  const oracle_dims* d = I->d;
  if (t >= d->S) return 0.0;
  return from_bf16_bits(x[(((b * d->S + t) * d->R + r) * d->G + g) * d->N + n]);
}
/* v[b,t,h,p], z and reduced dout likewise: [B,S,H,P] */
static double in_bshp(const oracle_inputs* I, const uint16_t* x, int64_t b, int64_t t,
                      int64_t h, int64_t p) {
  const oracle_dims* d = I->d;
  if (t >= d->S) return 0.0;
  return from_bf16_bits(x[((b * d->S + t) * d->H + h) * d->P + p]);
}
/* non-reduced dout[b,t,r,h,p]: [B,S,R,H,P] */
static double in_dout_rank(const oracle_inputs* I, int64_t b, int64_t t, int64_t r,
                           int64_t h, int64_t p) {
  const oracle_dims* d = I->d;
  if (t >= d->S) return 0.0;
  return from_bf16_bits(I->dout[(((b * d->S + t) * d->R + r) * d->H + h) * d->P + p]);
}
/* da_cs, da_cs_rev, dt: FP32 [B,H,S]; trap: BF16 [B,H,S] */
static double in_bhs(const oracle_inputs* I, const float* x, int64_t b, int64_t h, int64_t t) {
  const oracle_dims* d = I->d;
  if (t >= d->S) return 0.0;
  return (double)x[(b * d->H + h) * d->S + t];
}
static double in_trap(const oracle_inputs* I, int64_t b, int64_t h, int64_t t) {
  const oracle_dims* d = I->d;
  if (t >= d->S) return 0.0;
  return from_bf16_bits(I->trap[(b * d->H + h) * d->S + t]);
}
/* angles[b,t,h,i]: FP32 [B,S,H,N/div] */
static double in_angle(const oracle_inputs* I, int64_t b, int64_t t, int64_t h, int64_t i) {
  const oracle_dims* d = I->d;
  if (t >= d->S) return 0.0;
  int64_t w = d->N / d->div;
  return (double)I->angles[((b * d->S + t) * d->H + h) * w + i];
}

/* ------------------------------------------------------------------------ */
/* Trapezoid discretisation ([bf16ref], the gamma / shifted-gamma / factor
 * block; dt enters through a BF16 load):
 *   gamma[t]   = bf16(dt[t]) * sigmoid(trap[t])                (not rounded)
 *   shifted[t] = bf16(bf16(dt[t+1]) * sigmoid(-trap[t+1])), 0 at the last
 *                padded position
 *   factor[t]  = bf16(gamma[t] + shifted[t])
 * In exact mode [fp32ref]: dt unrounded and (1 - sigmoid(trap)) for the
 * shifted part, which is the same number as sigmoid(-trap). */
static double gamma_at(const oracle_inputs* I, int64_t b, int64_t h, int64_t t) {
  const oracle_dims* d = I->d;
  return bf(d, in_bhs(I, I->dt, b, h, t)) * sigmoid(in_trap(I, b, h, t));
}
static double shifted_at(const oracle_inputs* I, int64_t b, int64_t h, int64_t t, int64_t Sp) {
  const oracle_dims* d = I->d;
  if (t + 1 >= Sp) return 0.0;
  return bf(d, bf(d, in_bhs(I, I->dt, b, h, t + 1)) * sigmoid(-in_trap(I, b, h, t + 1)));
}

/* ------------------------------------------------------------------------ */
/* One (b,h) pair.  Output slots are compact per pair:
 *   states  [nc, N, P]   the state entering each chunk          ([doc], PR #100)
 *   qk_dot  [S, R, R]    same-token q.k, [r_out, r_in]
 *   dz      [S, P]       (has_z)
 *   dmimo_o [R, P]       (reduced)
 *   dmimo_z [R, P]       (has_z)
 *   out     [Sp, R, P]   the chunk output before gating (optional; the op
 *                        never returns it, the pins use it)                 */
typedef struct {
  double *states, *qk_dot, *dz, *dmimo_o, *dmimo_z, *out;
} pair_outputs;

static int run_pair(const oracle_inputs* I, int64_t b, int64_t h, pair_outputs* O) {
  const oracle_dims* d = I->d;
  const int64_t R = d->R, N = d->N, P = d->P, C = d->C, S = d->S;
  const int64_t nc = (S + C - 1) / C, Sp = nc * C, CR = C * R;
  /* Head h reads Q/K group g: repeat_interleave of the G axis ([bf16ref]). */
  const int64_t g = h / (d->H / d->G);
  const int64_t w = N / d->div, half = N / 2;

  double* qh = calloc((size_t)(CR * N), sizeof(double));    /* biased q   */
  double* kh = calloc((size_t)(CR * N), sizeof(double));    /* biased k   */
  double* qr = calloc((size_t)(CR * N), sizeof(double));    /* rotated q  */
  double* ks = calloc((size_t)(CR * N), sizeof(double));    /* k_scaled   */
  double* psi = calloc((size_t)(CR * P), sizeof(double));   /* PsiV       */
  double* qk = calloc((size_t)(C * R * R), sizeof(double)); /* qk_dot     */
  double* amat = calloc((size_t)(CR * CR), sizeof(double)); /* causal A   */
  double* outc = calloc((size_t)(CR * P), sizeof(double));  /* chunk out  */
  double* state = calloc((size_t)(N * P), sizeof(double));
  double* sb = calloc((size_t)(N * P), sizeof(double));
  double* gam = calloc((size_t)C, sizeof(double));
  double* fac = calloc((size_t)C, sizeof(double));
  if (!qh || !kh || !qr || !ks || !psi || !qk || !amat || !outc || !state || !sb || !gam ||
      !fac) {
    free(qh); free(kh); free(qr); free(ks); free(psi); free(qk); free(amat); free(outc);
    free(state); free(sb); free(gam); free(fac);
    return 1;
  }
  if (O->dmimo_o) memset(O->dmimo_o, 0, sizeof(double) * (size_t)(R * P));
  if (O->dmimo_z) memset(O->dmimo_z, 0, sizeof(double) * (size_t)(R * P));

  for (int64_t c = 0; c < nc; c++) {
    const int64_t t0 = c * C;

    /* Step 1. Biased Q/K: bf16(x + bf16(bias[h])) ([bf16ref]: the FP32 bias
     * is itself rounded to BF16 before the add, and the sum is rounded). */
    for (int64_t i = 0; i < C; i++)
      for (int64_t r = 0; r < R; r++)
        for (int64_t n = 0; n < N; n++) {
          int64_t j = i * R + r;
          qh[j * N + n] = bf(d, in_qk(I, I->q, b, t0 + i, r, g, n) +
                                    bf(d, (double)I->q_bias[(h * R + r) * N + n]));
          kh[j * N + n] = bf(d, in_qk(I, I->k, b, t0 + i, r, g, n) +
                                    bf(d, (double)I->k_bias[(h * R + r) * N + n]));
        }

    /* Step 2. Same-token QK of the biased, un-rotated q and k:
     * qk_dot[t,r,s] = bf16(sum_n qh[t,r,n] kh[t,s,n]) (einsum bhtrn,bhtsn). */
    for (int64_t i = 0; i < C; i++)
      for (int64_t r = 0; r < R; r++)
        for (int64_t s = 0; s < R; s++) {
          double acc = 0.0;
          for (int64_t n = 0; n < N; n++)
            acc += qh[(i * R + r) * N + n] * kh[(i * R + s) * N + n];
          qk[(i * R + r) * R + s] = bf(d, acc);
        }

    /* Step 3. Rotary on the pairs (m, N/2 + m), m < N/div, angle per
     * (b, t, h, m); other columns are copied ([bf16ref] _rotate). */
    for (int64_t i = 0; i < C; i++)
      for (int64_t r = 0; r < R; r++) {
        int64_t j = i * R + r;
        for (int64_t n = 0; n < N; n++) {
          qr[j * N + n] = qh[j * N + n];
          ks[j * N + n] = kh[j * N + n];
        }
        for (int64_t m = 0; m < w; m++) {
          double th = in_angle(I, b, t0 + i, h, m), cs = cos(th), sn = sin(th);
          double a = qh[j * N + m], e = qh[j * N + half + m];
          qr[j * N + m] = bf(d, cs * a - sn * e);
          qr[j * N + half + m] = bf(d, sn * a + cs * e);
          a = kh[j * N + m];
          e = kh[j * N + half + m];
          ks[j * N + m] = bf(d, cs * a - sn * e);
          ks[j * N + half + m] = bf(d, sn * a + cs * e);
        }
      }

    /* Step 4. PsiV = bf16(v * bf16(mimo_v)), value up-projected to R ranks. */
    for (int64_t i = 0; i < C; i++)
      for (int64_t r = 0; r < R; r++)
        for (int64_t p = 0; p < P; p++)
          psi[(i * R + r) * P + p] =
              bf(d, in_bshp(I, I->v, b, t0 + i, h, p) * bf(d, (double)I->mimo_v[(h * R + r) * P + p]));

    /* Step 5. gamma / factor, then k_scaled = bf16(k_rot * factor[t]). */
    for (int64_t i = 0; i < C; i++) {
      gam[i] = gamma_at(I, b, h, t0 + i);
      fac[i] = bf(d, gam[i] + shifted_at(I, b, h, t0 + i, Sp));
      for (int64_t r = 0; r < R; r++)
        for (int64_t n = 0; n < N; n++) {
          int64_t j = i * R + r;
          ks[j * N + n] = bf(d, ks[j * N + n] * fac[i]);
        }
    }

    /* Step 6.1. states[c] = bf16(state entering chunk c). */
    for (int64_t x = 0; x < N * P; x++) {
      sb[x] = bf(d, state[x]);
      O->states[c * N * P + x] = sb[x];
    }

    /* Step 6.2. inter[j,p] = (sum_n qr[j,n] bf16(state)[n,p]) * exp(da_cs[t_j]);
     * rows j = t*R + r (flatten of the chunk's token and rank axes). */
    for (int64_t j = 0; j < CR; j++) {
      double eda = exp(in_bhs(I, I->da_cs, b, h, t0 + j / R));
      for (int64_t p = 0; p < P; p++) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; n++) acc += qr[j * N + n] * sb[n * P + p];
        outc[j * P + p] = acc * eda;
      }
    }

    /* Step 6.3. A[i,j] = bf16(t_i > t_j ? (qr_i . ks_j) exp(segsum[c,t_i,t_j]) : 0).
     * Strictly causal on the token index: same-token pairs of different ranks
     * are excluded (the diagonal term below covers them). */
    const float* seg = I->segsum + ((b * d->H + h) * nc + c) * C * C;
    for (int64_t i = 0; i < CR; i++)
      for (int64_t j = 0; j < CR; j++) {
        int64_t ti = i / R, tj = j / R;
        double val = 0.0;
        if (ti > tj) {
          double acc = 0.0;
          for (int64_t n = 0; n < N; n++) acc += qr[i * N + n] * ks[j * N + n];
          val = acc * exp((double)seg[ti * C + tj]);
        }
        amat[i * CR + j] = bf(d, val);
      }

    /* Step 6.4. intra = A @ PsiV, added to inter. */
    for (int64_t i = 0; i < CR; i++)
      for (int64_t p = 0; p < P; p++) {
        double acc = 0.0;
        for (int64_t j = 0; j < CR; j++) acc += amat[i * CR + j] * psi[j * P + p];
        outc[i * P + p] += acc;
      }

    /* Step 6.5-6.6. Diagonal term, rank by rank with BF16 product and BF16
     * sum ([review]: no FP32 dot over ranks), scaled by gamma (not factor); then
     * out = bf16(inter + intra + diag + d[h] * PsiV). */
    for (int64_t i = 0; i < C; i++)
      for (int64_t o = 0; o < R; o++)
        for (int64_t p = 0; p < P; p++) {
          double dg = 0.0;
          for (int64_t r = 0; r < R; r++)
            dg = bf(d, dg + bf(d, qk[(i * R + o) * R + r] * psi[(i * R + r) * P + p]));
          dg = bf(d, dg * gam[i]);
          int64_t j = i * R + o;
          double x = outc[j * P + p] + dg;
          if (d->has_d) x += (double)I->dd[h] * psi[j * P + p];
          outc[j * P + p] = bf(d, x);
        }

    /* Step 6.7. k_state = bf16(k_scaled * exp(da_cs_rev[t])); the state
     * decays by exp(da_cs) at the chunk's last valid token and takes
     * k_state^T @ PsiV. */
    {
      int64_t last = (t0 + C < S ? t0 + C : S) - 1;
      double alpha = exp(in_bhs(I, I->da_cs, b, h, last));
      for (int64_t x = 0; x < N * P; x++) state[x] *= alpha;
      for (int64_t j = 0; j < CR; j++) {
        double edr = exp(in_bhs(I, I->da_cs_rev, b, h, t0 + j / R));
        for (int64_t n = 0; n < N; n++) {
          double kst = bf(d, ks[j * N + n] * edr);
          for (int64_t p = 0; p < P; p++) state[n * P + p] += kst * psi[j * P + p];
        }
      }
    }

    /* qk_dot and (optionally) out leave the chunk here; qk_dot only for t < S. */
    for (int64_t i = 0; i < C; i++) {
      if (t0 + i < S)
        for (int64_t x = 0; x < R * R; x++) O->qk_dot[(t0 + i) * R * R + x] = qk[i * R * R + x];
      if (O->out)
        for (int64_t x = 0; x < R * P; x++) O->out[(t0 + i) * R * P + x] = outc[i * R * P + x];
    }

    /* Step 7. Output-projection and gate gradients ([bf16ref] after the chunk
     * loop), with pz = z * mimo_z in full precision (mimo_z is not rounded):
     *   reduced, Z:    dmimo_o += out silu(pz) dout;  pre = bf16(bf16(dout bf16(mimo_o)) out)
     *   reduced, no Z: dmimo_o += out dout
     *   per-rank dout, Z: pre = bf16(dout[t,r] out)
     *   Z: gzp = pre sigmoid(pz) (1 + pz sigmoid(-pz)) (derivative of silu);
     *      dz = rank-ordered BF16 sum of gzp mimo_z;  dmimo_z += gzp z. */
    if (d->reduced || d->has_z) {
      for (int64_t i = 0; i < C; i++) {
        int64_t t = t0 + i;
        for (int64_t p = 0; p < P; p++) {
          double zt = d->has_z ? in_bshp(I, I->z, b, t, h, p) : 0.0;
          double dzacc = 0.0;
          for (int64_t r = 0; r < R; r++) {
            double o = outc[(i * R + r) * P + p];
            double pz = d->has_z ? zt * (double)I->mimo_z[(h * R + r) * P + p] : 0.0;
            double pre = 0.0;
            if (d->reduced) {
              double dt_ = in_bshp(I, I->dout, b, t, h, p);
              if (d->has_z) {
                O->dmimo_o[r * P + p] += o * (pz * sigmoid(pz)) * dt_;
                pre = bf(d, bf(d, dt_ * bf(d, (double)I->mimo_o[(h * R + r) * P + p])) * o);
              } else {
                O->dmimo_o[r * P + p] += o * dt_;
              }
            } else if (d->has_z) {
              pre = bf(d, in_dout_rank(I, b, t, r, h, p) * o);
            }
            if (d->has_z) {
              double gzp = pre * sigmoid(pz) * (1.0 + pz * sigmoid(-pz));
              dzacc = bf(d, dzacc + gzp * (double)I->mimo_z[(h * R + r) * P + p]);
              O->dmimo_z[r * P + p] += gzp * zt;
            }
          }
          if (d->has_z && t < S) O->dz[t * P + p] = dzacc;
        }
      }
    }
  }

  free(qh); free(kh); free(qr); free(ks); free(psi); free(qk); free(amat); free(outc);
  free(state); free(sb); free(gam); free(fac);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Entry point.  `pairs` lists n_pairs (b,h) pairs as 2*n_pairs int64 values;
 * outputs are written per pair at slot i of each compact output array (see
 * pair_outputs).  Optional outputs are NULL when absent.  Returns 0, or a
 * nonzero count of pairs that failed (allocation).  Pairs run in parallel
 * (OpenMP) when the library is built with it; each pair is sequential. */
int oracle_bwd_fwd(const oracle_dims* d, const uint16_t* dout, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, const float* q_bias,
                   const float* k_bias, const float* mimo_v, const float* mimo_o,
                   const uint16_t* z, const float* mimo_z, const float* angles,
                   const float* da_cs, const float* da_cs_rev, const float* dt,
                   const uint16_t* trap, const float* dd, const float* segsum,
                   int64_t n_pairs, const int64_t* pairs, double* states, double* qk_dot,
                   double* dz, double* dmimo_o, double* dmimo_z, double* out) {
  oracle_inputs I = {d,      dout,   q,      k,     v,         z,      trap,
                     q_bias, k_bias, mimo_v, mimo_o, mimo_z,   angles, da_cs,
                     da_cs_rev, dt,  dd,     segsum};
  const int64_t nc = (d->S + d->C - 1) / d->C, Sp = nc * d->C;
  const int64_t R = d->R, N = d->N, P = d->P, S = d->S;
  int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : failed)
  for (int64_t i = 0; i < n_pairs; i++) {
    pair_outputs O;
    O.states = states + i * nc * N * P;
    O.qk_dot = qk_dot + i * S * R * R;
    O.dz = dz ? dz + i * S * P : NULL;
    O.dmimo_o = dmimo_o ? dmimo_o + i * R * P : NULL;
    O.dmimo_z = dmimo_z ? dmimo_z + i * R * P : NULL;
    O.out = out ? out + i * Sp * R * P : NULL;
    failed += run_pair(&I, pairs[2 * i], pairs[2 * i + 1], &O);
  }
  return failed;
}
