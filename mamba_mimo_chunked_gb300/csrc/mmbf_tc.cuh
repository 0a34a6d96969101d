// Warp-specialised output kernel of mamba_mimo_bwd_fwd for the pages' timed
// shape family: R = 4, C = 16, N = P = 64, reduced dout (mimo_o given), Z and
// D optional (included by mmbf_kernels.cu inside namespace mmbf, after
// mmbf_fast.cuh, whose TMA, mbarrier, fragment and tensor-memory helpers it
// uses).
//
// What one chunk computes is the op document's chunk output (page "feat: add
// Triton-Ascend implementation of Mamba-3 mamba_mimo_bwd_fwd #125", section
// "Triton 实现", items 5-7, and the BF16 reference): every rounding point of
// the BF16 reference is kept, as in the other kernel families.  How it is
// computed here:
//
// * One CTA per (b*h, segment) and SM (all 512 tensor-memory columns), all
//   resident at once (a cooperative launch).  Phase A: the CTA sums its own
//   segment's state contributions (U of every chunk on tcgen05.mma, each
//   group of four warps folding its chunks with their decays) and publishes
//   the sum with a release flag.  Then it folds the sums of the earlier
//   segments of its (b,h) (acquire, bounded spin) into the state entering
//   the segment.  Phase C: it walks the segment's chunks with the FP32 state
//   in registers.
// * Contractions of a chunk on tcgen05.mma (64x64x64 BF16, FP32 accumulator
//   in tensor memory, M = 64 layout: row m at lane 32(m/16) + m%16,
//   double-buffered across chunks):
//     U       = PsiV^T k_state          (the chunk's state contribution, [p][n])
//     inter^T = bf16(state)^T Q_rot^T   ([p][j])
//     intra^T = PsiV^T A^T              ([p][j], A = bf16(mask(S) exp(segsum)))
//   and on mma.sync (register fragments): S = Q_rot Ks^T on the causal 16x16
//   blocks, the same-token qk_dot on the diagonal blocks.  Rows j of the
//   chunk are stored in the fragment order of fast::perm() inside each 16-row
//   block, so a thread that reads inter^T / intra^T as 16x256b fragments
//   holds all four ranks of one token for a pair of p values (p, p+8): the
//   rank-ordered BF16 diagonal and dz need no cross-lane traffic.
// * Warp roles in phase C (16 warps, 4 per scheduler):
//     0-7   epilogue: warp w reads p-block w%4 and the j-columns of tokens
//           8(w/4)..8(w/4)+7; diagonal, out, Z branch, dmimo partials, dz;
//     8-11  prologue: one 16-row j-block each; biased Q/K, same-token qk_dot,
//           rotary, k_scaled, k_state, PsiV, the token-scalar table; warp 8's
//           first thread loads dout and z (ring O);
//     12-15 state: p-block w%4 of the FP32 state, folded with U of the
//           previous chunk (tensor memory, issued a chunk ahead); bf16(state)
//           for inter^T and the states output; the causal rows 16(w%4).. of
//           A.  Warp 12's first thread issues inter^T and U of the next chunk,
//           warp 13's intra^T (an issue stalls its thread for about the MMA's
//           run time, so the accumulators go out from different threads);
//           warp 12's also stores states, warp 15's refills ring I.  Only the
//           fold is serial from chunk to chunk.
// * Two TMA rings: ring I (q, k, v, angles, segsum; the prologue writes Q_rot
//   and k_scaled over the raw q and k rows, k_state beside them) is freed when
//   the chunk's MMAs complete; ring O (PsiV, dout, z -> dz, the qk table) when
//   the epilogue is done and dz has left.  Four slots each.
// * All hand-offs are mbarriers.  Every wait is bounded (about a second of
//   %globaltimer); a wait that runs out records the tagged error word and sets
//   a CTA abort flag that ends every other wait at once, so the CTA drains its
//   copies in flight and leaves.

namespace tc {

constexpr unsigned kFull = 0xffffffffu;

template <int DIV_>
struct TCfg {
  using K = fast::Cfg<4, 16, 64, 64, DIV_, 1>;  // the shared prologue helpers' view
  static constexpr int R = 4, C = 16, N = 64, P = 64, CR = 64, DIV = DIV_, W = N / DIV_;
  static constexpr int NI = 4, NO = 4;            // ring depths
  static constexpr int TW = 8, TS = 4 * C;        // token table: window of 8 chunks, 64 floats per chunk
  static constexpr int QKS = K::QKS;              // words per token in the qk table
  static constexpr int NWARP = 16, NT = NWARP * 32;
  static constexpr int WP = 8, WS = 12, WM = 16;  // first prologue / state warp, end of the state warps
  // ring I slot
  static constexpr uint32_t I_Q = 0, I_K = 8192, I_KST = 16384, I_V = 24576, I_ANG = 26624, I_SEG = 28672,
                            I_BYTES = 29696;
  // ring O slot
  static constexpr uint32_t O_PSI = 0, O_DOUT = 8192, O_Z = 10240, O_QKD = 12288, O_BYTES = 14336;
  // CTA layout (offsets from the 1024-byte aligned base)
  static constexpr uint32_t RI = 0, RO = NI * I_BYTES, SBT = RO + NO * O_BYTES, ATT = SBT + 2 * 8192,
                            TOK = ATT + 2 * 8192, MVB = TOK + 2 * TW * TS * 4, QBS = MVB + R * P * 2,
                            KBS = QBS + R * K::LDB * 2, MZP = KBS + R * K::LDB * 2, MOP = MZP + R * 4 * 8 * 8,
                            BAR = MOP + R * 4 * 8 * 4;
  // barriers: full / pdone / ofree / fullO / PsiV per ring slot, the rest
  // per tensor-memory / tile buffer (two) or one
  enum : uint32_t {
    B_FULLI = 0, B_FULLO = 4, B_PDONE = 8, B_OFREE = 12, B_U = 16, B_M2 = 18, B_SBR = 20, B_TOKW = 22,
    // phase A of the single-kernel form: per group TMA (3 buffers), prologue done, MMA done (2 buffers)
    B_AFULL = 24, B_APA = 36, B_AU = 44, B_AUF = 52, NBAR = 60
  };

  static constexpr uint32_t MISC = BAR + ((NBAR * 8 + 15) & ~15u);  // tmem slot, abort flag, last-CTA flag
  // Phase A (the segment's own state sum, single-kernel form), laid over the
  // ring and tile regions before phase C uses them (below the parameter
  // tables): per group of four warps three staging buffers of raw k (k_state
  // is written over it), v and angles, and two PsiV tiles; the segment's
  // token scalars (factor, exp(da_cs_rev)) and chunk weights after MISC.
  static constexpr uint32_t A_K = 0, A_V = 8192, A_ANG = 10240, A_BUF = 12288;
  static constexpr uint32_t A_RAW = 0, A_PSI = 12 * A_BUF;
  static constexpr int LMAX = 64;  // longest segment of the single-kernel form
  static constexpr uint32_t A_FAC = (MISC + 16 + 127) & ~127u, A_EDR = A_FAC + LMAX * C * 4,
                            A_GAM = A_EDR + LMAX * C * 4, A_ALP = A_GAM + LMAX * 4, A_D4 = A_ALP + LMAX * 4,
                            A_DEC = A_D4 + LMAX * 4;
  static constexpr uint32_t SMEM = A_DEC + 16 + 1024;  // + alignment slack of the base
  // tensor-memory columns (two buffers of 64 each)
  static constexpr uint32_t T_S = 0, T_U = 128, T_I = 256, T_X = 384;
  static_assert(I_ANG + C * W * 4 <= I_SEG && I_SEG + C * C * 4 <= I_BYTES, "ring I slot");
  static_assert(O_QKD + C * QKS * 4 <= O_BYTES && QKS % 4 == 0 && O_QKD % 16 == 0, "ring O slot, qk table rows");
  static_assert(I_BYTES % 1024 == 0 && O_BYTES % 1024 == 0 && RO % 1024 == 0 && SBT % 1024 == 0, "alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(W == 16, "register prologue: N / rotary_dim_divisor = 16 rotated pairs");
  static_assert(A_PSI + 8 * 8192 <= MVB, "phase A layout");
  static_assert(A_BUF % 1024 == 0 && A_PSI % 1024 == 0 && 4 * 4096 * 4 <= A_PSI, "phase A alignment, reduction scratch");
};

__device__ __forceinline__ void arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about `ns` nanoseconds pass (it does not spin meanwhile, so a
// waiting warp takes no issue slots from the warps it waits for).
__device__ __forceinline__ bool try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t kSleepNs = 20000;  // bound and abort flag are checked every ~20 us of waiting
// Non-blocking test of phase `parity` (never suspends the thread).
__device__ __forceinline__ bool test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity`; false if the CTA is aborting or the wait
// ran out (then the abort flag is set and the error word recorded).
__device__ __forceinline__ bool wait_b(const Params& p, uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                       uint32_t code) {
  if (fast::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = fast::global_ns();
  while (true) {
    if (try_wait_sleep(bar, parity, kSleepNs)) return true;
    if (*abort_flag) return false;
    if (fast::global_ns() - t0 > fast::kWaitLimitNs) {
      *abort_flag = 1u;
      atomicExch(p.ws_err, (p.tag << 8) | code);
      return false;
    }
  }
}
// Bounded wait without the abort protocol (draining copies in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = fast::global_ns();
  while (!try_wait_sleep(bar, parity, kSleepNs))
    if (fast::global_ns() - t0 > fast::kWaitLimitNs) break;
}

// 64x64x64 BF16 MMA, FP32 accumulator in tensor memory (M = N = 64).  A is
// [M][K] (K-major: rows of 128 bytes along K) or [K][M] (MN-major); B is [N][K]
// (K-major) or [K][N] (MN-major); 128-byte swizzled tiles, 1024-byte aligned.
// A K-step of 16 advances 32 bytes inside a K-major row, 16 rows (2048 bytes)
// of an MN-major tile.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma64(uint32_t tmem_d, uint32_t a_saddr, uint32_t b_saddr) {
  constexpr uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (A_MN ? (1u << 15) : 0u) |
                             (B_MN ? (1u << 16) : 0u) | ((64u >> 3) << 17) | ((64u >> 4) << 24);
  // A K-step moves the start address (descriptor bits 0-13, in 16-byte units)
  // by 32 bytes (K-major) or 2048 bytes (MN-major); shared-memory addresses
  // stay below 256 KB, so the field never carries into the bits above it.
  constexpr uint64_t da = A_MN ? 2048 / 16 : 32 / 16, dbs = B_MN ? 2048 / 16 : 32 / 16;
  const uint64_t a0 = fast::umma_desc_mn128(a_saddr), b0 = fast::umma_desc_mn128(b_saddr);
  asm volatile(
      "{\n .reg .pred p0, p1;\n setp.ne.b32 p0, %9, 0;\n setp.eq.b32 p1, %9, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %5, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %7, %3, p1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %10, %3, p1;\n}\n" ::"r"(tmem_d),
      "l"(a0), "l"(b0), "r"(idesc), "l"(a0 + da), "l"(b0 + dbs), "l"(a0 + 2 * da), "l"(b0 + 2 * dbs),
      "l"(a0 + 3 * da), "r"(0u), "l"(b0 + 3 * dbs)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}

// Token of physical row i (0..63) of a chunk tile: rows are in perm<4> order
// inside each 16-row block.
__device__ __forceinline__ int token_of(int i) { return 4 * (i >> 4) + ((i & 7) >> 1); }

// The prologue of one 16-row j-block with its operands in registers.  With
// R = 4 every fragment row of a thread (rows perm(g), perm(g + 8) of the
// block) belongs to token j0/4 + g/2, and the bias row of fragment register
// e is rank 2(e & 1) + (g & 1).
template <class T>
struct RowRegs {
  // bf16(bias) pairs of the 16 fragment registers
  uint32_t b[4][4];
  __device__ __forceinline__ void load(const uint16_t* bias) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c2 = 2 * (lane & 3);
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const int r = 2 * (e & 1) + (g & 1);
#pragma unroll
      for (int kt = 0; kt < 4; kt++)
        b[kt][e] = *reinterpret_cast<const uint32_t*>(bias + r * T::K::LDB + kt * 16 + 8 * (e >> 1) + c2);
    }
  }
};
// x = bf16(x + bf16(bias)) on every fragment register.
__device__ __forceinline__ void add_bias_r(uint32_t (&f)[4][4], const uint32_t (&b)[4][4]) {
#pragma unroll
  for (int kt = 0; kt < 4; kt++)
#pragma unroll
    for (int e = 0; e < 4; e++) f[kt][e] = badd2(f[kt][e], b[kt][e]);
}
// Rotary (N = 64, N/4 = 16 rotated pairs (m, 32 + m)): the thread's columns
// m = 2(lane & 3) + {0, 1} (registers e = 0, 1) and 8 + the same (e = 2, 3)
// of tile 0 pair with tile 2; a0 / a1 are the token's angles at those
// columns.  Same arithmetic as the shared-table form.
template <class K>
__device__ __forceinline__ void rotate_r(uint32_t (&fq)[4][4], uint32_t (&fk)[4][4], bool with_q, float2 a0,
                                         float2 a1) {
  float2 sn0, cs0, sn1, cs1;
  fast::sincos_fast(a0.x, &sn0.x, &cs0.x);
  fast::sincos_fast(a0.y, &sn0.y, &cs0.y);
  fast::sincos_fast(a1.x, &sn1.x, &cs1.x);
  fast::sincos_fast(a1.y, &sn1.y, &cs1.y);
#pragma unroll
  for (int e = 0; e < 4; e++) {
    const float2 cs = (e >> 1) ? cs1 : cs0, sn = (e >> 1) ? sn1 : sn0;
    if (with_q) fast::rotate_regs<K>(fq[0][e], fq[2][e], cs, sn);
    fast::rotate_regs<K>(fk[0][e], fk[2][e], cs, sn);
  }
}
// k_scaled = bf16(k_rot * factor) (BF16 x BF16), factor of the thread's token.
__device__ __forceinline__ void scale_r(uint32_t (&f)[4][4], uint32_t fd) {
#pragma unroll
  for (int kt = 0; kt < 4; kt++)
#pragma unroll
    for (int e = 0; e < 4; e++) f[kt][e] = bmul2(f[kt][e], fd);
}
// k_state = bf16(k_scaled * exp(da_cs_rev)) (FP32 product), the thread's token.
__device__ __forceinline__ void kstate_r(uint32_t (&f)[4][4], float x) {
  const float2 x2 = make_float2(x, x);
#pragma unroll
  for (int kt = 0; kt < 4; kt++)
#pragma unroll
    for (int e = 0; e < 4; e++) f[kt][e] = fast::pack2(__fmul2_rn(fast::unpack2(f[kt][e]), x2));
}

// Raw token inputs of the window starting at chunk cw, one token per
// prologue thread (pt = 0..127: token cw*C + pt).
template <class T>
__device__ __forceinline__ fast::TokRaw tok_load(const Params& p, int bh, int cw, int pt) {
  fast::TokRaw r = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const int tg = cw * T::C + pt;
  const int64_t i = (int64_t)bh * p.S + tg;
  if (tg < p.S) {
    r.dt = __ldg(p.dt + i);
    r.tr = bf_f(__ldg(p.trap + i));
    r.a = __ldg(p.da_cs + i);
    r.ar = __ldg(p.da_cs_rev + i);
  }
  if (tg + 1 < p.S) {
    r.dtn = __ldg(p.dt + i + 1);
    r.trn = bf_f(__ldg(p.trap + i + 1));
  }
  return r;
}
// Token scalars of one token into the window table (same arithmetic as
// fast::token_window): gamma = bf16(dt) sigmoid(trap); factor = bf16(gamma +
// bf16(bf16(dt[t+1]) sigmoid(-trap[t+1]))) (0 shifted term at the last padded
// position) as a BF16 pair; exp(da_cs); exp(da_cs_rev).
template <class T>
__device__ __forceinline__ void tok_fill(const Params& p, const fast::TokRaw& v, float* tab, int cw, int pt) {
  const int tg = cw * T::C + pt;
  float* tok = tab + (pt / T::C) * T::TS;
  const int t = pt % T::C;
  const float gam = __fmul_rn(round_bf(v.dt), sigmoid_f(v.tr));
  float sh = 0.f;
  if (tg + 1 < p.nc * T::C) sh = round_bf(__fmul_rn(round_bf(v.dtn), 1.0f / (1.0f + expf(v.trn))));
  tok[t] = gam;
  reinterpret_cast<uint32_t*>(tok)[T::C + t] = fast::dup_bf(__fadd_rn(gam, sh));
  tok[2 * T::C + t] = expf(v.a);
  tok[3 * T::C + t] = expf(v.ar);
}

template <class T, int MODE>
__global__ void __launch_bounds__(T::NT, 1) out_kernel(const __grid_constant__ Params p) {
  using K = typename T::K;
  constexpr int R = T::R, C = T::C, N = T::N, P = T::P;
  const bool HZ = MODE >= 0 ? (MODE & 2) != 0 : p.has_z != 0;
  const bool HD = MODE >= 0 ? (MODE & 4) != 0 : p.has_d != 0;
  extern __shared__ __align__(128) unsigned char sm_raw[];
  unsigned char* sm;
  {
    const uint32_t a = smem_u32(sm_raw);
    sm = sm_raw + (((a + 1023u) & ~1023u) - a);
  }
  const uint32_t sb = smem_u32(sm);
  const int bh = blockIdx.x, seg = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H, grp = h / (p.H / p.G);
  const int c0 = seg * p.L, c1 = min(p.nc, c0 + p.L);
  int n = c1 - c0;  // chunks of phase C (0 if phase A stopped)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, cq = lane & 3, mi = lane >> 3, li = lane & 7;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + T::MISC + 4);
  auto bar = [&](uint32_t i) { return sb + T::BAR + 8u * i; };

  // ---- set-up: barriers, tensor memory, parameter tables
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; i++) {
      fast::mbar_init(bar(T::B_FULLI + i), 1);
      fast::mbar_init(bar(T::B_FULLO + i), 1);
      fast::mbar_init(bar(T::B_PDONE + i), 4);
      fast::mbar_init(bar(T::B_OFREE + i), 8);
    }
    for (int i = 0; i < 12; i++) fast::mbar_init(bar(T::B_AFULL + i), 1);
    // a group's chunk prologue done, per chunk parity: only the MMA thread
    // waits, so a warp may arrive for chunk k + 1 before a slower one has
    // arrived for k; with one barrier per parity that arrival cannot complete
    // chunk k's phase (and none for k + 2 comes before U_k has gone out,
    // since the warp's fold of k waits for it)
    for (int i = 0; i < 8; i++) fast::mbar_init(bar(T::B_APA + i), 4);
    for (int i = 0; i < 8; i++) {
      fast::mbar_init(bar(T::B_AU + i), 1);   // a group's U MMA done (per tensor-memory buffer)
      fast::mbar_init(bar(T::B_AUF + i), 4);  // the group's four warps folded that buffer
    }
    for (int i = 0; i < 2; i++) {
      fast::mbar_init(bar(T::B_U + i), 1);
      fast::mbar_init(bar(T::B_M2 + i), 2);  // inter^T and intra^T, two issuing threads
      // chunk c's issue: the four state warps and the eight epilogue warps
      // done with chunk c - 2's products
      fast::mbar_init(bar(T::B_SBR + i), 4 + 8);
      fast::mbar_init(bar(T::B_TOKW + i), 4);
    }
    *abort_flag = 0u;
    fast::mbar_fence_init();
  }
  uint32_t* tm_slot = reinterpret_cast<uint32_t*>(sm + T::MISC);
  if (warp == T::WS) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(smem_u32(tm_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  {
    uint16_t* mvb = reinterpret_cast<uint16_t*>(sm + T::MVB);
    uint16_t* qbs = reinterpret_cast<uint16_t*>(sm + T::QBS);
    uint16_t* kbs = reinterpret_cast<uint16_t*>(sm + T::KBS);
    for (int e = threadIdx.x; e < R * P; e += T::NT) mvb[e] = f_bf(p.mimo_v[(int64_t)h * R * P + e]);
    for (int e = threadIdx.x; e < R * N; e += T::NT) {
      const int at = (e / N) * K::LDB + e % N;
      qbs[at] = f_bf(p.q_bias[(int64_t)h * R * N + e]);
      kbs[at] = f_bf(p.k_bias[(int64_t)h * R * N + e]);
    }
    float2* mzp = reinterpret_cast<float2*>(sm + T::MZP);
    uint32_t* mop = reinterpret_cast<uint32_t*>(sm + T::MOP);
    for (int e = threadIdx.x; e < R * 4 * 8; e += T::NT) {
      const int o = e / 32, mt = (e / 8) % 4, gg = e % 8;
      const float* mo = p.mimo_o + ((int64_t)h * R + o) * P + mt * 16 + gg;
      mop[e] = (uint32_t)f_bf(mo[0]) | ((uint32_t)f_bf(mo[8]) << 16);
      if (HZ) {
        const float* mz = p.mimo_z + ((int64_t)h * R + o) * P + mt * 16 + gg;
        mzp[e] = make_float2(mz[0], mz[8]);
      }
    }
  }
  fast::tm_fence_before();
  __syncthreads();
  fast::tm_fence_after();
  const uint32_t tmem = *tm_slot;

  // TMA loads of chunk c0 + i into its ring slots (one thread each ring)
  auto load_I = [&](int i) {
    const int c = c0 + i, s = i % T::NI;
    const uint32_t base = sb + T::RI + s * T::I_BYTES, full = bar(T::B_FULLI + s);
    const int t0 = c * C;
    uint32_t bytes = 2 * 8192 + C * P * 2 + C * T::W * 4 + C * C * 4;
    if (i == 0 && (p.test_flags & 1)) bytes += 16;  // test hook: this wait runs out (nothing faults)
    fast::mbar_expect_tx(full, bytes);
    fast::tma_load_5d(base + T::I_Q, &p.tm_q, 0, grp, 0, t0, b, full);
    fast::tma_load_5d(base + T::I_K, &p.tm_k, 0, grp, 0, t0, b, full);
    fast::tma_load_4d(base + T::I_V, &p.tm_v, 0, h, t0, b, full);
    fast::tma_load_4d(base + T::I_ANG, &p.tm_ang, 0, h, t0, b, full);
    fast::bulk_load(base + T::I_SEG, p.segsum + ((int64_t)bh * p.nc + c) * C * C, C * C * 4, full);
  };
  auto load_O = [&](int i) {
    const int c = c0 + i, s = i % T::NO;
    const uint32_t base = sb + T::RO + s * T::O_BYTES, full = bar(T::B_FULLO + s);
    const int t0 = c * C;
    fast::mbar_expect_tx(full, C * P * 2 * (HZ ? 2 : 1));
    fast::tma_load_4d(base + T::O_DOUT, &p.tm_dout, 0, h, t0, b, full);
    if (HZ) fast::tma_load_4d(base + T::O_Z, &p.tm_z, 0, h, t0, b, full);
  };
  const unsigned int flag_value = (p.tag << 8) | 0x5au;
  if (p.fused) {
    // =====================================================================
    // Phase A (single-kernel form): this segment's own state sum
    //   sum = sum_c gamma_c U_c,  gamma_c = prod_{c' > c in the segment} alpha_c',
    // U_c = PsiV_c^T k_state_c (tcgen05.mma), alpha_c = exp(da_cs[last valid
    // token of c]) -- the chunk recurrence state = alpha state + U unrolled
    // over the segment -- and its decay prod alpha_c, published for the
    // later segments of (b,h).  Four groups of four warps take every fourth
    // chunk (warp 4w + q: j-block q and tensor-memory lane quarter q of
    // group w); each keeps its partial sum in registers.  U_k is a
    // tcgen05.mma into the group's tensor-memory buffer k & 1 (columns
    // 64 (2w + (k & 1))), issued by the group's first thread once the four
    // warps wrote k_state and PsiV; the warps fold it one chunk later, so the
    // MMA runs under the next chunk's prologue.
    // =====================================================================
    const int na = c1 - c0;
    uint32_t* afac = reinterpret_cast<uint32_t*>(sm + T::A_FAC);
    float* aedr = reinterpret_cast<float*>(sm + T::A_EDR);
    float* agam = reinterpret_cast<float*>(sm + T::A_GAM);
    float* aalp = reinterpret_cast<float*>(sm + T::A_ALP);
    float* adec = reinterpret_cast<float*>(sm + T::A_DEC);
    float* ad4 = reinterpret_cast<float*>(sm + T::A_D4);
    // token scalars of the segment (the arithmetic of tok_fill)
    for (int e = threadIdx.x; e < na * C; e += T::NT) {
      const int tg = c0 * C + e;
      const int64_t ix = (int64_t)bh * p.S + tg;
      float dtv = 0.f, trv = 0.f, dtn = 0.f, trn = 0.f, arv = 0.f;
      if (tg < p.S) {
        dtv = __ldg(p.dt + ix);
        trv = bf_f(__ldg(p.trap + ix));
        arv = __ldg(p.da_cs_rev + ix);
      }
      if (tg + 1 < p.S) {
        dtn = __ldg(p.dt + ix + 1);
        trn = bf_f(__ldg(p.trap + ix + 1));
      }
      const float gam = __fmul_rn(round_bf(dtv), sigmoid_f(trv));
      float sh = 0.f;
      if (tg + 1 < p.nc * C) sh = round_bf(__fmul_rn(round_bf(dtn), 1.0f / (1.0f + expf(trn))));
      afac[e] = fast::dup_bf(__fadd_rn(gam, sh));
      aedr[e] = expf(arv);
    }
    for (int e = threadIdx.x; e < na; e += T::NT) {
      const int c = c0 + e;
      aalp[e] = expf(__ldg(p.da_cs + (int64_t)bh * p.S + min(c * C + C, p.S) - 1));
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // suffix products gamma_c, and the segment decay
      float gg = 1.f;
      for (int e = na - 1; e >= 0; e--) {
        agam[e] = gg;
        gg *= aalp[e];
      }
      *adec = gg;
    }
    // decay from a group's previous chunk through chunk e: prod of alpha over (e - 4, e]
    for (int e = threadIdx.x; e < na; e += T::NT)
      ad4[e] = e >= 4 ? ((aalp[e - 3] * aalp[e - 2]) * aalp[e - 1]) * aalp[e] : 1.f;
    __syncthreads();
    const int w = warp >> 2, q = warp & 3;
    const int kw = na > w ? (na - w + 3) / 4 : 0;  // chunks of group w: w + 4k
    const bool gl = (q == 0) && lane == 0;         // the group's MMA thread
    const bool gt = (q == 1) && lane == 0;         // the group's TMA thread
    const uint16_t* mvb = reinterpret_cast<const uint16_t*>(sm + T::MVB);
    RowRegs<T> kb;  // k bias pairs in registers
    kb.load(reinterpret_cast<const uint16_t*>(sm + T::KBS));
    const int tq = 4 * q + (g >> 1);  // the token (within a chunk) of this thread's fragment rows
    auto abuf = [&](int k) { return (uint32_t)(T::A_RAW + (w * 3 + k % 3) * T::A_BUF); };
    auto apsi = [&](int k) { return (uint32_t)(T::A_PSI + (w * 2 + (k & 1)) * 8192); };
    const uint32_t tl_lane = (uint32_t)(32 * q) << 16;
    auto load_A = [&](int k) {
      const int t0 = (c0 + w + 4 * k) * C;
      const uint32_t dst = sb + abuf(k), full = bar(T::B_AFULL + w * 3 + k % 3);
      uint32_t bytes = 8192 + C * P * 2 + C * T::W * 4;
      if (w == 0 && k == 0 && (p.test_flags & 1)) bytes += 16;  // test hook: this wait runs out
      fast::mbar_expect_tx(full, bytes);
      fast::tma_load_5d(dst + T::A_K, &p.tm_k, 0, grp, 0, t0, b, full);
      fast::tma_load_4d(dst + T::A_V, &p.tm_v, 0, h, t0, b, full);
      fast::tma_load_4d(dst + T::A_ANG, &p.tm_ang, 0, h, t0, b, full);
    };
    int loaded_a = 0, issued_a = 0;  // staging loads (TMA thread), U MMAs (MMA thread)
    if (gt) {
      loaded_a = min(3, kw);
      for (int k = 0; k < loaded_a; k++) load_A(k);
    }
    // acc: the group's running sum over its chunks c_0 < c_1 < ... (stride 4),
    // acc = (prod of alpha over (c_{k-1}, c_k]) acc + U_{c_k}, so that at the
    // end gamma_{c_last} acc = sum_k gamma_{c_k} U_{c_k}
    float acc[8][4];
#pragma unroll
    for (int nn = 0; nn < 8; nn++) acc[nn][0] = acc[nn][1] = acc[nn][2] = acc[nn][3] = 0.f;
    // fold U_k into acc: round(acc * decay) + U_k; then the buffer is free
    auto fold = [&](int k) -> bool {
      if (!__all_sync(kFull, wait_b(p, bar(T::B_AU + w * 2 + (k & 1)), (k >> 1) & 1, abort_flag, 4))) return false;
      // U_k is done: chunk k's staging buffer takes chunk k + 3
      if (gt && k + 3 < kw) {
        load_A(k + 3);
        loaded_a = k + 4;
      }
      const int i = w + 4 * k;
      // decay from the group's previous chunk through this one: prod of alpha over (c_{k-1}, c_k]
      const float dk = ad4[i];  // 1 for the group's first chunk (i < 4)
      fast::tm_fence_after();
      float u[8][4];
      fast::tm_ld_frag<8>(tmem + tl_lane + 64 * (w * 2 + (k & 1)), u);
      const float2 d2 = make_float2(dk, dk);
#pragma unroll
      for (int nn = 0; nn < 8; nn++) {
        const float2 x = __fadd2_rn(__fmul2_rn(make_float2(acc[nn][0], acc[nn][1]), d2), make_float2(u[nn][0], u[nn][1]));
        const float2 y = __fadd2_rn(__fmul2_rn(make_float2(acc[nn][2], acc[nn][3]), d2), make_float2(u[nn][2], u[nn][3]));
        acc[nn][0] = x.x; acc[nn][1] = x.y; acc[nn][2] = y.x; acc[nn][3] = y.y;
      }
      fast::tm_fence_before();
      __syncwarp();
      if (lane == 0) arrive(bar(T::B_AUF + w * 2 + (k & 1)));
      return true;
    };
    bool aok = true;
    for (int k = 0; aok && k < kw; k++) {
      const int i = w + 4 * k;
      unsigned char* bp = sm + abuf(k);
      if (!__all_sync(kFull, wait_b(p, bar(T::B_AFULL + w * 3 + k % 3), (k / 3) & 1, abort_flag, 1))) break;
      // the token's angles, factor and exp(da_cs_rev) in one round trip
      const float* ang = reinterpret_cast<const float*>(bp + T::A_ANG) + tq * T::W + 2 * cq;
      const float2 an0 = *reinterpret_cast<const float2*>(ang), an1 = *reinterpret_cast<const float2*>(ang + 8);
      const uint32_t fd = afac[i * C + tq];
      const float ed = aedr[i * C + tq];
      uint32_t kf[4][4];
      fast::load_rows<K>(kf, reinterpret_cast<const uint16_t*>(bp + T::A_K), 16 * q);
      add_bias_r(kf, kb.b);
      rotate_r<K>(kf, kf, false, an0, an1);
      scale_r(kf, fd);
      kstate_r(kf, ed);
      __syncwarp();  // this warp's raw k rows are read before k_state overwrites them
      fast::store_rows<K, true>(kf, reinterpret_cast<uint16_t*>(bp + T::A_K), 16 * q);
      // PsiV tile k & 1 was read by U_{k-2}, which the fold of k - 2 waited for
      fast::psi_rows<K>(reinterpret_cast<const uint16_t*>(bp + T::A_V), mvb,
                        reinterpret_cast<uint16_t*>(sm + apsi(k)), 16 * q);
      fast::fence_proxy_async();  // the MMA reads k_state and PsiV
      __syncwarp();
      if (lane == 0) arrive(bar(T::B_APA + w * 2 + (k & 1)));
      if (gl) {  // U_k, once the group's four warps are done and buffer k & 1 is folded
        aok = wait_b(p, bar(T::B_APA + w * 2 + (k & 1)), (k >> 1) & 1, abort_flag, 4) &&
              (k < 2 || wait_b(p, bar(T::B_AUF + w * 2 + (k & 1)), ((k - 2) >> 1) & 1, abort_flag, 4));
        if (aok) {
          fast::tm_fence_after();
          mma64<true, true>(tmem + 64 * (w * 2 + (k & 1)), sb + apsi(k), sb + abuf(k) + T::A_K);
          mma_commit(bar(T::B_AU + w * 2 + (k & 1)));
          issued_a = k + 1;
        }
      }
      aok = __all_sync(kFull, aok);
      if (aok && k >= 1) aok = fold(k - 1);
    }
    if (aok && kw > 0) aok = fold(kw - 1);
    __syncwarp();
    if (gl && issued_a > 0)  // the group's last MMA completes before the area and tensor memory are reused
      drain_wait(bar(T::B_AU + w * 2 + ((issued_a - 1) & 1)), ((issued_a - 1) >> 1) & 1);
    if (kw > 0) {
      const float gl_last = agam[w + 4 * (kw - 1)];
#pragma unroll
      for (int nn = 0; nn < 8; nn++)
#pragma unroll
        for (int e = 0; e < 4; e++) acc[nn][e] *= gl_last;
    }
    __syncwarp();
    if (gt && *abort_flag)  // every staging load landed before the area is reused
      for (int k = max(0, loaded_a - 3); k < loaded_a; k++) drain_wait(bar(T::B_AFULL + w * 3 + k % 3), (k / 3) & 1);
    __syncthreads();
    // the four group partials, summed in group order, published with a flag
    float* red4 = reinterpret_cast<float*>(sm + T::A_RAW);  // [4][N][P] FP32 over the staging area
    {
#pragma unroll
      for (int nn = 0; nn < 8; nn++)
#pragma unroll
        for (int e = 0; e < 4; e++)
          red4[w * N * P + (8 * nn + 2 * cq + (e & 1)) * P + 16 * q + g + 8 * (e >> 1)] = acc[nn][e];
    }
    __syncthreads();
    if (!*abort_flag) {
      if (seg + 1 < p.nseg) {  // (the last segment's sum is never needed)
        float* dsts = p.ws_state + ((int64_t)bh * p.nseg + seg) * N * P;
        for (int e = threadIdx.x; e < N * P; e += T::NT)
          dsts[e] = ((red4[e] + red4[N * P + e]) + red4[2 * N * P + e]) + red4[3 * N * P + e];
      }
      if (threadIdx.x == 0) {
        p.ws_decay[(int64_t)bh * p.nseg + seg] = *adec;
        if (seg == 0) p.ws_count[bh] = 0u;  // read by this head's CTAs after they saw this flag
      }
      __threadfence();
      __syncthreads();
      // (test hook, bit 2: the first segment of each head never publishes, so
      // the later segments' look-back runs out; nothing faults or hangs)
      if (threadIdx.x == 0 && !((p.test_flags & 4) && seg == 0))
        asm volatile("st.release.gpu.global.u32 [%0], %1;\n" ::"l"(p.ws_flag + (int64_t)bh * p.nseg + seg),
                     "r"(flag_value)
                     : "memory");
    }
    __syncthreads();
    if (*abort_flag) n = 0;  // phase A stopped: no phase C (the error word is set)
  }
  const int first_i = min(T::NI, n), first_o = min(T::NO, n);  // loads issued below (thread 0)
  if (threadIdx.x == 0) {
    for (int i = 0; i < first_i; i++) load_I(i);
    for (int i = 0; i < first_o; i++) load_O(i);
  }

  // ---- the state entering this segment: the segment sums of the earlier
  //      segments of (b,h) folded in order (acc = acc * decay_s + sum_s),
  //      every thread below 512 eight consecutive elements
  if (p.fused) {
    // the earlier segments of this head have published their sums (all CTAs
    // of a single-kernel launch are resident at once: a cooperative launch)
    for (int s2 = threadIdx.x; n > 0 && s2 < seg; s2 += T::NT) {
      const unsigned int* f = p.ws_flag + (int64_t)bh * p.nseg + s2;
      const uint64_t t0 = fast::global_ns();
      while (true) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(f) : "memory");
        if (v == flag_value) break;
        if (*abort_flag) break;
        if (fast::global_ns() - t0 > fast::kWaitLimitNs) {
          *abort_flag = 1u;
          atomicExch(p.ws_err, (p.tag << 8) | 5u);
          break;
        }
        __nanosleep(128);
      }
    }
    __syncthreads();
    if (*abort_flag) {  // a wait ran out: no phase C; the first loads land before the CTA leaves
      if (threadIdx.x == 0) {
        for (int i = 0; i < first_i; i++) drain_wait(bar(T::B_FULLI + i), 0);
        for (int i = 0; i < first_o; i++) drain_wait(bar(T::B_FULLO + i), 0);
      }
      n = 0;
    }
  } else {
    fast::pdl_wait();
  }
  float* xs = reinterpret_cast<float*>(sm + T::SBT);  // 16 KB scratch (SB and A tiles are unused yet)
  if (threadIdx.x < 512) {
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    const float* base = p.ws_state + (int64_t)bh * p.nseg * N * P + threadIdx.x * 8;
    const float* dec = p.ws_decay + (int64_t)bh * p.nseg;
    for (int s0 = 0; s0 < seg; s0 += 8) {
      float4 x0[8], x1[8];
      float d[8];
#pragma unroll
      for (int q = 0; q < 8; q++) {
        if (s0 + q < seg) {
          const float4* src = reinterpret_cast<const float4*>(base + (int64_t)(s0 + q) * N * P);
          x0[q] = __ldcg(src);
          x1[q] = __ldcg(src + 1);
          d[q] = __ldcg(dec + s0 + q);
        }
      }
#pragma unroll
      for (int q = 0; q < 8; q++) {
        if (s0 + q < seg) {
          a0 = make_float4(fmaf(a0.x, d[q], x0[q].x), fmaf(a0.y, d[q], x0[q].y), fmaf(a0.z, d[q], x0[q].z),
                           fmaf(a0.w, d[q], x0[q].w));
          a1 = make_float4(fmaf(a1.x, d[q], x1[q].x), fmaf(a1.y, d[q], x1[q].y), fmaf(a1.z, d[q], x1[q].z),
                           fmaf(a1.w, d[q], x1[q].w));
        }
      }
    }
    reinterpret_cast<float4*>(xs)[2 * threadIdx.x] = a0;
    reinterpret_cast<float4*>(xs)[2 * threadIdx.x + 1] = a1;
  }
  __syncthreads();
  // State warps: their FP32 state^T slice (p-block q, all n) in the 16x256b
  // fragment layout: st[nn][e] = state[n = 8nn + 2cq + (e&1)][p = 16q + g + 8(e>>1)].
  float st[8][4];
  if (warp >= T::WS && warp < T::WM) {
    const int q = warp - T::WS;
#pragma unroll
    for (int nn = 0; nn < 8; nn++)
#pragma unroll
      for (int e = 0; e < 4; e++) st[nn][e] = xs[(8 * nn + 2 * cq + (e & 1)) * P + 16 * q + g + 8 * (e >> 1)];
  }
  __syncthreads();  // the scratch is read before any tile is written

  float* tokb = reinterpret_cast<float*>(sm + T::TOK);
  auto tok_of = [&](int i) { return tokb + (i % (2 * T::TW)) * T::TS; };
  auto decay_of = [&](int i) {  // exp(da_cs[last valid token of chunk c0 + i])
    const int c = c0 + i;
    return tok_of(i)[2 * C + min(c * C + C, p.S) - 1 - c * C];
  };

  if (warp < T::WP) {
    // =====================================================================
    // Epilogue warps: pure compute on chunks whose inter^T / intra^T are in
    // tensor memory; dz goes straight to global memory.
    // =====================================================================
    const int q = warp & 3, hc = warp >> 2;
    const uint32_t tl_lane = (uint32_t)(32 * q) << 16;
    float2 mzr[4];
    uint32_t mor[4];
    {
      const float2* mzp = reinterpret_cast<const float2*>(sm + T::MZP);
      const uint32_t* mop = reinterpret_cast<const uint32_t*>(sm + T::MOP);
#pragma unroll
      for (int o = 0; o < 4; o++) {
        mzr[o] = HZ ? mzp[(o * 4 + q) * 8 + g] : make_float2(0.f, 0.f);
        mor[o] = mop[(o * 4 + q) * 8 + g];
      }
    }
    const float dval = HD ? p.d[h] : 0.f;
    float2 cdmo[4], cdmz[4];
#pragma unroll
    for (int o = 0; o < 4; o++) cdmo[o] = cdmz[o] = make_float2(0.f, 0.f);
    // the first two chunks' tensor-memory buffers are free from the start
    if (lane == 0) {
      if (n > 0) arrive(bar(T::B_SBR));
      if (n > 1) arrive(bar(T::B_SBR + 1));
    }
    for (int i = 0; i < n; i++) {
      const int c = c0 + i, so = i % T::NO, s2 = i & 1;
      unsigned char* op = sm + T::RO + so * T::O_BYTES;
      if (!__all_sync(kFull, wait_b(p, bar(T::B_M2 + s2), (i >> 1) & 1, abort_flag, 3))) break;
      if (!__all_sync(kFull, wait_b(p, bar(T::B_PDONE + i % T::NI), (i / T::NI) & 1, abort_flag, 3))) break;
      if (!__all_sync(kFull, wait_b(p, bar(T::B_FULLO + so), (i / T::NO) & 1, abort_flag, 1))) break;
      fast::tm_fence_after();
      float vi[4][4], vx[4][4];
      fast::tm_ld_frag<4>(tmem + tl_lane + T::T_I + 64 * s2 + 32 * hc, vi);
      fast::tm_ld_frag<4>(tmem + tl_lane + T::T_X + 64 * s2 + 32 * hc, vx);
      fast::tm_fence_before();
      __syncwarp();
      if (lane == 0 && i + 2 < n) arrive(bar(T::B_SBR + s2));  // this parity's buffers take chunk c + 2
      const float* tok = tok_of(i);
      const uint16_t* psi = reinterpret_cast<const uint16_t*>(op + T::O_PSI);
      const uint32_t* qkd = reinterpret_cast<const uint32_t*>(op + T::O_QKD);
      const uint16_t* zt = reinterpret_cast<const uint16_t*>(op + T::O_Z);
      const uint16_t* dt_ = reinterpret_cast<const uint16_t*>(op + T::O_DOUT);
#pragma unroll
      for (int tt = 0; tt < 2; tt++) {
        const int jb = 2 * hc + tt, tl = 4 * jb + cq;
        const float gam = tok[tl], ed = tok[2 * C + tl];
        const float2 gam2 = make_float2(gam, gam), ed2 = make_float2(ed, ed);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(a0, a1, a2, a3, psi + fast::swz128(16 * jb + (mi >> 1) * 8 + li, 16 * q + (mi & 1) * 8));
        uint32_t ps[4];  // PsiV of rank o at (p, p + 8)
        ps[0] = fast::lo_lo(a0, a1);
        ps[1] = fast::hi_hi(a0, a1);
        ps[2] = fast::lo_lo(a2, a3);
        ps[3] = fast::hi_hi(a2, a3);
        uint32_t qr[4][4];  // same-token bf16(qh . kh)[o][r], both halves
#pragma unroll
        for (int o = 0; o < 4; o++) {
          const uint4 v = *reinterpret_cast<const uint4*>(qkd + tl * T::QKS + o * 4);
          qr[o][0] = v.x; qr[o][1] = v.y; qr[o][2] = v.z; qr[o][3] = v.w;
        }
        const int pr = 16 * q + g;
        float2 z2 = make_float2(0.f, 0.f);
        if (HZ) z2 = fast::unpack2((uint32_t)zt[fast::swz128(tl, pr)] | ((uint32_t)zt[fast::swz128(tl, pr + 8)] << 16));
        const uint32_t dob =
            (uint32_t)dt_[fast::swz128(tl, pr)] | ((uint32_t)dt_[fast::swz128(tl, pr + 8)] << 16);
        uint32_t dzacc = 0u;
#pragma unroll
        for (int o = 0; o < 4; o++) {
          const int kk = 2 * tt + (o >> 1), bb = o & 1;
          // diagonal: rank-ordered BF16 products and sums, then * gamma, rounded
          uint32_t dacc = bmul2(qr[o][0], ps[0]);
#pragma unroll
          for (int r = 1; r < R; r++) dacc = badd2(dacc, bmul2(qr[o][r], ps[r]));
          const uint32_t dgb = fast::pack2(__fmul2_rn(fast::unpack2(dacc), gam2));
          // out = bf16(inter * exp(da_cs) + intra + diag + d * PsiV)
          float2 x = __ffma2_rn(make_float2(vi[kk][bb], vi[kk][bb + 2]), ed2, make_float2(vx[kk][bb], vx[kk][bb + 2]));
          x = fast::add_bf2_f32(dgb, x);
          if (HD) x = __ffma2_rn(make_float2(dval, dval), fast::unpack2(ps[o]), x);
          const uint32_t ob = fast::pack2(x);
          if (HZ) {
            const float2 mz = mzr[o];
            const float2 pz = __fmul2_rn(z2, mz);
            const float2 tq = __fmul2_rn(pz, make_float2(-fast::kLog2e, -fast::kLog2e));
            const float2 den =
                __fadd2_rn(make_float2(fast::ex2_approx(tq.x), fast::ex2_approx(tq.y)), make_float2(1.f, 1.f));
            const float2 sg = make_float2(fast::rcp_approx(den.x), fast::rcp_approx(den.y));
            const float2 silu = __fmul2_rn(pz, sg);
            // dmimo_o partials: out * dout (exact) * silu(pz)
            const float2 od = fast::fma_bf2_f32(ob, dob, make_float2(-0.f, -0.f));
            cdmo[o] = __ffma2_rn(od, silu, cdmo[o]);
            const uint32_t preb = bmul2(bmul2(dob, mor[o]), ob);
            const float2 pre = fast::unpack2(preb);
            // sigmoid(pz) (1 + pz (1 - sigmoid(pz))) = sigmoid + silu (1 - sigmoid)
            const float2 om = __fadd2_rn(make_float2(1.f, 1.f), make_float2(-sg.x, -sg.y));
            const float2 gz = __fmul2_rn(pre, __ffma2_rn(silu, om, sg));
            cdmz[o] = __ffma2_rn(gz, z2, cdmz[o]);
            // dz: BF16 running sum over the ranks in order
            dzacc = fast::pack2(fast::add_bf2_f32(dzacc, __fmul2_rn(gz, mz)));
          } else {
            cdmo[o] = fast::fma_bf2_f32(ob, dob, cdmo[o]);
          }
        }
        const int tg = c * C + tl;
        if (HZ && tg < p.S) {  // dz[b, t, h, p] and [.., p + 8]
          uint16_t* dzp = p.dz + (((int64_t)b * p.S + tg) * p.H + h) * P + pr;
          dzp[0] = (uint16_t)(dzacc & 0xffffu);
          dzp[8] = (uint16_t)(dzacc >> 16);
        }
      }
      // this warp is done with the chunk's ring O slot
      __syncwarp();
      if (lane == 0) arrive(bar(T::B_OFREE + so));
    }
    // ---- fixed-order reduction of the dmimo partials of this segment:
    //      the four lanes of a row group (tokens), then the two warps of a
    //      p-block (token halves)
#pragma unroll
    for (int o = 0; o < 4; o++) {
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        cdmo[o].x += __shfl_xor_sync(0xffffffffu, cdmo[o].x, m);
        cdmo[o].y += __shfl_xor_sync(0xffffffffu, cdmo[o].y, m);
        cdmz[o].x += __shfl_xor_sync(0xffffffffu, cdmz[o].x, m);
        cdmz[o].y += __shfl_xor_sync(0xffffffffu, cdmz[o].y, m);
      }
    }
    // red[hc][which][o][p] (FP32, 2 x 2 x 4 x 64) in ring I slot 0 (idle now)
    // after the barrier below
    __syncwarp();
    fast::tm_fence_before();
    __syncthreads();  // (A) every role has left its loop
    float* red = reinterpret_cast<float*>(sm + T::RI);
    if (cq == 0) {
#pragma unroll
      for (int o = 0; o < 4; o++) {
        const int pr = 16 * q + g;
        red[((hc * 2 + 0) * 4 + o) * P + pr] = cdmo[o].x;
        red[((hc * 2 + 0) * 4 + o) * P + pr + 8] = cdmo[o].y;
        red[((hc * 2 + 1) * 4 + o) * P + pr] = cdmz[o].x;
        red[((hc * 2 + 1) * 4 + o) * P + pr + 8] = cdmz[o].y;
      }
    }
  } else if (warp < T::WS) {
    // =====================================================================
    // Prologue warps: one 16-row j-block each.  Thread 0 of warp 8 also
    // loads dout and z into ring O slots the epilogue has released.
    // =====================================================================
    const int jw = warp - T::WP, j0 = 16 * jw, pt = threadIdx.x - T::WP * 32;
    const bool load_thread = pt == 0;  // issues the ring O loads
    int loaded_o = min(T::NO, n);
    const int tq = (j0 >> 2) + (g >> 1);  // the token (within a chunk) of this thread's fragment rows

    const uint16_t* mvb = reinterpret_cast<const uint16_t*>(sm + T::MVB);
    fast::TokRaw traw = tok_load<T>(p, bh, c0, pt);
    for (int i = 0; i < n; i++) {
      const int c = c0 + i, si = i % T::NI, so = i % T::NO;
      unsigned char* ip = sm + T::RI + si * T::I_BYTES;
      unsigned char* op = sm + T::RO + so * T::O_BYTES;
      if (i % T::TW == 0) {  // token scalars of the window starting at chunk c
        const int wi = i / T::TW;
        tok_fill<T>(p, traw, tokb + (wi & 1) * T::TW * T::TS, c, pt);
        if (c + T::TW < c1) traw = tok_load<T>(p, bh, c + T::TW, pt);
        __syncwarp();
        if (lane == 0) arrive(bar(T::B_TOKW + (wi & 1)));
        if (!__all_sync(kFull, wait_b(p, bar(T::B_TOKW + (wi & 1)), (wi >> 1) & 1, abort_flag, 4)))
          break;
      }
      const float* tok = tok_of(i);
      if (!__all_sync(kFull, wait_b(p, bar(T::B_FULLI + si), (i / T::NI) & 1, abort_flag, 1)))
        break;
      if (!__all_sync(kFull, i < T::NO || wait_b(p, bar(T::B_OFREE + so), ((i / T::NO) - 1) & 1, abort_flag, 4)))
        break;
      if (load_thread && i >= T::NO) {  // the epilogue is done with this ring O slot: dout, z of chunk c
        fast::fence_proxy_async();
        load_O(i);
        loaded_o = i + 1;
      }
      uint16_t* qt = reinterpret_cast<uint16_t*>(ip + T::I_Q);
      uint16_t* kt = reinterpret_cast<uint16_t*>(ip + T::I_K);
      // every per-chunk scalar in one shared-memory round trip: the biases,
      // the token's angles, factor and exp(da_cs_rev)
      RowRegs<T> qb, kb;
      qb.load(reinterpret_cast<const uint16_t*>(sm + T::QBS));
      kb.load(reinterpret_cast<const uint16_t*>(sm + T::KBS));
      const float* ang = reinterpret_cast<const float*>(ip + T::I_ANG) + tq * T::W + 2 * cq;
      const float2 an0 = *reinterpret_cast<const float2*>(ang), an1 = *reinterpret_cast<const float2*>(ang + 8);
      const uint32_t fd = reinterpret_cast<const uint32_t*>(tok)[C + tq];
      const float ed = tok[3 * C + tq];
      uint32_t qf[4][4], kf[4][4];
      fast::load_rows<K>(qf, qt, j0);
      fast::load_rows<K>(kf, kt, j0);
      add_bias_r(qf, qb.b);  // bf16(q + bf16(bias)), bf16(k + bf16(bias))
      add_bias_r(kf, kb.b);
      {  // same-token qk_dot from the diagonal 16x16 tile of Qh Kh^T
        uint32_t* qkd = reinterpret_cast<uint32_t*>(op + T::O_QKD);
        float qa[2][4];
#pragma unroll
        for (int ht = 0; ht < 2; ht++) qa[ht][0] = qa[ht][1] = qa[ht][2] = qa[ht][3] = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < 4; k4++) {
          mma16816(qa[0], qf[k4][0], qf[k4][1], qf[k4][2], qf[k4][3], kf[k4][0], kf[k4][2]);
          mma16816(qa[1], qf[k4][0], qf[k4][1], qf[k4][2], qf[k4][3], kf[k4][1], kf[k4][3]);
        }
        // Fragment rows g, g + 8 are ranks 2hh + (g & 1) of token g / 2 of the
        // block, columns 2 cq, 2 cq + 1 of tile ht ranks 2ht, 2ht + 1 of token
        // cq: the lanes with g / 2 = cq hold token 4 jw + cq's qk values, ranks
        // o = (g & 1) and 2 + (g & 1), all four columns.  Each writes two rows
        // of the token's [R][R] block: the BF16 table for the epilogue (both
        // halves), and the output.
        if ((g >> 1) == cq) {
          const int tl = 4 * jw + cq;
          const bool inb = c * C + tl < p.S;
          uint32_t* qrow = qkd + tl * T::QKS;
          uint2* grow = reinterpret_cast<uint2*>(p.qk_dot + ((int64_t)bh * p.S + c * C + tl) * (R * R));
#pragma unroll
          for (int hh = 0; hh < 2; hh++) {
            const int o = 2 * hh + (g & 1);
            const uint32_t v0 = f_bf(qa[0][2 * hh]), v1 = f_bf(qa[0][2 * hh + 1]);
            const uint32_t v2 = f_bf(qa[1][2 * hh]), v3 = f_bf(qa[1][2 * hh + 1]);
            *reinterpret_cast<uint4*>(qrow + o * R) =
                make_uint4(v0 | (v0 << 16), v1 | (v1 << 16), v2 | (v2 << 16), v3 | (v3 << 16));
            if (inb) grow[o] = make_uint2(v0 | (v1 << 16), v2 | (v3 << 16));
          }
        }
      }
      rotate_r<K>(qf, kf, true, an0, an1);
      __syncwarp();  // this warp's raw q / k rows are read before they are overwritten
      fast::store_rows<K, true>(qf, qt, j0);  // Q_rot, rows in fragment order
      scale_r(kf, fd);
      fast::store_rows<K, true>(kf, kt, j0);  // k_scaled
      kstate_r(kf, ed);
      fast::store_rows<K, true>(kf, reinterpret_cast<uint16_t*>(ip + T::I_KST), j0);
      // PsiV = bf16(v * bf16(mimo_v)), this warp's rows, into the ring O slot
      fast::psi_rows<K, 16>(reinterpret_cast<const uint16_t*>(ip + T::I_V), mvb,
                            reinterpret_cast<uint16_t*>(op + T::O_PSI), j0);
      fast::fence_proxy_async();
      __syncwarp();
      if (lane == 0) arrive(bar(T::B_PDONE + si));
    }
    __syncwarp();
    if (load_thread && *abort_flag)  // after an abort: the ring O loads in flight land first
      for (int i = max(0, loaded_o - T::NO); i < loaded_o; i++) {
        const uint32_t bf = bar(T::B_FULLO + i % T::NO), ph = (i / T::NO) & 1;
        drain_wait(bf, ph);
      }
    __syncwarp();
    fast::tm_fence_before();
    __syncthreads();  // (A)
  } else if (warp < T::WM) {
    // =====================================================================
    // State warps: p-block q of the FP32 state in registers and rows 16q..
    // of the causal matrix.  Per chunk c: the state entering c, folded from
    // the one entering c - 1 and U of chunk c - 1 (tensor memory; its MMA
    // went out with chunk c - 2's products, so it is long done); bf16 of it
    // for inter^T and the states output; A = bf16(mask(Q_rot Ks^T)
    // exp(segsum)) for j-block q (mma.sync on the prologue's tiles, causal
    // blocks only).  Then the chunk's MMAs go out from the two warps with the
    // fewest A blocks, one accumulator per issuing thread (an issue stalls
    // its thread for about the MMA's run time): warp 12's first thread the
    // states store, inter^T, then U of the next chunk (its own barrier, so
    // that the epilogue of c never waits for the prologue of c + 1), warp
    // 13's intra^T.  Only the fold is serial from chunk to chunk.
    // =====================================================================
    const int q = warp - T::WS;
    const int mma_role = lane != 0 ? -1 : q < 2 ? q : -1;  // 0 store, inter, U; 1 intra
    int last_m = -1, last_u = -1;  // last chunk this thread committed products / U for
    const bool loader = threadIdx.x == T::WS * 32 + 96;  // refills ring I
    int loaded_i = min(T::NI, n);                        // ring I chunks issued
    const uint32_t tl_lane = (uint32_t)(32 * q) << 16;
    {  // blocks of A above the token-block diagonal stay 0 (both buffers)
      uint16_t* at = reinterpret_cast<uint16_t*>(sm + T::ATT);
      for (int e = lane; e < 2 * 16 * 8; e += 32) {  // 2 buffers x 16 rows x 8 chunks of 16 bytes
        const int bf = e / 128, r = (e / 8) % 16, ch = e % 8;
        if (ch >= 2 * (q + 1))
          *reinterpret_cast<uint4*>(at + bf * 4096 + fast::swz128(16 * q + r, ch * 8)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // U of the first chunk: PsiV^T k_state, into tensor-memory buffer 0
    bool alive = true;
    if (mma_role == 0 && n > 0) {
      alive = wait_b(p, bar(T::B_PDONE), 0, abort_flag, 2);
      if (alive) {
        fast::tm_fence_after();
        mma64<true, true>(tmem + T::T_U, sb + T::RO + T::O_PSI, sb + T::RI + T::I_KST);
        mma_commit(bar(T::B_U));
        last_u = 0;
      }
    }
    alive = __all_sync(kFull, alive);
    for (int i = 0; alive && i < n; i++) {
      const int c = c0 + i, s2 = i & 1, si = i % T::NI, so = i % T::NO;
      unsigned char* ip = sm + T::RI + si * T::I_BYTES;
      // state entering chunk c = round(state * alpha_{c-1}) + U_{c-1} (FP32).
      // Chunk c - 2's MMAs are done: U_{c-1} is ready and the SB / A buffers
      // of this parity are free (and so is the states store that read SB).
      if (i >= 1) {
        if (!__all_sync(kFull, (i < 2 || wait_b(p, bar(T::B_M2 + s2), ((i - 2) >> 1) & 1, abort_flag, 2)) &&
                                   wait_b(p, bar(T::B_U + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, 2)))
          break;
        // chunk c - 2 is done with its ring I slot (prologue, A, every MMA):
        // it takes chunk c + 2
        if (loader && i >= 2 && i + 2 < n) {
          load_I(i + 2);
          loaded_i = i + 3;
        }
        fast::tm_fence_after();
        float u[8][4];
        fast::tm_ld_frag<8>(tmem + tl_lane + T::T_U + 64 * ((i - 1) & 1), u);
        const float a = decay_of(i - 1);
        const float2 a2 = make_float2(a, a);
#pragma unroll
        for (int nn = 0; nn < 8; nn++) {
          const float2 x = __fadd2_rn(__fmul2_rn(make_float2(st[nn][0], st[nn][1]), a2), make_float2(u[nn][0], u[nn][1]));
          const float2 y = __fadd2_rn(__fmul2_rn(make_float2(st[nn][2], st[nn][3]), a2), make_float2(u[nn][2], u[nn][3]));
          st[nn][0] = x.x; st[nn][1] = x.y; st[nn][2] = y.x; st[nn][3] = y.y;
        }
      }
      uint16_t* sbt = reinterpret_cast<uint16_t*>(sm + T::SBT + s2 * 8192);
#pragma unroll
      for (int nn = 0; nn < 4; nn++) {
        const uint32_t r0 = fast::pack2(make_float2(st[2 * nn][0], st[2 * nn][1]));
        const uint32_t r1 = fast::pack2(make_float2(st[2 * nn][2], st[2 * nn][3]));
        const uint32_t r2 = fast::pack2(make_float2(st[2 * nn + 1][0], st[2 * nn + 1][1]));
        const uint32_t r3 = fast::pack2(make_float2(st[2 * nn + 1][2], st[2 * nn + 1][3]));
        fast::stsm_x4_t(sbt + fast::swz128(nn * 16 + (mi >> 1) * 8 + li, q * 16 + (mi & 1) * 8), r0, r1, r2, r3);
      }
      // the prologue of chunk c is done: Q_rot, k_scaled for A
      if (!__all_sync(kFull, wait_b(p, bar(T::B_PDONE + si), (i / T::NI) & 1, abort_flag, 2))) break;
      {  // A rows 16q..: S = Q_rot Ks^T on causal blocks jb <= q, rows and columns in tile order
        const uint16_t* qt = reinterpret_cast<const uint16_t*>(ip + T::I_Q);
        const uint16_t* kt = reinterpret_cast<const uint16_t*>(ip + T::I_K);
        const float* es = reinterpret_cast<const float*>(ip + T::I_SEG);
        uint16_t* at = reinterpret_cast<uint16_t*>(sm + T::ATT + s2 * 8192);
        uint32_t qf[4][4];
#pragma unroll
        for (int k4 = 0; k4 < 4; k4++)
          ldsm_x4(qf[k4][0], qf[k4][1], qf[k4][2], qf[k4][3],
                  qt + fast::swz128(16 * q + (lane & 15), k4 * 16 + (lane >> 4) * 8));
        const int trow = 4 * q + (g >> 1);
        for (int jb = 0; jb <= q; jb++) {
          float sa[2][4];
#pragma unroll
          for (int ht = 0; ht < 2; ht++) sa[ht][0] = sa[ht][1] = sa[ht][2] = sa[ht][3] = 0.f;
#pragma unroll
          for (int k4 = 0; k4 < 4; k4++) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3, kt + fast::swz128(16 * jb + (mi >> 1) * 8 + li, k4 * 16 + (mi & 1) * 8));
            mma16816(sa[0], qf[k4][0], qf[k4][1], qf[k4][2], qf[k4][3], b0, b1);
            mma16816(sa[1], qf[k4][0], qf[k4][1], qf[k4][2], qf[k4][3], b2, b3);
          }
          // exp(segsum) of (row token, column token) if the row's token is
          // later, else 0 (a select: the entries on and above the diagonal
          // are never read)
          const int tcol = 4 * jb + cq;
          const float e = trow > tcol ? fast::exp_fast(es[trow * C + tcol]) : 0.f;
          const float2 e2 = make_float2(e, e);
          const uint32_t r0 = fast::pack2(__fmul2_rn(make_float2(sa[0][0], sa[0][1]), e2));
          const uint32_t r1 = fast::pack2(__fmul2_rn(make_float2(sa[0][2], sa[0][3]), e2));
          const uint32_t r2 = fast::pack2(__fmul2_rn(make_float2(sa[1][0], sa[1][1]), e2));
          const uint32_t r3 = fast::pack2(__fmul2_rn(make_float2(sa[1][2], sa[1][3]), e2));
          fast::stsm_x4(at + fast::swz128(16 * q + li + 8 * (mi & 1), 16 * jb + 8 * (mi >> 1)), r0, r1, r2, r3);
        }
      }
      fast::tm_fence_before();    // U_{c-1} is read before its buffer takes U_{c+1}
      fast::fence_proxy_async();  // SB and A tiles before the MMAs and the store read them
      __syncwarp();
      if (lane == 0) arrive(bar(T::B_SBR + s2));
      bool ok = true;
      if (mma_role >= 0) {
        // every state warp is done with chunk c (SB, A, U_{c-1} folded) and
        // the epilogue has read chunk c - 2's products
        ok = wait_b(p, bar(T::B_SBR + s2), (i >> 1) & 1, abort_flag, 2);
        if (ok) {
          fast::tm_fence_after();
          if (mma_role == 0) {
            // states[c] = bf16(state entering chunk c): one tile store
            fast::tma_store_2d(&p.tm_states, sb + T::SBT + s2 * 8192, 0, (int)(((int64_t)bh * p.nc + c) * N));
            mma64<true, false>(tmem + T::T_I + 64 * s2, sb + T::SBT + s2 * 8192,
                               sb + T::RI + si * T::I_BYTES + T::I_Q);
            asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");  // SB read before it is released
            mma_commit(bar(T::B_M2 + s2));
            last_m = i;
            if (i + 1 < n && (ok = wait_b(p, bar(T::B_PDONE + (i + 1) % T::NI), ((i + 1) / T::NI) & 1,
                                          abort_flag, 2))) {
              // U_{c+1} = PsiV_{c+1}^T k_state_{c+1} (their prologue is done)
              fast::tm_fence_after();
              mma64<true, true>(tmem + T::T_U + 64 * ((i + 1) & 1),
                                sb + T::RO + ((i + 1) % T::NO) * T::O_BYTES + T::O_PSI,
                                sb + T::RI + ((i + 1) % T::NI) * T::I_BYTES + T::I_KST);
              mma_commit(bar(T::B_U + ((i + 1) & 1)));
              last_u = i + 1;
            }
          } else {
            mma64<true, false>(tmem + T::T_X + 64 * s2, sb + T::RO + so * T::O_BYTES + T::O_PSI,
                               sb + T::ATT + s2 * 8192);
            mma_commit(bar(T::B_M2 + s2));
            last_m = i;
          }
        }
      }
      if (!__all_sync(kFull, ok)) break;
    }
    __syncwarp();
    if (mma_role == 0) fast::tma_store_wait_all();
    if (last_m >= 0)  // this thread's MMAs complete before tensor memory is released
      drain_wait(bar(T::B_M2 + (last_m & 1)), (last_m >> 1) & 1);
    if (last_u >= 0) drain_wait(bar(T::B_U + (last_u & 1)), (last_u >> 1) & 1);
    __syncwarp();
    if (loader && *abort_flag)  // after an abort: the ring I loads in flight land first
      for (int i = max(0, loaded_i - T::NI); i < loaded_i; i++) drain_wait(bar(T::B_FULLI + i % T::NI), (i / T::NI) & 1);
    __syncwarp();
    fast::tm_fence_before();
    __syncthreads();  // (A)
  }

  // ---- (after barrier A) the dmimo partials of this segment; tensor memory released
  __syncthreads();  // (B) red[] complete
  if (warp == T::WS) {
    fast::tm_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem) : "memory");
  }
  const float* red = reinterpret_cast<const float*>(sm + T::RI);
  float* dst = p.ws_grad + ((int64_t)bh * p.nseg + seg) * 2 * R * P;
  for (int e = threadIdx.x; e < 2 * R * P; e += T::NT) {
    // e = which * R * P + o * P + pp; token halves summed in order
    dst[e] = red[e] + red[2 * R * P + e];
  }
  // The last CTA of this (b,h) to finish sums the segments' partials in
  // segment order (the result does not depend on which CTA is last).
  __threadfence();
  __syncthreads();
  unsigned int* last = reinterpret_cast<unsigned int*>(sm + T::MISC + 8);
  if (threadIdx.x == 0) *last = (atomicAdd(p.ws_count + bh, 1u) == (unsigned int)p.nseg - 1u) ? 1u : 0u;
  __syncthreads();
  if (*last) {
    __threadfence();
    for (int e = threadIdx.x; e < 2 * R * P; e += T::NT) {
      const float* src = p.ws_grad + (int64_t)bh * p.nseg * 2 * R * P + e;
      float sum = 0.f;
      for (int s = 0; s < p.nseg; s++) sum += __ldcg(src + (int64_t)s * 2 * R * P);
      const int which = e / (R * P), x = e % (R * P);
      if (which == 0) p.dmimo_o[(int64_t)bh * R * P + x] = sum;
      if (which == 1 && HZ) p.dmimo_z[(int64_t)bh * R * P + x] = sum;
    }
  }
}

}  // namespace tc
