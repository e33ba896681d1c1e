// Fused chunked forward of the gated delta rule on the GB300 tensor cores.
//
// One CTA owns one (sequence, head, 64-wide slice of the value dimension) and
// walks that sequence's 64-token chunks in order ("Optimization Quartet",
// Triton GDN kernel section 3.2: intra-chunk parallel work, a serial carry of
// the state between chunks; chunk size 64 per "v1.0 Architecture & Design
// Spec" section 2.3).  The fp32 state never leaves the chip: it lives in the
// MMA accumulator registers of the carry warps for the whole sequence
// ("Model Architecture Walkthrough", section 6.3: state kept on chip).
//
// The chunk algebra (gated delta rule of Yang et al., arXiv 2412.06464) in the
// transposed-state form H = S^T (dk x dv), with G the chunk-local prefix sum of
// the log-gates and Gamma_ij = exp(G_i - G_j) (the unrolled decay weight of
// "Model Architecture Walkthrough", section 5.3.1):
//   A  = strictly_lower(diag(beta) K K^T (.) Gamma),   P = (Q K^T (.) Gamma)_{i>=j}
//   (I + A) W  = diag(beta exp(G)) K,   (I + A) U~ = diag(beta) V
//   U  = U~ - W H0                      (the only products that involve the state)
//   O  = diag(exp(G)) Q H0 + P U
//   H' = exp(G_C) H0 + (diag(exp(G_C - G)) K)^T U
//
// Roles (320 threads, one CTA per SM):
//   warp 8    producer: per chunk, the gate vectors (prefix sums of the
//             log-gates, their exponentials, beta) from plain loads prefetched
//             a chunk ahead, then TMA loads of the Q, K, V tiles into a ring of
//             input slots (mbarrier completion with transaction bytes).
//   warp 9    MMA issuer: allocates tensor memory, and per chunk issues one
//             tcgen05.mma chain [Q; K] K^T (M = 128, N = 64) straight from the
//             TMA-written shared tiles into a double-buffered TMEM accumulator.
//   warps 0-3 prep: per chunk, 16x16 diagonal blocks of (I + A)^-1 in fp32,
//             their off-diagonal couplings on tf32 tensor cores, and a blocked
//             forward substitution on bf16 tensor cores that yields W and U~
//             for the carry (2-stage ring).
//   warps 4-7 carry: each warp owns 16 value columns and keeps H^T for them in
//             registers (fp32); the serial chain U -> H' never leaves the warp
//             (MMA accumulators are re-packed in registers as the bf16 A
//             operands of the next products).  Forms O and stores it with
//             coalesced 16-byte stores.  Between chunks these warps also drain
//             the TMEM accumulator of chunk c+2 (decay mask, P and A rows),
//             which balances the two warp groups.
// Every wait on an mbarrier is bounded; on timeout the kernel records
// GDN_ERR_TIMEOUT in the status word and the roles leave their loops.
#include "gdn_tc_common.cuh"

namespace gdn {

namespace {

using namespace ptx;
using namespace tc;

constexpr int kPrepThreads = 128;
constexpr int kCarryThreads = 128;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kTcThreads = 320;
constexpr uint32_t kBarPrep = 1, kBarCarry = 2;
constexpr uint32_t kTmemCols = 128;  // two 64-column fp32 accumulators
constexpr uint32_t kIdescS = umma_idesc_bf16(128, 64);

template <int DK, int NIN>
struct TcLayout {
  // Input slot: Q and K sub-tiles interleaved [Q0 K0 Q1 K1] (each [64][64] bf16,
  // 128-byte swizzle) so that [Q; K] is one 128-row MMA operand per 64-column
  // sub-tile; then V, then the gate vectors.
  static constexpr int SUB = 8192;
  static constexpr int QK_PAIR = 2 * SUB;
  static constexpr int OFF_V = (DK / 64) * QK_PAIR;
  static constexpr int OFF_GATE = OFF_V + SUB;
  // f32 [8][64]: G*log2e, gamma, decay-to-end, beta, E, output gate (kFEpi)
  static constexpr int GATE = 2048;
  static constexpr int SLOT = OFF_GATE + GATE;
  static constexpr int STAGE = (DK / 64) * SUB + 2 * SUB;  // W, U~, P of one chunk
  static constexpr int OFF_IN = 0;
  static constexpr int OFF_ST = OFF_IN + NIN * SLOT;
  static constexpr int OFF_OST = OFF_ST + 2 * STAGE;  // three O staging tiles
  static constexpr int A_LD = 68;
  static constexpr int OFF_A = OFF_OST + 3 * SUB;       // f32 [2][64][A_LD]
  static constexpr int TF_LD = 20;                       // f32 row stride (80 B)
  static constexpr int OFF_TF = OFF_A + 2 * 64 * A_LD * 4;  // f32 [4][16][TF_LD]
  static constexpr int TB_LD = 24;                       // bf16 row stride (48 B)
  static constexpr int OFF_TB = OFF_TF + 4 * 16 * TF_LD * 4;      // bf16 [2][4][16][TB_LD]
  static constexpr int OFF_MB = OFF_TB + 2 * 4 * 16 * TB_LD * 2;  // bf16 [6][16][TB_LD]
  static constexpr int OFF_GC = OFF_MB + 6 * 16 * TB_LD * 2;      // f32 [NIN] exp(G_C)
  static constexpr int OFF_VOTE = OFF_GC + 64;                    // int [2 groups][2][4]
  static constexpr int OFF_TMEM = OFF_VOTE + 64;                  // u32 TMEM base
  static constexpr int OFF_BAR = OFF_TMEM + 16;
  static constexpr int NBAR = 2 * NIN + 10;
  static constexpr int OFF_FLAG = OFF_BAR + NBAR * 8;
  // kFL2 only: per input slot, fp32 vectors r_q [0,64), r_k [64,128),
  // G - log2 r_k [128,192) and E r_k [192,256); then the two mbarriers that
  // gather the drain threads' norms of a chunk
  static constexpr int RN_SLOT = 4 * 64;
  static constexpr int OFF_RN = OFF_FLAG + 16;
  static constexpr int OFF_NBAR = OFF_RN + NIN * RN_SLOT * 4;
  static constexpr int BYTES = OFF_NBAR + 16;
  static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
  static_assert(SLOT % 1024 == 0 && STAGE % 1024 == 0, "tiles need 1024-byte alignment");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Fused GDN block parts, as in the head_dim_k = 64 kernel: beta logits in
// every instance; the mask kF selects the instance with the q/k L2
// normalisation folded into fp32 row factors and column vectors (kFL2) and
// the one with the output epilogue (kFEpi), so that the plain pass carries
// none of their code.
constexpr int kFL2 = 1, kFEpi = 2;

template <int DK, int NIN, int kF>
__global__ void __launch_bounds__(kTcThreads, 1)
gdn_fwd_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_o) {
  using L = TcLayout<DK, NIN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv, col0 = tile * kDvt;

  int64_t start, len;
  if (!sequence_bounds(p, n, h, start, len)) return;  // uniform over the CTA
  if ((p.flags & GDN_DEBUG_CHECKS) &&
      !debug_ranges_ok(p, n, h, start, len, col0, kDvt, 2, true))
    return;  // recorded; nothing was accessed
  if (len == 0) {   // an empty sequence: the state passes through
    pass_state_through(p, n, h, col0, kDvt);
    return;
  }
  const int nc = (int)((len + 63) / 64);

  Shared S;
  S.abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_FLAG);
  int *votes = reinterpret_cast<int *>(smem + L::OFF_VOTE);
  float *sgc = reinterpret_cast<float *>(smem + L::OFF_GC);
  auto bar = [&](int i) { return sbase + L::OFF_BAR + 8u * i; };
  auto full_in = [&](int s) { return bar(s); };
  auto empty_in = [&](int s) { return bar(NIN + s); };
  auto full_st = [&](int s) { return bar(2 * NIN + s); };
  auto empty_st = [&](int s) { return bar(2 * NIN + 2 + s); };
  auto tmem_full = [&](int s) { return bar(2 * NIN + 4 + s); };
  auto tmem_empty = [&](int s) { return bar(2 * NIN + 6 + s); };
  auto s_ready = [&](int s) { return bar(2 * NIN + 8 + s); };
  auto slot_base = [&](int s) { return sbase + L::OFF_IN + s * L::SLOT; };
  auto gate_ptr = [&](int s) {
    return reinterpret_cast<float *>(smem + L::OFF_IN + s * L::SLOT + L::OFF_GATE);
  };

  if (tid == 0) {
    for (int s = 0; s < NIN; ++s) {
      mbar_init(full_in(s), 1);
      mbar_init(empty_in(s), kCarryThreads);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(full_st(s), kPrepThreads);
      mbar_init(empty_st(s), kCarryThreads);
      mbar_init(tmem_full(s), 1);
      mbar_init(tmem_empty(s), kCarryThreads);
      mbar_init(s_ready(s), kCarryThreads);
    }
    if constexpr ((kF & kFL2) != 0) {
      mbar_init(sbase + L::OFF_NBAR, kCarryThreads);
      mbar_init(sbase + L::OFF_NBAR + 8, kCarryThreads);
    }
    *S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(sbase + L::OFF_TMEM, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(smem + L::OFF_TMEM);

  const int lrow = lane & 7, lmi = lane >> 3;  // ldmatrix: row within matrix, matrix index
  const int g = lane >> 2, t = lane & 3;       // mma fragment coordinates

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const __nv_bfloat16 *betap = static_cast<const __nv_bfloat16 *>(p.beta);
    float gv0 = 0.f, gv1 = 0.f, bv0 = 0.f, bv1 = 0.f, og0 = 1.f, og1 = 1.f;
    auto load_gates = [&](int c) {
      gv0 = gv1 = bv0 = bv1 = 0.f;
      og0 = og1 = 1.f;
      const int64_t t0 = (int64_t)c * 64 + 2 * lane;
      if (c < nc && t0 < len) {
        const size_t off = (size_t)(start + t0) * H + h;
        gv0 = p.g[off];
        bv0 = __bfloat162float(betap[off]);
        if (t0 + 1 < len) {
          gv1 = p.g[off + H];
          bv1 = __bfloat162float(betap[off + H]);
        }
        if constexpr ((kF & kFEpi) != 0) {
          if (p.out_gate) {
            og0 = p.out_gate[off];
            og1 = t0 + 1 < len ? p.out_gate[off + H] : 1.f;
          }
        }
        if (p.flags & GDN_BETA_LOGITS) {  // beta from logits (uniform branch, any instance)
          bv0 = beta_value(bv0, p.flags);
          bv1 = t0 + 1 < len ? beta_value(bv1, p.flags) : 0.f;
        }
      }
    };
    load_gates(0);
    constexpr uint32_t kTx = 2 * (DK / 64) * L::SUB + L::SUB;
    int issued = 0;
    for (int c = 0; c < nc; ++c) {
      const int slot = c % NIN;
      GDN_PHASE(0);
      bool ok = true;
      if (c >= NIN) ok = role_wait(empty_in(slot), ((c / NIN) - 1) & 1, S, p, n, h, 1);
      GDN_PHASE(1);
      if (!__all_sync(0xffffffffu, ok)) break;
      {
        // G (log2 units), gamma = 2^G, decay to the chunk end, beta, and
        // E_j = 2^(G_b - G_j) with b the last token of j's 16-token block.
        const float x0 = gv0 * kLog2e, x1 = gv1 * kLog2e;
        float s = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, s, off);
          if (lane >= off) s += y;
        }
        const float G0 = s - x1, G1 = s;
        const float Gl = __shfl_sync(0xffffffffu, G1, 31);
        const float Gb = __shfl_sync(0xffffffffu, G1, (lane & ~7) | 7);
        float *gate = gate_ptr(slot);
        *reinterpret_cast<float2 *>(gate + 2 * lane) = make_float2(G0, G1);
        *reinterpret_cast<float2 *>(gate + 64 + 2 * lane) = make_float2(ex2(G0), ex2(G1));
        *reinterpret_cast<float2 *>(gate + 128 + 2 * lane) =
            make_float2(ex2(Gl - G0), ex2(Gl - G1));
        *reinterpret_cast<float2 *>(gate + 192 + 2 * lane) = make_float2(bv0, bv1);
        *reinterpret_cast<float2 *>(gate + 256 + 2 * lane) =
            make_float2(ex2(Gb - G0), ex2(Gb - G1));
        if (lane == 0) sgc[slot] = ex2(Gl);
        if constexpr ((kF & kFEpi) != 0)
          *reinterpret_cast<float2 *>(gate + 320 + 2 * lane) = make_float2(og0, og1);
      }
      load_gates(c + 1);
      __syncwarp();
      if (lane == 0) {
        const uint32_t sb = slot_base(slot);
        const int row = (int)(start + (int64_t)c * 64);
        mbar_arrive_expect_tx(full_in(slot), kTx);
#pragma unroll
        for (int sub = 0; sub < DK / 64; ++sub) {
          tma_load_3d(sb + sub * L::QK_PAIR, &tmap_q, sub * 64, h, row, full_in(slot));
          tma_load_3d(sb + sub * L::QK_PAIR + L::SUB, &tmap_k, sub * 64, h, row, full_in(slot));
        }
        tma_load_3d(sb + L::OFF_V, &tmap_v, col0, h, row, full_in(slot));
      }
      GDN_PHASE(2);
      ++issued;
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (lane == 0)
      for (int c = issued - NIN < 0 ? 0 : issued - NIN; c < issued; ++c)
        mbar_wait_bounded(full_in(c % NIN), (c / NIN) & 1, kWaitTimeoutNs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nc; ++c) {
        const int slot = c % NIN, buf = c & 1;
        GDN_PHASE(0);
        bool ok = role_wait(full_in(slot), (c / NIN) & 1, S, p, n, h, 5);
        GDN_PHASE(1);
        if (ok && c >= 2) ok = role_wait(tmem_empty(buf), ((c >> 1) - 1) & 1, S, p, n, h, 6);
        GDN_PHASE(2);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sb = slot_base(slot);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t a = sb + (kk >> 2) * L::QK_PAIR + (kk & 3) * 32;  // [Q; K] rows
          umma_bf16(tmem_base + buf * 64, umma_desc_sw128(a), umma_desc_sw128(a + L::SUB),
                    kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(tmem_full(buf));
        ++issued;
      }
      // every issued MMA has landed before tensor memory is released
      for (int c = issued - 2 < 0 ? 0 : issued - 2; c < issued; ++c)
        mbar_wait_bounded(tmem_full(c & 1), (c >> 1) & 1, kWaitTimeoutNs);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ prep
    const int ptid = tid;
    float *sTf = reinterpret_cast<float *>(smem + L::OFF_TF);
    __nv_bfloat16 *sTB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_TB);
    __nv_bfloat16 *sMB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_MB);
    const uint32_t TBa = smem_u32(sTB), MBa = smem_u32(sMB);
    int *vote = votes;  // prep votes: [0..7]

    for (int c = 0; c < nc; ++c) {
      const int slot = c % NIN, stage = c & 1;
      const int valid = (int)(len - (int64_t)c * 64 < 64 ? len - (int64_t)c * 64 : 64);
      GDN_PHASE(0);
      // A and P of this chunk are in shared memory (and the stage is free: the
      // carry warps wrote P only after they finished chunk c-2)
      bool ok = role_wait(s_ready(stage), (c >> 1) & 1, S, p, n, h, 2);
      if (ok) ok = role_wait(full_in(slot), (c / NIN) & 1, S, p, n, h, 3);
      ok = __all_sync(0xffffffffu, ok) && !*S.abort_flag;
      GDN_PHASE(1);

      const uint32_t Qs = slot_base(slot), Ks = Qs + L::SUB, Vs = Qs + L::OFF_V;
      const float *gate = gate_ptr(slot);
      const float *gam = gate + 64, *beta = gate + 192;
      const float *sA = reinterpret_cast<const float *>(smem + L::OFF_A) + stage * 64 * L::A_LD;
      const uint32_t Ws = sbase + L::OFF_ST + stage * L::STAGE;
      const uint32_t Us = Ws + (DK / 64) * L::SUB;

      // ---- rows past the end of the sequence: zero Q, K, V (the MMA has read them) ----
      if (ok && valid < 64) {
        constexpr int gq = DK / 8;  // 16-byte granules per Q/K row
        constexpr int per_row = 2 * gq + 8;
        for (int idx = ptid; idx < (64 - valid) * per_row; idx += kPrepThreads) {
          const int row = valid + idx / per_row, q = idx % per_row;
          uint32_t a;
          if (q < gq) a = qk_addr(Qs, row, q * 8);
          else if (q < 2 * gq) a = qk_addr(Ks, row, (q - gq) * 8);
          else a = tile_addr(Vs, row, (q - 2 * gq) * 8);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
        }
        fence_proxy_async_smem();
      }
      if (lane == 0) vote[(c & 1) * 4 + warp] = ok ? 1 : 0;
      named_sync(kBarPrep, kPrepThreads);
      GDN_PHASE(2);
      {
        const int *v = vote + (c & 1) * 4;
        if (!(v[0] && v[1] && v[2] && v[3])) break;
      }

      // ---- 16x16 diagonal blocks of T = (I + A)^-1: right-looking substitution,
      //      one block per warp, one column per lane, fp32 ----
      if (lane < 16) {
        const int l = lane, w = warp;
        const float *Ab = sA + (16 * w) * L::A_LD + 16 * w;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == l) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < 15; ++k) {
          const float xk = x[k];
#pragma unroll
          for (int r = k + 1; r < 16; ++r) x[r] = fmaf(-Ab[r * L::A_LD + k], xk, x[r]);
        }
        const float bj = beta[16 * w + l];
        float bgj = bj * gam[16 * w + l];
        if constexpr ((kF & kFL2) != 0)  // W = T diag(beta gamma r_k) K
          bgj *= reinterpret_cast<const float *>(smem + L::OFF_RN)[slot * L::RN_SLOT + 64 + 16 * w + l];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          sTf[(w * 16 + r) * L::TF_LD + l] = x[r];
          sTB[((0 * 4 + w) * 16 + r) * L::TB_LD + l] = __float2bfloat16_rn(x[r] * bgj);
          sTB[((1 * 4 + w) * 16 + r) * L::TB_LD + l] = __float2bfloat16_rn(x[r] * bj);
        }
      }
      GDN_PHASE(3);
      named_sync(kBarPrep, kPrepThreads);
      GDN_PHASE(4);

      // ---- M_ik = T_ii A_ik (i > k), tf32 tensor cores, stored negated as bf16 ----
#pragma unroll 1
      for (int blk = warp; blk < 6; blk += 4) {
        const int i = blk == 0 ? 1 : (blk < 3 ? 2 : 3);
        const int k = blk - (i * (i - 1)) / 2;
        const float *T = sTf + (i * 16) * L::TF_LD;
        const float *Ak = sA + (16 * i) * L::A_LD + 16 * k;
        float acc[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint32_t a0 = to_tf32(T[g * L::TF_LD + 8 * ks + t]);
          const uint32_t a1 = to_tf32(T[(g + 8) * L::TF_LD + 8 * ks + t]);
          const uint32_t a2 = to_tf32(T[g * L::TF_LD + 8 * ks + t + 4]);
          const uint32_t a3 = to_tf32(T[(g + 8) * L::TF_LD + 8 * ks + t + 4]);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b0 = to_tf32(Ak[(8 * ks + t) * L::A_LD + 8 * nt + g]);
            const uint32_t b1 = to_tf32(Ak[(8 * ks + t + 4) * L::A_LD + 8 * nt + g]);
            mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
          }
        }
        __nv_bfloat16 *M = sMB + blk * 16 * L::TB_LD;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          *reinterpret_cast<uint32_t *>(M + g * L::TB_LD + 8 * nt + 2 * t) =
              pack_bf16(-acc[nt][0], -acc[nt][1]);
          *reinterpret_cast<uint32_t *>(M + (g + 8) * L::TB_LD + 8 * nt + 2 * t) =
              pack_bf16(-acc[nt][2], -acc[nt][3]);
        }
      }
      GDN_PHASE(5);
      named_sync(kBarPrep, kPrepThreads);
      GDN_PHASE(6);

      // ---- block forward substitution: X_i = T_ii B_i + sum_k (-M_ik) X_k, X = [W | U~].
      //      Terms that do not depend on the previous block row are formed first or
      //      while the other warps catch up, leaving one product per level on the
      //      critical path. ----
      {
        constexpr int NP = (DK + kDvt) / 16;  // 16-column pairs of [W | U~]
        constexpr int PPW = NP / 4;          // pairs per warp
        const int arow = lrow + (lmi & 1) * 8, acol = (lmi >> 1) * 8;
        float lacc[4][PPW][2][4];
#pragma unroll
        for (int lv = 0; lv < 4; ++lv)
#pragma unroll
          for (int pp = 0; pp < PPW; ++pp) {
            const int pi = warp + 4 * pp;
            const bool isW = 16 * pi < DK;
            const int col = isW ? 16 * pi : 16 * pi - DK;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) lacc[lv][pp][nt][e] = 0.f;
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(TBa + ((((isW ? 0 : 1) * 4 + lv) * 16 + arow) * L::TB_LD + acol) * 2, a0,
                    a1, a2, a3);
            const int brow = 16 * lv + lrow + (lmi & 1) * 8, bcol = col + (lmi >> 1) * 8;
            ldsm_x4_t(isW ? qk_addr(Ks, brow, bcol) : tile_addr(Vs, brow, bcol), b0, b1, b2, b3);
            mma_bf16(lacc[lv][pp][0], a0, a1, a2, a3, b0, b1);
            mma_bf16(lacc[lv][pp][1], a0, a1, a2, a3, b2, b3);
          }
#pragma unroll
        for (int lv = 0; lv < 4; ++lv) {
          // B fragments of X_{lv-1} for every pair (rows 16(lv-1)..), reused below
          uint32_t xb[PPW][4];
          if (lv > 0) {
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp) {
              const int pi = warp + 4 * pp;
              const bool isW = 16 * pi < DK;
              const int col = isW ? 16 * pi : 16 * pi - DK;
              ldsm_x4_t(tile_addr(isW ? Ws : Us, 16 * (lv - 1) + lrow + (lmi & 1) * 8,
                                  col + (lmi >> 1) * 8),
                        xb[pp][0], xb[pp][1], xb[pp][2], xb[pp][3]);
            }
            const int blk = (lv * (lv - 1)) / 2 + (lv - 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(MBa + ((blk * 16 + arow) * L::TB_LD + acol) * 2, a0, a1, a2, a3);
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp) {
              mma_bf16(lacc[lv][pp][0], a0, a1, a2, a3, xb[pp][0], xb[pp][1]);
              mma_bf16(lacc[lv][pp][1], a0, a1, a2, a3, xb[pp][2], xb[pp][3]);
            }
          }
          // store X_lv
#pragma unroll
          for (int pp = 0; pp < PPW; ++pp) {
            const int pi = warp + 4 * pp;
            const bool isW = 16 * pi < DK;
            const int col = isW ? 16 * pi : 16 * pi - DK;
            const uint32_t xt = isW ? Ws : Us;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(
                                 tile_addr(xt, 16 * lv + g + 8 * hf, col + 8 * nt + 2 * t)),
                             "r"(pack_bf16(lacc[lv][pp][nt][2 * hf], lacc[lv][pp][nt][2 * hf + 1]))
                             : "memory");
          }
          // X_{lv-1} terms of the later block rows
          if (lv > 0) {
#pragma unroll
            for (int l2 = lv + 1; l2 < 4; ++l2) {
              const int blk = (l2 * (l2 - 1)) / 2 + (lv - 1);
              uint32_t a0, a1, a2, a3;
              ldsm_x4(MBa + ((blk * 16 + arow) * L::TB_LD + acol) * 2, a0, a1, a2, a3);
#pragma unroll
              for (int pp = 0; pp < PPW; ++pp) {
                mma_bf16(lacc[l2][pp][0], a0, a1, a2, a3, xb[pp][0], xb[pp][1]);
                mma_bf16(lacc[l2][pp][1], a0, a1, a2, a3, xb[pp][2], xb[pp][3]);
              }
            }
          }
          if (lv < 3) named_sync(kBarPrep, kPrepThreads);
        }
      }
      GDN_PHASE(7);
      mbar_arrive(full_st(stage));
    }
  } else {
    // ------------------------------------------------------------ carry
    const int cw = warp - 4;  // value columns 16cw .. 16cw+15 of the tile; TMEM lane quarter
    const int ctid = tid - kPrepThreads;
    int *vote = votes + 8;
    const size_t state_off = ((size_t)n * H + h) * (size_t)DK * dv + col0 + 16 * cw;

    // Drain the TMEM accumulator of chunk cc: this thread owns row r = 32cw + lane
    // of [Q; K] K^T, i.e. row r of P (r < 64) or row r - 64 of A.  Returns false
    // if a wait gave up.
    auto s_epilogue = [&](int cc) -> bool {
      const int slot = cc % NIN, buf = cc & 1;
      [[maybe_unused]] const int c = cc;  // phase stamps of the drain go to chunk cc
      GDN_PHASE(8);
      bool ok = role_wait(tmem_full(buf), (cc >> 1) & 1, S, p, n, h, 7);
      if (ok) ok = role_wait(full_in(slot), (cc / NIN) & 1, S, p, n, h, 8);
      GDN_PHASE(9);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      {
        const uint32_t ta = tmem_base + ((uint32_t)(32 * cw) << 16) + buf * 64;
        tmem_ld32(ta, v0);
        tmem_ld32(ta + 32, v1);
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive(tmem_empty(buf));
      GDN_PHASE(10);

      const int valid = (int)(len - (int64_t)cc * 64 < 64 ? len - (int64_t)cc * 64 : 64);
      const float *gate = gate_ptr(slot);
      const float *G2 = gate, *beta = gate + 192, *E = gate + 256;
      const int r = 32 * cw + lane;
      const bool isP = cw < 2;
      const int i = isP ? r : r - 64;
      const int ilim = isP ? i + 1 : i;  // P keeps j <= i, A keeps j < i
      const bool rowok = i < valid;
      const float Gi = G2[i];
      float bi = isP ? 1.f : beta[i];
      // column vectors: G_j and E_j, or under the normalisation G_j - log2 r_k_j
      // and E_j r_k_j (the column factor r_k folded in)
      const float *Gc = G2, *Ec = E;
      if constexpr ((kF & kFL2) != 0) {
        // this thread's row norm (q_i for P rows, k_i for A rows) from the
        // tile, shared with the other drain threads
        float *rn = reinterpret_cast<float *>(smem + L::OFF_RN) + slot * L::RN_SLOT;
        const uint32_t tb = slot_base(slot) + (isP ? 0 : L::SUB);
        float ss = 0.f;
#pragma unroll
        for (int q8 = 0; q8 < DK / 8; ++q8) {
          uint32_t w[4];
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                       : "r"(qk_addr(tb, i, 8 * q8)));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
          }
        }
        const float rr = rsqrtf(ss + 1e-6f);
        if (isP) {
          rn[i] = rr;
        } else {
          rn[64 + i] = rr;
          rn[128 + i] = Gi - __log2f(rr);
          rn[192 + i] = E[i] * rr;
        }
        const uint32_t nb = sbase + L::OFF_NBAR + 8 * (cc & 1);
        mbar_arrive(nb);
        if (!__all_sync(0xffffffffu, role_wait(nb, (cc >> 1) & 1, S, p, n, h, 30))) return false;
        bi *= rr;  // row factor: r_q (P) or beta_i r_k (A)
        Gc = rn + 128;
        Ec = rn + 192;
      }
      float val[64];
      // Gamma_ij = 2^(G_i - G_j): a direct exponent for the 16-column blocks that
      // meet this warp's rows; for blocks entirely before them, two factors that
      // are both <= 1: 2^(G_i - G_b) * 2^(G_b - G_j), b the block's last token.
      if ((cw & 1) == 0) {  // rows 0..31: columns 0..31
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 gg = *reinterpret_cast<const float4 *>(Gc + 4 * j4);
          const float gj[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            const float sv = __uint_as_float(v0[j]) * bi * ex2(Gi - gj[e]);
            val[j] = (rowok && j < ilim) ? sv : 0.f;
          }
        }
      } else {  // rows 32..63: columns 0..31 factored, 32..63 direct
        const float F0 = ex2(Gi - G2[15]) * bi, F1 = ex2(Gi - G2[31]) * bi;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 ee = *reinterpret_cast<const float4 *>(Ec + 4 * j4);
          const float ej[4] = {ee.x, ee.y, ee.z, ee.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            const float sv = __uint_as_float(v0[j]) * (j < 16 ? F0 : F1) * ej[e];
            val[j] = rowok ? sv : 0.f;
          }
        }
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 gg = *reinterpret_cast<const float4 *>(Gc + 32 + 4 * j4);
          const float gj[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 32 + 4 * j4 + e;
            const float sv = __uint_as_float(v1[j - 32]) * bi * ex2(Gi - gj[e]);
            val[j] = (rowok && j < ilim) ? sv : 0.f;
          }
        }
      }
      // Only the blocks on or below the diagonal are read later: row i needs
      // columns 0 .. 16*(i/16)+15, i.e. 32 columns for rows 0..31, 64 beyond.
      const int ncols = (cw & 1) == 0 ? 32 : 64;
      if (isP) {
        const uint32_t Ps = sbase + L::OFF_ST + buf * L::STAGE + (DK / 64) * L::SUB + L::SUB;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (8 * q < ncols)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(tile_addr(Ps, i, 8 * q)),
                         "r"(pack_bf16(val[8 * q], val[8 * q + 1])),
                         "r"(pack_bf16(val[8 * q + 2], val[8 * q + 3])),
                         "r"(pack_bf16(val[8 * q + 4], val[8 * q + 5])),
                         "r"(pack_bf16(val[8 * q + 6], val[8 * q + 7]))
                         : "memory");
      } else {
        float *Arow = reinterpret_cast<float *>(smem + L::OFF_A) + (buf * 64 + i) * L::A_LD;
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (4 * q < ncols)
            *reinterpret_cast<float4 *>(Arow + 4 * q) =
                make_float4(val[4 * q], val[4 * q + 1], val[4 * q + 2], val[4 * q + 3]);
      }
      GDN_PHASE(11);
      mbar_arrive(s_ready(buf));
      return true;
    };

    // H^T accumulators: rows = value column (g, g+8), columns = key index
    float hacc[DK / 8][4];
#pragma unroll
    for (int nt = 0; nt < DK / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vc = g + 8 * (e >> 1), kd = 8 * nt + 2 * t + (e & 1);
        hacc[nt][e] = p.s0 ? p.s0[state_off + (size_t)kd * dv + vc] : 0.f;
      }

    bool alive = s_epilogue(0);
    if (alive && nc > 1) alive = s_epilogue(1);

    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
    for (int c = 0; c < nc && alive; ++c) {
      const int slot = c % NIN, stage = c & 1;
      const int valid = (int)(len - (int64_t)c * 64 < 64 ? len - (int64_t)c * 64 : 64);
      GDN_PHASE(0);
      bool ok = role_wait(full_st(stage), (c >> 1) & 1, S, p, n, h, 4);
      ok = __all_sync(0xffffffffu, ok) && !*S.abort_flag;
      GDN_PHASE(1);

      const uint32_t Qs = slot_base(slot), Ks = Qs + L::SUB;
      const uint32_t Ws = sbase + L::OFF_ST + stage * L::STAGE;
      const uint32_t Us = Ws + (DK / 64) * L::SUB, Ps = Us + L::SUB;
      const float *gate = gate_ptr(slot);
      const float *gam = gate + 64, *dec = gate + 128;
      const float gC = sgc[slot];

      // bf16 A operand of H^T (accumulator layout re-packed in registers)
      uint32_t hb[DK / 16][4];
#pragma unroll
      for (int s = 0; s < DK / 16; ++s) {
        hb[s][0] = pack_bf16(hacc[2 * s][0], hacc[2 * s][1]);
        hb[s][1] = pack_bf16(hacc[2 * s][2], hacc[2 * s][3]);
        hb[s][2] = pack_bf16(hacc[2 * s + 1][0], hacc[2 * s + 1][1]);
        hb[s][3] = pack_bf16(hacc[2 * s + 1][2], hacc[2 * s + 1][3]);
      }

      // acc = -U~^T  (transposed load of this warp's 16 columns)
      float uacc[8][4];
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(tile_addr(Us, 16 * jp + lrow + (lmi >> 1) * 8, 16 * cw + (lmi & 1) * 8), r0,
                  r1, r2, r3);
        uacc[2 * jp][0] = -bf16_lo(r0);
        uacc[2 * jp][1] = -bf16_hi(r0);
        uacc[2 * jp][2] = -bf16_lo(r1);
        uacc[2 * jp][3] = -bf16_hi(r1);
        uacc[2 * jp + 1][0] = -bf16_lo(r2);
        uacc[2 * jp + 1][1] = -bf16_hi(r2);
        uacc[2 * jp + 1][2] = -bf16_lo(r3);
        uacc[2 * jp + 1][3] = -bf16_hi(r3);
      }
      // acc += H^T W^T  (so U^T = -acc);  O^T = H^T Q^T
      float oacc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[j][e] = 0.f;
#pragma unroll
      for (int s = 0; s < DK / 16; ++s)
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          const int brow = 16 * jp + lrow + (lmi >> 1) * 8, bcol = 16 * s + (lmi & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(tile_addr(Ws, brow, bcol), b0, b1, b2, b3);
          mma_bf16(uacc[2 * jp], hb[s][0], hb[s][1], hb[s][2], hb[s][3], b0, b1);
          mma_bf16(uacc[2 * jp + 1], hb[s][0], hb[s][1], hb[s][2], hb[s][3], b2, b3);
          ldsm_x4(qk_addr(Qs, brow, bcol), b0, b1, b2, b3);
          mma_bf16(oacc[2 * jp], hb[s][0], hb[s][1], hb[s][2], hb[s][3], b0, b1);
          mma_bf16(oacc[2 * jp + 1], hb[s][0], hb[s][1], hb[s][2], hb[s][3], b2, b3);
        }
      GDN_PHASE(2);
      // U^T as bf16 A operands: plain (for O) and scaled by exp(G_C - G_j) (for H')
      uint32_t ub[4][4], ubd[4][4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int j0 = 16 * s + 2 * t, j1 = j0 + 8;
        float d00 = dec[j0], d01 = dec[j0 + 1], d10 = dec[j1], d11 = dec[j1 + 1];
        if constexpr ((kF & kFL2) != 0) {  // Ud = diag(d r_k) U
          const float *rk = reinterpret_cast<const float *>(smem + L::OFF_RN) + slot * L::RN_SLOT + 64;
          d00 *= rk[j0]; d01 *= rk[j0 + 1]; d10 *= rk[j1]; d11 *= rk[j1 + 1];
        }
        const float *u0 = uacc[2 * s], *u1 = uacc[2 * s + 1];
        ub[s][0] = pack_bf16(-u0[0], -u0[1]);
        ub[s][1] = pack_bf16(-u0[2], -u0[3]);
        ub[s][2] = pack_bf16(-u1[0], -u1[1]);
        ub[s][3] = pack_bf16(-u1[2], -u1[3]);
        ubd[s][0] = pack_bf16(-u0[0] * d00, -u0[1] * d01);
        ubd[s][1] = pack_bf16(-u0[2] * d00, -u0[3] * d01);
        ubd[s][2] = pack_bf16(-u1[0] * d10, -u1[1] * d11);
        ubd[s][3] = pack_bf16(-u1[2] * d10, -u1[3] * d11);
      }
      // H^T <- gamma_C H^T + (U^T diag(dec)) K   (the serial chain)
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) hacc[nt][e] *= gC;
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int q = 0; q < DK / 16; ++q) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(qk_addr(Ks, 16 * s + lrow + (lmi & 1) * 8, 16 * q + (lmi >> 1) * 8), b0, b1,
                    b2, b3);
          mma_bf16(hacc[2 * q], ubd[s][0], ubd[s][1], ubd[s][2], ubd[s][3], b0, b1);
          mma_bf16(hacc[2 * q + 1], ubd[s][0], ubd[s][1], ubd[s][2], ubd[s][3], b2, b3);
        }
      GDN_PHASE(3);
      // O^T: scale the H-part by gamma_i, then add U^T P^T (lower-triangular blocks only)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float ga = gam[8 * j + 2 * t], gb = gam[8 * j + 2 * t + 1];
        if constexpr ((kF & kFL2) != 0) {  // O = diag(gamma r_q) Q H + P U
          const float *rq = reinterpret_cast<const float *>(smem + L::OFF_RN) + slot * L::RN_SLOT;
          ga *= rq[8 * j + 2 * t];
          gb *= rq[8 * j + 2 * t + 1];
        }
        oacc[j][0] *= ga;
        oacc[j][1] *= gb;
        oacc[j][2] *= ga;
        oacc[j][3] *= gb;
      }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (s <= pp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(tile_addr(Ps, 16 * pp + lrow + (lmi >> 1) * 8, 16 * s + (lmi & 1) * 8), b0,
                    b1, b2, b3);
            mma_bf16(oacc[2 * pp], ub[s][0], ub[s][1], ub[s][2], ub[s][3], b0, b1);
            mma_bf16(oacc[2 * pp + 1], ub[s][0], ub[s][1], ub[s][2], ub[s][3], b2, b3);
          }
      GDN_PHASE(4);
      if constexpr ((kF & kFEpi) != 0) {
        // block epilogue (o + D_h v) * gate, with v from this chunk's V tile:
        // ldmatrix.trans hands each thread v at (token 8j + 2t, +1; column
        // 16cw + g, +8), the accumulator's own layout
        const uint32_t Vs = slot_base(slot) + L::OFF_V;
        const float dh = p.d_skip ? p.d_skip[h] : 0.f;
        const float *ogate = gate_ptr(slot) + 320;  // staged by the producer
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          uint32_t vb[4];
          ldsm_x4_t(tile_addr(Vs, 16 * jp + 8 * (lmi >> 1) + lrow, 16 * cw + 8 * (lmi & 1)), vb[0],
                    vb[1], vb[2], vb[3]);
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = 2 * jp + jj;
            const float2 og = *reinterpret_cast<const float2 *>(ogate + 8 * j + 2 * t);
            const uint32_t lo = vb[2 * jj], hi = vb[2 * jj + 1];  // columns g and g + 8
            oacc[j][0] = block_epilogue(oacc[j][0], bf16_lo(lo), dh, og.x);
            oacc[j][1] = block_epilogue(oacc[j][1], bf16_hi(lo), dh, og.y);
            oacc[j][2] = block_epilogue(oacc[j][2], bf16_lo(hi), dh, og.x);
            oacc[j][3] = block_epilogue(oacc[j][3], bf16_hi(hi), dh, og.y);
          }
        }
      }
      // this chunk's input slot is no longer read (its stage is reused by this
      // warp group's own epilogue of chunk c+2, after the barrier below)
      mbar_arrive(empty_in(slot));

      // O^T -> staging tile [token][col] (transposed store).  A full chunk leaves
      // by one TMA store; the last partial chunk by plain stores of its rows.
      // Three staging tiles: after issuing the store of chunk c, the issuing
      // thread waits until the store of chunk c-1 has read its tile, which is
      // reused at chunk c+2.
      const uint32_t Os = sbase + L::OFF_OST + (c % 3) * L::SUB;
#pragma unroll
      for (int jp = 0; jp < 4; ++jp)
        stsm_x4_t(tile_addr(Os, 16 * jp + lrow + (lmi >> 1) * 8, 16 * cw + (lmi & 1) * 8),
                  pack_bf16(oacc[2 * jp][0], oacc[2 * jp][1]),
                  pack_bf16(oacc[2 * jp][2], oacc[2 * jp][3]),
                  pack_bf16(oacc[2 * jp + 1][0], oacc[2 * jp + 1][1]),
                  pack_bf16(oacc[2 * jp + 1][2], oacc[2 * jp + 1][3]));
      if (valid == 64) fence_proxy_async_smem();
      if (lane == 0) vote[(c & 1) * 4 + cw] = ok ? 1 : 0;
      GDN_PHASE(5);
      named_sync(kBarCarry, kCarryThreads);
      GDN_PHASE(6);
      {
        const int *v = vote + (c & 1) * 4;
        if (!(v[0] && v[1] && v[2] && v[3])) break;
      }
      if (valid == 64) {
        if (ctid == 0) {
          tma_store_3d(&tmap_o, col0, h, (int)(start + (int64_t)c * 64), Os);
          bulk_commit();
          bulk_wait_read<1>();
        }
      } else {
        for (int idx = ctid; idx < valid * 8; idx += kCarryThreads) {
          const int row = idx >> 3, ch = idx & 7;
          uint32_t w0, w1, w2, w3;
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                       : "r"(tile_addr(Os, row, ch * 8)));
          __nv_bfloat16 *dst =
              o + ((size_t)(start + (int64_t)c * 64 + row) * H + h) * dv + col0 + ch * 8;
          *reinterpret_cast<uint4 *>(dst) = make_uint4(w0, w1, w2, w3);
        }
      }
      // the accumulator two chunks ahead (its P tile is stage c&1, free now)
      if (c + 2 < nc) alive = s_epilogue(c + 2);
      GDN_PHASE(7);
    }
    if (ctid == 0) bulk_wait_all();  // O stores done reading staging before exit
    if (p.sN && !*S.abort_flag) {
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vc = g + 8 * (e >> 1), kd = 8 * nt + 2 * t + (e & 1);
          p.sN[state_off + (size_t)kd * dv + vc] = hacc[nt][e];
        }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int DK, int NIN>
cudaError_t launch_tc(const FwdParams &p, cudaStream_t stream) {
  using L = TcLayout<DK, NIN>;
  const int64_t tokens = p.cu ? p.seq_len : (int64_t)p.num_seqs * p.seq_len;
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap(&tq, p.q, DK, p.num_heads, tmap_rows(p, tokens, p.ext.q, DK)) ||
      !make_tmap(&tk, p.k, DK, p.num_heads, tmap_rows(p, tokens, p.ext.k, DK)) ||
      !make_tmap(&tv, p.v, p.dv, p.num_heads, tmap_rows(p, tokens, p.ext.v, p.dv)) ||
      !make_tmap(&to, p.o, p.dv, p.num_heads, tmap_rows(p, tokens, p.ext.o, p.dv)))
    return cudaErrorInvalidValue;
  // the block parts fused into the pass run in their own instantiation
  const int feat = ((p.flags & GDN_QK_L2NORM) ? kFL2 : 0) | ((p.d_skip || p.out_gate) ? kFEpi : 0);
  auto kern = feat == 0        ? gdn_fwd_tc_kernel<DK, NIN, 0>
              : feat == kFL2   ? gdn_fwd_tc_kernel<DK, NIN, kFL2>
              : feat == kFEpi  ? gdn_fwd_tc_kernel<DK, NIN, kFEpi>
                               : gdn_fwd_tc_kernel<DK, NIN, kFL2 | kFEpi>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (err != cudaSuccess) return err;
  const dim3 grid(p.dv / kDvt, p.num_heads, p.num_seqs);
  kern<<<grid, kTcThreads, L::ALLOC, stream>>>(p, tq, tk, tv, to);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(int dk, int dv) { return (dk == 64 || dk == 128) && dv % kDvt == 0; }

cudaError_t launch_fwd_tc(const FwdParams &p, cudaStream_t stream) {
  switch (p.dk) {
    case 64: return launch_fwd_tc64(p, stream);
    case 128: return launch_tc<128, 2>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

