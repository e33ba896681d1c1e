// Chunk-size variants of the tensor-core forward: chunk_size 32 and 128 for
// head_dim_k = 64, bf16 storage ("v1.0 Architecture & Design Spec", section
// 2.3, sweeps chunk_size over {32, 64, 128}; the result depends on it only
// through rounding).  Every chunk product runs on tcgen05 with fp32
// accumulators in tensor memory; the phases of a chunk run one after the
// other (the 64-token kernel overlaps them across chunks), so this kernel
// answers what a chunk size costs in products, inverse depth and drains, at
// a fraction of the 64-token kernel's overlap.
//
// Chunk algebra as in the 64-token kernel (gated delta rule, H = S^T):
//   A = strictly_lower(diag(beta) K K^T (.) Gamma),  P = (Q K^T (.) Gamma)_{i>=j}
//   (I + A) W = diag(beta gamma) K,  (I + A) U~ = diag(beta) V
//   U = U~ - W H,  O = diag(gamma) Q H + P U,  H' = gamma_C H + K^T diag(d) U
// with G the chunk's log2-unit gate prefix sum, gamma = 2^G, d = 2^(G_C - G),
// Gamma_ij = 2^(G_i - G_j) ("Model Architecture Walkthrough", section 5.3.1).
// (I + A)^-1 is applied by the blocked scheme of the 64-token kernel with C/16
// levels: fp32 16x16 diagonal inverses, tf32 couplings M_ik = T_ii A_ik, and a
// left-looking bf16 substitution for the columns of [W | U~].
//
// One CTA (8 warps) owns one (sequence, head, 64-wide value slice).  An input
// slot holds K | Q | W | V (U~ written over V), [C][64] bf16 tiles with the
// 128-byte swizzle.  Products, all M = 128 (accumulator row r in TMEM lane r):
//   C = 32:  S  = [K; Q; *] K^T      rows 0..31 K K^T (A), 32..63 Q K^T (P)
//            D1 = [Q; W; *] H        rows 0..31 Q H,       32..63 W H
//   C = 128: S_A = K K^T, S_P = Q K^T, D1_W = W H, D1_Q = Q H (one product each)
//   both:    DH = [K^T; Q^T] Ud      rows 0..63 K^T Ud (the state increment)
//            PU = [P; *] U           rows 0..C-1 P U
// "*" rows are whatever shared memory follows; their results are never read.
// The fp32 state stays in registers of warps 0, 1, 4, 5 (lane quarters 0, 1:
// key row = 32 * quarter + lane, value columns 0..31 / 32..63).
// Every wait is bounded; a timeout records GDN_ERR_TIMEOUT and ends the loop.
//
// The GDN block parts of gdn_fwd run here too (runtime branches; this kernel
// is not tuned for them): beta from logits, the q/k L2 normalisation folded
// into fp32 row and column factors (r_q, r_k) as in the 64-token kernel, and
// the output epilogue (o + D_h v) * gate.
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kDK = 64;
constexpr int kThreadsC = 256;  // 8 warps

template <int C>
struct LayoutC {
  static constexpr int T = C * 128;  // one [C][64] bf16 tile
  static constexpr int SK = 0, SQ = T, SW = 2 * T, SV = 3 * T;
  // C = 32: room so that the M = 128 operand [Q; W; *] (rows 64..127 past V)
  // stays inside the allocation
  static constexpr int OFF_PAD = 4 * T, PAD = C == 32 ? 4096 : 0;
  // P [C][C] bf16 as 64-column sub-tiles (C = 32: one, columns 32..63 unused)
  static constexpr int PSUB = C * 128, NPSUB = C == 128 ? 2 : 1;
  static constexpr int OFF_P = OFF_PAD + PAD;
  static constexpr int OFF_H = OFF_P + NPSUB * PSUB;  // H [64][64] bf16
  static constexpr int OFF_U = OFF_H + 8192;          // U [C][64] bf16
  static constexpr int OFF_UD = OFF_U + T;            // Ud [C][64] bf16
  static constexpr int NB = C / 16;                   // 16-row blocks
  static constexpr int A_LD = 20, A_BLK = 16 * A_LD;  // fp32 blocks (r, c), c <= r
  static constexpr int OFF_A = OFF_UD + T;
  static constexpr int TB_LD = 16;                    // bf16 16x16 tiles, column-major
  static constexpr int OFF_TB = OFF_A + NB * (NB + 1) / 2 * A_BLK * 4;
  static constexpr int NMB = NB * (NB - 1) / 2;       // couplings M_ik, i > k
  static constexpr int OFF_MB = OFF_TB + 2 * NB * 16 * TB_LD * 2;
  static constexpr int OFF_G = OFF_MB + NMB * 16 * TB_LD * 2;  // f32 [6][C]: G, gamma, d, beta, r_q, r_k
  static constexpr int OFF_MISC = OFF_G + 6 * C * 4;  // f32 gamma_C, f32 out-gate scratch unused, u32 TMEM
  static constexpr int OFF_BAR = OFF_MISC + 64;       // mbarriers: TMA, MMA
  static constexpr int BYTES = OFF_BAR + 64;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(OFF_P % 1024 == 0 && OFF_H % 1024 == 0 && OFF_U % 1024 == 0 &&
                OFF_UD % 1024 == 0, "tiles need 1024-byte alignment");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// TMEM columns
template <int C> struct ColsC;
template <> struct ColsC<32> {
  static constexpr uint32_t S = 0, D1 = 64, DH = 128, PU = 192, ALLOC = 256;
};
template <> struct ColsC<128> {
  static constexpr uint32_t SA = 0, SP = 128, D1W = 256, D1Q = 320, DH = 384, PU = 448, ALLOC = 512;
};

template <int C>
__global__ void __launch_bounds__(kThreadsC, 1)
gdn_fwd_tcc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v) {
  using L = LayoutC<C>;
  using TC = ColsC<C>;
  constexpr int NB = L::NB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wq = warp & 3;
  const int tile = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv, col0 = tile * kDvt;

  int64_t start, len;
  if (!sequence_bounds(p, n, h, start, len)) return;  // uniform over the CTA
  if ((p.flags & GDN_DEBUG_CHECKS) &&
      !debug_ranges_ok(p, n, h, start, len, col0, kDvt, 2, true))
    return;  // recorded; nothing was accessed
  if (len == 0) {  // an empty sequence: the state passes through
    pass_state_through(p, n, h, col0, kDvt);
    return;
  }
  const int nc = (int)((len + C - 1) / C);
  const bool l2 = (p.flags & GDN_QK_L2NORM) != 0;
  const bool epi = p.d_skip != nullptr || p.out_gate != nullptr;

  float *sG = reinterpret_cast<float *>(smem + L::OFF_G);  // G (log2 units)
  float *sGam = sG + C, *sDec = sG + 2 * C, *sBeta = sG + 3 * C, *sRq = sG + 4 * C,
        *sRk = sG + 5 * C;
  float *sMisc = reinterpret_cast<float *>(smem + L::OFF_MISC);
  const uint32_t barTma = sbase + L::OFF_BAR, barMma = sbase + L::OFF_BAR + 8;
  auto S1 = [&](uint32_t addr) -> uint32_t & {
    return *reinterpret_cast<uint32_t *>(smem + (addr - sbase));
  };
  auto S4 = [&](uint32_t addr) -> uint4 & {
    return *reinterpret_cast<uint4 *>(smem + (addr - sbase));
  };

  if (tid == 0) {
    mbar_init(barTma, 1);
    mbar_init(barMma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(sbase + L::OFF_MISC + 8, TC::ALLOC);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::OFF_MISC + 8);
  auto tm = [&](uint32_t col) { return tmem + ((uint32_t)(32 * wq) << 16) + col; };
  const int lrow = lane & 7, lmi = lane >> 3;  // ldmatrix: row within matrix, matrix index
  const int g = lane >> 2, t = lane & 3;       // mma fragment coordinates

  auto load_tiles = [&](int c) {  // one thread
    const int row = (int)(start + (int64_t)c * C);
    mbar_arrive_expect_tx(barTma, 3 * L::T);
    tma_load_3d(sbase + L::SK, &tmap_k, 0, h, row, barTma);
    tma_load_3d(sbase + L::SQ, &tmap_q, 0, h, row, barTma);
    tma_load_3d(sbase + L::SV, &tmap_v, col0, h, row, barTma);
  };
  uint32_t ph_tma = 0, ph_mma = 0;
  // wait for the products issued so far (one commit), all threads
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait_bounded(barMma, ph_mma, kWaitTimeoutNs);
    ph_mma ^= 1;
    if (!ok && tid == 0) report(p.status, GDN_ERR_TIMEOUT, (uint32_t)n, (uint32_t)h, 40);
    return __syncthreads_and(ok) != 0;
  };

  // E2a state: warps 0, 1, 4, 5 (lane quarters 0, 1), key row 32 wq + lane,
  // value columns cb .. cb + 31
  const bool is_state = wq < 2;
  const int krow = 32 * wq + lane, cb = warp >= 4 ? 32 : 0;
  const size_t state_row = ((size_t)n * H + h) * (size_t)kDK * dv + (size_t)krow * dv + col0 + cb;
  float hrow[32];
  auto store_h = [&]() {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      S4(tile_addr(sbase + L::OFF_H, krow, cb + 8 * q)) =
          make_uint4(pack_bf16(hrow[8 * q], hrow[8 * q + 1]), pack_bf16(hrow[8 * q + 2], hrow[8 * q + 3]),
                     pack_bf16(hrow[8 * q + 4], hrow[8 * q + 5]), pack_bf16(hrow[8 * q + 6], hrow[8 * q + 7]));
  };
  if (is_state) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p.s0) v4 = *reinterpret_cast<const float4 *>(p.s0 + state_row + 4 * q);
      hrow[4 * q] = v4.x;
      hrow[4 * q + 1] = v4.y;
      hrow[4 * q + 2] = v4.z;
      hrow[4 * q + 3] = v4.w;
    }
    store_h();
  }
  if (tid == 0) load_tiles(0);
  bool tma_pending = true;  // (thread 0's view) a load into the slot has not been waited for
  const float dh = p.d_skip ? p.d_skip[h] : 0.f;
  const __nv_bfloat16 *betap = static_cast<const __nv_bfloat16 *>(p.beta);
  int done = 0;  // chunks completed

  for (int c = 0; c < nc; ++c) {
    const int valid = (int)(len - (int64_t)c * C < C ? len - (int64_t)c * C : C);
    const int64_t tok0 = start + (int64_t)c * C;
    // ---- gates (warp 0): G in log2 units, gamma, d = 2^(G_C - G), beta ----
    if (warp == 0) {
      constexpr int PER = C / 32;  // tokens per lane
      float x[PER], b[PER];
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int i = PER * lane + e;
        x[e] = 0.f;
        b[e] = 0.f;
        if (i < valid) {
          const size_t off = (size_t)(tok0 + i) * H + h;
          x[e] = p.g[off] * kLog2e;
          b[e] = beta_value(__bfloat162float(betap[off]), p.flags);
        }
        s += x[e];
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
      }
      float run = s;  // inclusive prefix through this lane's last token
#pragma unroll
      for (int e = PER - 1; e >= 0; --e) {
        sG[PER * lane + e] = run;
        run -= x[e];
      }
      const float Gl = __shfl_sync(0xffffffffu, s, 31);
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int i = PER * lane + e;
        const float Gi = sG[i];
        sGam[i] = ex2(Gi);
        sDec[i] = ex2(Gl - Gi);
        sBeta[i] = b[e];
      }
      if (lane == 0) sMisc[0] = ex2(Gl);
    }
    // ---- the chunk's tiles ----
    bool ok = true;
    if (tid == 0) {
      ok = mbar_wait_bounded(barTma, ph_tma, kWaitTimeoutNs);
      if (!ok) report(p.status, GDN_ERR_TIMEOUT, (uint32_t)n, (uint32_t)h, 41);
      tma_pending = !ok;
    }
    if (ok) ph_tma ^= 1;
    if (!__syncthreads_and(ok)) break;
    // ---- q/k row norms (folded into fp32 factors) ----
    if (l2 && tid < 2 * C) {
      const int i = tid % C;
      const uint32_t tb = sbase + (tid < C ? L::SQ : L::SK);
      float ss = 0.f;
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const uint4 x4 = S4(tile_addr(tb, i, 8 * q8));
        const uint32_t w[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
          ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
      }
      (tid < C ? sRq : sRk)[i] = rsqrtf(ss + 1e-6f);
    }
    // ---- S = [K; Q] K^T ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if constexpr (C == 32) {
          umma_bf16(tmem + TC::S, umma_desc_sw128(sbase + L::SK + kk * 32),
                    umma_desc_sw128(sbase + L::SK + kk * 32), umma_idesc_bf16(128, 32), kk > 0);
        } else {
          umma_bf16(tmem + TC::SA, umma_desc_sw128(sbase + L::SK + kk * 32),
                    umma_desc_sw128(sbase + L::SK + kk * 32), umma_idesc_bf16(128, 128), kk > 0);
          umma_bf16(tmem + TC::SP, umma_desc_sw128(sbase + L::SQ + kk * 32),
                    umma_desc_sw128(sbase + L::SK + kk * 32), umma_idesc_bf16(128, 128), kk > 0);
        }
      }
      umma_commit(barMma);
    }
    __syncthreads();  // the norms
    if (!wait_mma()) break;
    tc_fence_after();
    // ---- drains: A (fp32 16x16 blocks on or below the diagonal) and P (bf16) ----
    float *sA = reinterpret_cast<float *>(smem + L::OFF_A);
    auto drain16 = [&](uint32_t taddr, int i, int j0, bool isP) {
      // one row i, columns j0 .. j0 + 15 of the product in taddr's lane
      uint32_t v[16];
      tmem_ld16(taddr, v);
      tmem_wait_ld();
      const bool rowok = i < valid;
      const float Gi = sG[i];
      float rf = isP ? 1.f : sBeta[i];
      if (l2) rf *= isP ? sRq[i] : sRk[i];
      float val[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = j0 + e;
        const bool keep = rowok && (isP ? j <= i : j < i);
        float x = __uint_as_float(v[e]) * rf * ex2(Gi - sG[j < C ? j : C - 1]);
        if (l2) x *= sRk[j < C ? j : C - 1];
        val[e] = keep ? x : 0.f;
      }
      if (isP) {
        const uint32_t pb = sbase + L::OFF_P;
        S4(swz<L::PSUB>(pb, i, j0)) = make_uint4(pack_bf16(val[0], val[1]), pack_bf16(val[2], val[3]),
                                                 pack_bf16(val[4], val[5]), pack_bf16(val[6], val[7]));
        S4(swz<L::PSUB>(pb, i, j0 + 8)) =
            make_uint4(pack_bf16(val[8], val[9]), pack_bf16(val[10], val[11]),
                       pack_bf16(val[12], val[13]), pack_bf16(val[14], val[15]));
      } else if ((j0 >> 4) <= (i >> 4)) {
        const int rb = i >> 4, cbk = j0 >> 4;
        float *dst = sA + ((rb * (rb + 1)) / 2 + cbk) * L::A_BLK + (i & 15) * L::A_LD;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4 *>(dst + 4 * q) =
              make_float4(val[4 * q], val[4 * q + 1], val[4 * q + 2], val[4 * q + 3]);
      }
    };
    if constexpr (C == 32) {
      // quarter 0: A rows (K K^T), quarter 1: P rows (Q K^T); warps 0,1 take
      // columns 0..15, warps 4,5 columns 16..31
      if (wq < 2) {
        const int i = lane, j0 = warp >= 4 ? 16 : 0;
        drain16(tm(TC::S + j0), i, j0, wq == 1);
      }
    } else {
      // every quarter: rows 32 wq + lane of A and of P; the two warps of a
      // quarter split the 128 columns
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const int j0 = (warp >= 4 ? 64 : 0) + 16 * q, i = 32 * wq + lane;
        drain16(tm(TC::SA + j0), i, j0, false);
        drain16(tm(TC::SP + j0), i, j0, true);
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- prep: 16x16 diagonal inverses of (I + A) (fp32; one per half-warp),
    // stored over A_bb, and T_bb diag(beta gamma r_k) / T_bb diag(beta) in bf16
    // (column-major) for the substitution ----
    __nv_bfloat16 *sTB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_TB);
    __nv_bfloat16 *sMB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_MB);
    const uint32_t TBa = sbase + L::OFF_TB, MBa = sbase + L::OFF_MB;
    if (warp < NB / 2) {
      const int blk = 2 * warp + (lane >> 4), l = lane & 15;
      {
        const float *Ab = sA + ((blk * (blk + 1)) / 2 + blk) * L::A_BLK;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float s0 = (r == l) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
          for (int k4 = 0; k4 < r; k4 += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(Ab + r * L::A_LD + k4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (k4 + e < r) {
                if (e & 1) s1 = fmaf(-av[e], x[k4 + e], s1);
                else s0 = fmaf(-av[e], x[k4 + e], s0);
              }
            }
          }
          x[r] = s0 + s1;
        }
        __syncwarp();
        float *tcol = sA + ((blk * (blk + 1)) / 2 + blk) * L::A_BLK + l * L::A_LD;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4 *>(tcol + 4 * q) =
              make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        const int j = 16 * blk + l;
        const float bj = sBeta[j];
        float bgj = bj * sGam[j];
        if (l2) bgj *= sRk[j];
        uint32_t wg[8], wb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          wg[e] = pack_bf16(x[2 * e] * bgj, x[2 * e + 1] * bgj);
          wb[e] = pack_bf16(x[2 * e] * bj, x[2 * e + 1] * bj);
        }
        uint4 *tg = reinterpret_cast<uint4 *>(sTB + ((0 * NB + blk) * 16 + l) * L::TB_LD);
        uint4 *tb = reinterpret_cast<uint4 *>(sTB + ((1 * NB + blk) * 16 + l) * L::TB_LD);
        tg[0] = make_uint4(wg[0], wg[1], wg[2], wg[3]);
        tg[1] = make_uint4(wg[4], wg[5], wg[6], wg[7]);
        tb[0] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        tb[1] = make_uint4(wb[4], wb[5], wb[6], wb[7]);
      }
    }
    __syncthreads();
    // ---- couplings M_ik = T_ii A_ik (i > k) on tf32 tensor cores, stored negated ----
#pragma unroll 1
    for (int blk = warp; blk < L::NMB; blk += 8) {
      int i = 1;
      while ((i * (i + 1)) / 2 <= blk) ++i;  // blk in [i(i-1)/2, i(i+1)/2)
      const int k = blk - (i * (i - 1)) / 2;
      const float *Tm = sA + ((i * (i + 1)) / 2 + i) * L::A_BLK;  // T_ii, column-major
      const float *Ak = sA + ((i * (i + 1)) / 2 + k) * L::A_BLK;
      float acc[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t a0 = to_tf32(Tm[(8 * ks + t) * L::A_LD + g]);
        const uint32_t a1 = to_tf32(Tm[(8 * ks + t) * L::A_LD + g + 8]);
        const uint32_t a2 = to_tf32(Tm[(8 * ks + t + 4) * L::A_LD + g]);
        const uint32_t a3 = to_tf32(Tm[(8 * ks + t + 4) * L::A_LD + g + 8]);
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
    __syncthreads();
    // ---- left-looking substitution X_i = T_ii B_i + sum_{k<i} (-M_ik) X_k for
    // X = [W | U~], B = [K | V]: warp w takes 16 columns (warps 0-3 W, 4-7 U~);
    // a warp reads back only its own columns of earlier block rows ----
    {
      const int arow = lrow + (lmi & 1) * 8, acol = (lmi >> 1) * 8;
      const int trow = lrow + (lmi >> 1) * 8, tcol = (lmi & 1) * 8;  // column-major T tiles
      const bool isW = warp < 4;
      const uint32_t xt = sbase + (isW ? L::SW : L::SV), bsrc = sbase + (isW ? L::SK : L::SV);
      const int tbv = isW ? 0 : 1, col = 16 * (warp & 3);
#pragma unroll 1
      for (int lv = 0; lv < NB; ++lv) {
        float acc[2][4];
        {
          uint32_t ta[4], tb[4];
          ldsm_x4_t(TBa + (((tbv * NB + lv) * 16 + trow) * L::TB_LD + tcol) * 2, ta[0], ta[1],
                    ta[2], ta[3]);
          ldsm_x4_t(tile_addr(bsrc, 16 * lv + arow, col + acol), tb[0], tb[1], tb[2], tb[3]);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
            mma_bf16(acc[nt], ta[0], ta[1], ta[2], ta[3], tb[2 * nt], tb[2 * nt + 1]);
          }
        }
        // (U~ overwrites V row block lv only after V's rows lv were read above)
#pragma unroll 1
        for (int k = 0; k < lv; ++k) {
          const int blk = (lv * (lv - 1)) / 2 + k;
          uint32_t ma[4], xb[4];
          ldsm_x4(MBa + ((blk * 16 + arow) * L::TB_LD + acol) * 2, ma[0], ma[1], ma[2], ma[3]);
          ldsm_x4_t(tile_addr(xt, 16 * k + arow, col + acol), xb[0], xb[1], xb[2], xb[3]);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            mma_bf16(acc[nt], ma[0], ma[1], ma[2], ma[3], xb[2 * nt], xb[2 * nt + 1]);
        }
        __syncwarp();  // every lane has read row block lv of V (U~ goes over it)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            S1(tile_addr(xt, 16 * lv + g + 8 * hf, col + 8 * nt + 2 * t)) =
                pack_bf16(acc[nt][2 * hf], acc[nt][2 * hf + 1]);
        __syncwarp();
      }
    }
    fence_proxy_async_smem();  // W (and P, H) are read by the tensor cores
    __syncthreads();
    // ---- MMA1: Q H and W H ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bh = umma_desc_sw128_mn(sbase + L::OFF_H + kk * 2048, 8192);
        if constexpr (C == 32) {
          umma_bf16(tmem + TC::D1, umma_desc_sw128(sbase + L::SQ + kk * 32), bh,
                    umma_idesc_bf16(128, 64, 0, 1), kk > 0);
        } else {
          umma_bf16(tmem + TC::D1W, umma_desc_sw128(sbase + L::SW + kk * 32), bh,
                    umma_idesc_bf16(128, 64, 0, 1), kk > 0);
          umma_bf16(tmem + TC::D1Q, umma_desc_sw128(sbase + L::SQ + kk * 32), bh,
                    umma_idesc_bf16(128, 64, 0, 1), kk > 0);
        }
      }
      umma_commit(barMma);
    }
    if (!wait_mma()) break;
    tc_fence_after();
    // ---- E1: U = U~ - W H, Ud = diag(d r_k) U (bf16, row = token) ----
    auto e1_row = [&](uint32_t taddr, int i, int c0) {  // 32 columns c0.. of row i
      uint32_t w[32];
      tmem_ld32(taddr, w);
      uint4 xu[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) xu[q] = S4(tile_addr(sbase + L::SV, i, c0 + 8 * q));
      tmem_wait_ld();
      float di = sDec[i];
      if (l2) di *= sRk[i];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t x[4] = {xu[q].x, xu[q].y, xu[q].z, xu[q].w};
        uint32_t pu[4], pd[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float u0 = bf16_lo(x[e]) - __uint_as_float(w[8 * q + 2 * e]);
          const float u1 = bf16_hi(x[e]) - __uint_as_float(w[8 * q + 2 * e + 1]);
          pu[e] = pack_bf16(u0, u1);
          pd[e] = pack_bf16(u0 * di, u1 * di);
        }
        S4(tile_addr(sbase + L::OFF_U, i, c0 + 8 * q)) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
        S4(tile_addr(sbase + L::OFF_UD, i, c0 + 8 * q)) = make_uint4(pd[0], pd[1], pd[2], pd[3]);
      }
    };
    if constexpr (C == 32) {
      if (wq == 1) e1_row(tm(TC::D1 + cb), lane, cb);  // W H rows 32..63 (quarter 1)
    } else {
      e1_row(tm(TC::D1W + cb), 32 * wq + lane, cb);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    // ---- MMA3 (the state increment) and MMA2 (P U) ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        umma_bf16(tmem + TC::DH, umma_desc_sw128_mn(sbase + L::SK + kk * 2048, L::T),
                  umma_desc_sw128_mn(sbase + L::OFF_UD + kk * 2048, 8192),
                  umma_idesc_bf16(128, 64, 1, 1), kk > 0);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        umma_bf16(tmem + TC::PU,
                  umma_desc_sw128(sbase + L::OFF_P + (kk >> 2) * L::PSUB + (kk & 3) * 32),
                  umma_desc_sw128_mn(sbase + L::OFF_U + kk * 2048, 8192),
                  umma_idesc_bf16(128, 64, 0, 1), kk > 0);
      umma_commit(barMma);
    }
    if (!wait_mma()) break;
    tc_fence_after();
    // the slot is free: the next chunk's tiles load under the state update and output
    if (tid == 0 && c + 1 < nc) {
      load_tiles(c + 1);
      tma_pending = true;
    }
    // ---- E2a: H <- gamma_C H + K^T Ud ----
    if (is_state) {
      const float gC = sMisc[0];
      uint32_t w[32];
      tmem_ld32(tm(TC::DH + cb), w);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) hrow[j] = fmaf(gC, hrow[j], __uint_as_float(w[j]));
      store_h();
    }
    // ---- E2b: O = diag(gamma r_q) Q H + P U, then (o + D_h v) * gate ----
    auto out_row = [&](uint32_t tq, uint32_t tp, int i, int c0) {  // 32 columns c0.. of row i
      uint32_t a[32], b[32];
      tmem_ld32(tq, a);
      tmem_ld32(tp, b);
      tmem_wait_ld();
      if (i >= valid) return;
      float gi = sGam[i];
      if (l2) gi *= sRq[i];
      const size_t oidx = (size_t)(tok0 + i) * H + h;
      __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.o) + oidx * dv + col0 + c0;
      float og = 1.f;
      const __nv_bfloat16 *vrow = static_cast<const __nv_bfloat16 *>(p.v) + oidx * dv + col0 + c0;
      if (epi && p.out_gate) og = p.out_gate[oidx];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          o[e] = fmaf(gi, __uint_as_float(a[8 * q + e]), __uint_as_float(b[8 * q + e]));
        if (epi) {
          const uint4 v4 = reinterpret_cast<const uint4 *>(vrow)[q];
          const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[2 * e] = block_epilogue(o[2 * e], bf16_lo(vw[e]), dh, og);
            o[2 * e + 1] = block_epilogue(o[2 * e + 1], bf16_hi(vw[e]), dh, og);
          }
        }
        reinterpret_cast<uint4 *>(orow)[q] = make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]),
                                                        pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
      }
    };
    if constexpr (C == 32) {
      if (wq == 0) out_row(tm(TC::D1 + cb), tm(TC::PU + cb), lane, cb);  // rows 0..31
    } else {
      out_row(tm(TC::D1Q + cb), tm(TC::PU + cb), 32 * wq + lane, cb);
    }
    tc_fence_before();
    fence_proxy_async_smem();  // H for the next MMA1
    __syncthreads();
    ++done;
  }
  // a load still in flight lands before the CTA leaves
  if (tid == 0 && tma_pending) mbar_wait_bounded(barTma, ph_tma, kWaitTimeoutNs);
  // the state leaves through the E2a warps
  if (is_state && p.sN && done == nc) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4 *>(p.sN + state_row + 4 * q) =
          make_float4(hrow[4 * q], hrow[4 * q + 1], hrow[4 * q + 2], hrow[4 * q + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TC::ALLOC);
  }
}

template <int C>
cudaError_t launch_tcc(const FwdParams &p, cudaStream_t stream) {
  using L = LayoutC<C>;
  const int64_t tokens = p.cu ? p.seq_len : (int64_t)p.num_seqs * p.seq_len;
  CUtensorMap tq, tk, tv;
  if (!make_tmap(&tq, p.q, kDK, p.num_heads, tmap_rows(p, tokens, p.ext.q, kDK), C) ||
      !make_tmap(&tk, p.k, kDK, p.num_heads, tmap_rows(p, tokens, p.ext.k, kDK), C) ||
      !make_tmap(&tv, p.v, p.dv, p.num_heads, tmap_rows(p, tokens, p.ext.v, p.dv), C))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(gdn_fwd_tcc_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (err != cudaSuccess) return err;
  const dim3 grid(p.dv / kDvt, p.num_heads, p.num_seqs);
  gdn_fwd_tcc_kernel<C><<<grid, kThreadsC, L::ALLOC, stream>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace

bool tcc_supported(int chunk, int dk, int dv) {
  return (chunk == 32 || chunk == 128) && dk == 64 && dv % kDvt == 0;
}

cudaError_t launch_fwd_tcc(const FwdParams &p, int chunk, cudaStream_t stream) {
  switch (chunk) {
    case 32: return launch_tcc<32>(p, stream);
    case 128: return launch_tcc<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
