// Fused chunked forward of the gated delta rule for head_dim_k = 64, with every
// chunk product on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory) -- including the serial state chain.
//
// One CTA owns one (sequence, head, 64-wide slice of the value dimension) and
// walks that sequence's 64-token chunks in order ("Optimization Quartet",
// Triton GDN kernel section 3.2: intra-chunk parallel work, serial carry of the
// state; chunk size 64 per "v1.0 Architecture & Design Spec" section 2.3).
// The fp32 state never leaves the chip ("Model Architecture Walkthrough",
// section 6.3): it is held in registers by two carry warps, one key row per
// thread, and handed to the tensor cores as a bf16 shared-memory operand.
//
// Chunk algebra (gated delta rule, Yang et al. arXiv 2412.06464), H = S^T:
//   A = strictly_lower(diag(beta) K K^T (.) Gamma),  P = (Q K^T (.) Gamma)_{i>=j}
//   (I + A) W = diag(beta gamma) K,  (I + A) U~ = diag(beta) V      [prep warps]
//   U  = U~ - W H,   O = diag(gamma) Q H + P U,
//   H' = gamma_C H + K^T diag(exp(G_C - G)) U                        [carry]
// with gamma = exp(G), Gamma_ij = exp(G_i - G_j) ("Model Architecture
// Walkthrough", section 5.3.1).  The carry per chunk, all M = 128 products:
//   MMA1  D1  = [W; Q] H            rows 0..63 = W H, rows 64..127 = Q H
//   E1    U = U~ - W H, Ud = diag(exp(G_C - G)) U  -> shared (bf16, row-major)
//   MMA3  DH  = [K^T; *] Ud          rows 0..63 = K^T Ud  (the state increment)
//   MMA2  DPU = [*; P] U             rows 64..127 = P U
//   E2a   H <- gamma_C H + DH  (registers), bf16 copy -> shared for the next MMA1
//   E2b   O = diag(gamma) Q H + P U -> bf16 -> TMA store
// "*" rows are whatever finite tile precedes/follows in shared memory; their
// products land in accumulator rows nobody reads.  H, U and Ud are MN-major
// operands (row-major tiles, no transposes); K^T is the MN-major view of the
// TMA-loaded K tile.
//
// Roles (320 threads, one CTA per SM):
//   warp 8     producer: gate vectors + TMA loads of Q, K, V (ring of 3 slots)
//   warp 9     MMA issuer: one thread polls the ready-barriers of every
//              product and issues whichever is ready (tcgen05.mma + commit)
//   warps 0-3  prep: diagonal 16x16 inverses of (I + A) (fp32), couplings
//              (tf32 mma), blocked substitution for W (into the input slot,
//              right before Q) and U~ (bf16 mma); warps 0,1 first drain the
//              P rows of the chunk's Q K^T accumulator
//   warps 4,5  carry chain (E1, E2a), the state in registers
//   warps 6,7  output (E2b) + drain of the A rows of K K^T two chunks ahead
// Every wait is bounded; a timeout records GDN_ERR_TIMEOUT and ends the loops.
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

using namespace ptx;
using namespace tc;

constexpr int DK = 64, NIN = 3;
constexpr int kThreads64 = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr uint32_t kBarPrep = 1;
constexpr uint32_t kTmemCols = 512;
// TMEM column map: S double buffer, D1 double buffer, DPU double buffer, DH.
constexpr uint32_t kColS = 0, kColD1 = 128, kColPU = 256, kColH = 384;

constexpr uint32_t kIdescS = umma_idesc_bf16(128, 64);           // K-major x K-major
constexpr uint32_t kIdescKM = umma_idesc_bf16(128, 64, 0, 1);    // K-major A, MN-major B
constexpr uint32_t kIdescMM = umma_idesc_bf16(128, 64, 1, 1);    // MN-major A and B

struct L64 {
  static constexpr int SUB = 8192;
  // input slot: W (written by prep) | Q | K | V | gates  -> [W;Q] and [Q;K] contiguous
  static constexpr int SW = 0, SQ = SUB, SK = 2 * SUB, SV = 3 * SUB, SG = 4 * SUB;
  static constexpr int SLOT = 4 * SUB + 2048;
  // stage: U~ | P  -> [U~; P] contiguous
  static constexpr int TU = 0, TP = SUB;
  static constexpr int STAGE = 2 * SUB;
  static constexpr int OFF_IN = 0;
  static constexpr int OFF_ST = OFF_IN + NIN * SLOT;
  static constexpr int OFF_H = OFF_ST + 2 * STAGE;   // state H [dk][dv] bf16
  static constexpr int OFF_U = OFF_H + SUB;          // U  [token][dv] bf16
  static constexpr int OFF_UD = OFF_U + SUB;         // Ud [token][dv] bf16
  static constexpr int OFF_OST = OFF_UD + SUB;       // O staging [token][dv] bf16
  static constexpr int A_LD = 68;
  static constexpr int OFF_A = OFF_OST + SUB;        // f32 [2][64][A_LD]
  static constexpr int TF_LD = 20;
  static constexpr int OFF_TF = OFF_A + 2 * 64 * A_LD * 4;
  static constexpr int TB_LD = 24;
  static constexpr int OFF_TB = OFF_TF + 4 * 16 * TF_LD * 4;
  static constexpr int OFF_MB = OFF_TB + 2 * 4 * 16 * TB_LD * 2;
  static constexpr int OFF_GC = OFF_MB + 6 * 16 * TB_LD * 2;
  static constexpr int OFF_VOTE = OFF_GC + 64;
  static constexpr int OFF_TMEM = OFF_VOTE + 64;
  static constexpr int OFF_BAR = OFF_TMEM + 16;
  static constexpr int NBAR = 32;
  static constexpr int OFF_FLAG = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_FLAG + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(SLOT % 1024 == 0 && OFF_ST % 1024 == 0 && OFF_H % 1024 == 0, "alignment");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// mbarrier indices
enum : int {
  B_FULL_IN = 0,     // [3]  TMA bytes landed (+ producer arrival)
  B_EMPTY_IN = 3,    // [3]  carry warps done with the slot (128)
  B_FULL_ST = 6,     // [2]  prep wrote W and U~ (128)
  B_TMEM_FULL = 8,   // [2]  Q K^T / K K^T accumulator ready (commit)
  B_TMEM_EMPTY = 10, // [2]  ... drained (128)
  B_S_READY = 12,    // [2]  P and A in shared memory (128)
  B_H_READY = 14,    //      bf16 state written for the next MMA1 (64)
  B_D1_FULL = 15,    // [2]  MMA1 done (commit)
  B_D1_FREE = 17,    // [2]  D1 drained (128)
  B_U_READY = 19,    //      U and Ud written (64)
  B_DH_FULL = 20,    //      MMA3 done (commit)
  B_PU_FULL = 21,    // [2]  MMA2 done (commit)
  B_PU_FREE = 23,    // [2]  DPU drained (64)
  B_OST_FULL = 25,   //      O rows staged (64)
  B_OST_FREE = 26,   //      staging tile read by the store (1)
};

// One thread drains one row i of a 64-column fp32 accumulator of [Q; K] K^T
// (taddr: this warp's TMEM lane quarter at the buffer's first column) into a
// masked, decayed row of P (bf16, swizzled tile at Ps) or of A (fp32, Arow):
//   P_ij = S_ij 2^(G_i - G_j) (j <= i),   A_ij = beta_i S_ij 2^(G_i - G_j) (j < i)
// with G in log2 units.  The warp owns rows 32*half .. 32*half+31.  Per
// 16-column block: blocks after those rows are zero (no load, no arithmetic);
// blocks before them use two factors that are both <= 1,
// 2^(G_i - G_b) * E_j with E_j = 2^(G_b - G_j) precomputed per token (b the
// block's last token); the two blocks that meet the rows take one exponent
// per element.  One shared (not inlined) copy keeps the instruction footprint
// small.
__device__ __noinline__ void drain_s_row(uint32_t taddr, const float *G2, const float *E, int i,
                                         int half, bool isP, float bi, int ilim, bool rowok,
                                         uint32_t Ps, float *Arow, uint8_t *smem,
                                         uint32_t sbase) {
  const float Gi = G2[i];
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    float val[16];
    if (cb >= 2 * half + 2) {  // entirely above the diagonal for these rows
      if (!isP) continue;
#pragma unroll
      for (int e = 0; e < 16; ++e) val[e] = 0.f;
    } else {
      uint32_t v[16];
      tmem_ld16(taddr + 16 * cb, v);
      float f[16];
      const bool before = cb < 2 * half;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = *reinterpret_cast<const float4 *>((before ? E : G2) + 16 * cb + 4 * q);
        f[4 * q] = x.x;
        f[4 * q + 1] = x.y;
        f[4 * q + 2] = x.z;
        f[4 * q + 3] = x.w;
      }
      const float scale = before ? bi * ex2(Gi - G2[16 * cb + 15]) : bi;
      tmem_wait_ld();
      if (before) {
#pragma unroll
        for (int e = 0; e < 16; ++e) val[e] = rowok ? __uint_as_float(v[e]) * scale * f[e] : 0.f;
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = 16 * cb + e;
          const float x = __uint_as_float(v[e]) * scale * ex2(Gi - f[e]);
          val[e] = (rowok && j < ilim) ? x : 0.f;
        }
      }
    }
    if (isP) {
      *reinterpret_cast<uint4 *>(smem + (tile_addr(Ps, i, 16 * cb) - sbase)) =
          make_uint4(pack_bf16(val[0], val[1]), pack_bf16(val[2], val[3]),
                     pack_bf16(val[4], val[5]), pack_bf16(val[6], val[7]));
      *reinterpret_cast<uint4 *>(smem + (tile_addr(Ps, i, 16 * cb + 8) - sbase)) =
          make_uint4(pack_bf16(val[8], val[9]), pack_bf16(val[10], val[11]),
                     pack_bf16(val[12], val[13]), pack_bf16(val[14], val[15]));
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4 *>(Arow + 16 * cb + 4 * q) =
            make_float4(val[4 * q], val[4 * q + 1], val[4 * q + 2], val[4 * q + 3]);
    }
  }
}

__global__ void __launch_bounds__(kThreads64, 1)
gdn_fwd_tc64_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_o) {
  using L = L64;
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
  const int nc = (int)((len + 63) / 64);

  Shared S;
  S.abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_FLAG);
  int *votes = reinterpret_cast<int *>(smem + L::OFF_VOTE);
  float *sgc = reinterpret_cast<float *>(smem + L::OFF_GC);
  auto bar = [&](int i) { return sbase + L::OFF_BAR + 8u * i; };
  auto slot_base = [&](int s) { return sbase + L::OFF_IN + s * L::SLOT; };
  auto stage_base = [&](int s) { return sbase + L::OFF_ST + s * L::STAGE; };
  auto gate_ptr = [&](int s) {
    return reinterpret_cast<float *>(smem + L::OFF_IN + s * L::SLOT + L::SG);
  };
  auto valid_rows = [&](int c) {
    return (int)(len - (int64_t)c * 64 < 64 ? len - (int64_t)c * 64 : 64);
  };

  if (tid == 0) {
    for (int s = 0; s < NIN; ++s) {
      mbar_init(bar(B_FULL_IN + s), 1);
      mbar_init(bar(B_EMPTY_IN + s), 128);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_FULL_ST + s), 128);
      mbar_init(bar(B_TMEM_FULL + s), 1);
      mbar_init(bar(B_TMEM_EMPTY + s), 128);
      mbar_init(bar(B_S_READY + s), 128);
      mbar_init(bar(B_D1_FULL + s), 1);
      mbar_init(bar(B_D1_FREE + s), 128);
      mbar_init(bar(B_PU_FULL + s), 1);
      mbar_init(bar(B_PU_FREE + s), 64);
    }
    mbar_init(bar(B_H_READY), 64);
    mbar_init(bar(B_U_READY), 64);
    mbar_init(bar(B_DH_FULL), 1);
    mbar_init(bar(B_OST_FULL), 64);
    mbar_init(bar(B_OST_FREE), 1);
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
  // plain shared-memory accesses at a byte address (left to the compiler to schedule)
  auto S4 = [&](uint32_t addr) -> uint4 & { return *reinterpret_cast<uint4 *>(smem + (addr - sbase)); };
  auto S1 = [&](uint32_t addr) -> uint32_t & {
    return *reinterpret_cast<uint32_t *>(smem + (addr - sbase));
  };

  // Drain the [Q; K] K^T accumulator of chunk cc.  A warp reaches the TMEM lane
  // quarter warp % 4: quarters 0,1 hold rows of P = Q K^T (drained by prep warps
  // 0,1), quarters 2,3 rows of A = K K^T (drained by the output warps 6,7).
  auto s_epilogue = [&](int cc) -> bool {
  const int wq = warp & 3;
  const bool chain = wq < 2;  // P rows
  const int row = 32 * (wq & 1) + lane;
  const int cw = wq;
  auto tm = [&](uint32_t col) { return tmem_base + ((uint32_t)(32 * wq) << 16) + col; };
    const int slot = cc % NIN, buf = cc & 1;
    [[maybe_unused]] const int c = cc;  // chunk index of the phase stamps
    GDN_PHASE(8);
    bool ok = role_wait(bar(B_TMEM_FULL + buf), (cc >> 1) & 1, S, p, n, h, 7);
    if (ok) ok = role_wait(bar(B_FULL_IN + slot), (cc / NIN) & 1, S, p, n, h, 8);
    // the P tile of this stage was last read by MMA2 of chunk cc-2
    if (ok && chain && cc >= 2)
      ok = role_wait(bar(B_PU_FULL + buf), ((cc - 2) >> 1) & 1, S, p, n, h, 10);
    GDN_PHASE(9);
    if (!__all_sync(0xffffffffu, ok)) return false;
    tc_fence_after();
    const int valid = valid_rows(cc);
    const float *gate = gate_ptr(slot);
    const float *G2 = gate, *beta = gate + 192, *E = gate + 256;
    const bool isP = chain;
    const int i = row;
    const int ilim = isP ? i + 1 : i;  // P keeps j <= i, A keeps j < i
    const bool rowok = i < valid;
    const float bi = isP ? 1.f : beta[i];
    const uint32_t Ps = stage_base(buf) + L::TP;
    float *Arow = reinterpret_cast<float *>(smem + L::OFF_A) + (buf * 64 + i) * L::A_LD;
    drain_s_row(tm(kColS + buf * 64), G2, E, i, cw & 1, isP, bi, ilim, rowok, Ps, Arow, smem,
                sbase);
    tc_fence_before();
    mbar_arrive(bar(B_TMEM_EMPTY + buf));
    if (isP) fence_proxy_async_smem();
    GDN_PHASE(10);
    mbar_arrive(bar(B_S_READY + buf));
    return true;
  };


  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const __nv_bfloat16 *betap = static_cast<const __nv_bfloat16 *>(p.beta);
    float gv0 = 0.f, gv1 = 0.f, bv0 = 0.f, bv1 = 0.f;
    auto load_gates = [&](int c) {
      gv0 = gv1 = bv0 = bv1 = 0.f;
      const int64_t t0 = (int64_t)c * 64 + 2 * lane;
      if (c < nc && t0 < len) {
        const size_t off = (size_t)(start + t0) * H + h;
        gv0 = p.g[off];
        bv0 = __bfloat162float(betap[off]);
        if (t0 + 1 < len) {
          gv1 = p.g[off + H];
          bv1 = __bfloat162float(betap[off + H]);
        }
      }
    };
    load_gates(0);
    constexpr uint32_t kTx = 3 * L::SUB;
    int issued = 0;
    for (int c = 0; c < nc; ++c) {
      const int slot = c % NIN;
      GDN_PHASE(0);
      bool ok = true;
      if (c >= NIN) ok = role_wait(bar(B_EMPTY_IN + slot), ((c / NIN) - 1) & 1, S, p, n, h, 1);
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
      }
      load_gates(c + 1);
      __syncwarp();
      if (lane == 0) {
        const uint32_t sb = slot_base(slot);
        const int row = (int)(start + (int64_t)c * 64);
        mbar_arrive_expect_tx(bar(B_FULL_IN + slot), kTx);
        tma_load_3d(sb + L::SQ, &tmap_q, 0, h, row, bar(B_FULL_IN + slot));
        tma_load_3d(sb + L::SK, &tmap_k, 0, h, row, bar(B_FULL_IN + slot));
        tma_load_3d(sb + L::SV, &tmap_v, col0, h, row, bar(B_FULL_IN + slot));
      }
      GDN_PHASE(2);
      ++issued;
    }
    if (lane == 0)
      for (int c = issued - NIN < 0 ? 0 : issued - NIN; c < issued; ++c)
        mbar_wait_bounded(bar(B_FULL_IN + c % NIN), (c / NIN) & 1, kWaitTimeoutNs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // One thread polls the barriers of three independent product streams and
    // issues whichever is ready: Q K^T of chunk cs, MMA1 of chunk c1, MMA3 and
    // MMA2 of chunk c3 (c3 <= c1 <= c3 + 1 keeps one carry product in flight).
    if (lane == 0) {
      int cs = 0, c1 = 0, c3 = 0;
      uint64_t last = globaltimer_ns();
      uint32_t spins = 0;
      while (c3 < nc) {
        bool prog = false;
        if (cs < nc && mbar_test(bar(B_FULL_IN + cs % NIN), (cs / NIN) & 1) &&
            (cs < 2 || mbar_test(bar(B_TMEM_EMPTY + (cs & 1)), ((cs >> 1) - 1) & 1))) {
          tc_fence_after();
          const uint32_t a = slot_base(cs % NIN) + L::SQ;  // [Q; K]
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem_base + kColS + (cs & 1) * 64, umma_desc_sw128(a + kk * 32),
                      umma_desc_sw128(a + L::SUB + kk * 32), kIdescS, kk > 0);
          umma_commit(bar(B_TMEM_FULL + (cs & 1)));
          ++cs;
          prog = true;
        }
        if (c1 < nc && c1 == c3 && mbar_test(bar(B_FULL_ST + (c1 & 1)), (c1 >> 1) & 1) &&
            mbar_test(bar(B_H_READY), c1 & 1) &&
            (c1 < 2 || mbar_test(bar(B_D1_FREE + (c1 & 1)), ((c1 >> 1) - 1) & 1))) {
          tc_fence_after();
          const uint32_t a = slot_base(c1 % NIN) + L::SW;  // [W; Q]
          const uint32_t b = sbase + L::OFF_H;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem_base + kColD1 + (c1 & 1) * 64, umma_desc_sw128(a + kk * 32),
                      umma_desc_sw128_mn(b + kk * 2048, L::SUB), kIdescKM, kk > 0);
          umma_commit(bar(B_D1_FULL + (c1 & 1)));
          ++c1;
          prog = true;
        }
        if (c3 < c1 && mbar_test(bar(B_U_READY), c3 & 1) &&
            (c3 < 2 || mbar_test(bar(B_PU_FREE + (c3 & 1)), ((c3 >> 1) - 1) & 1))) {
          tc_fence_after();
          // MMA3: state increment [K^T; V^T] Ud (K^T = MN-major view of the K tile;
          // the V tile is the second, unread, M block)
          const uint32_t kt = slot_base(c3 % NIN) + L::SK;
          const uint32_t ud = sbase + L::OFF_UD, u = sbase + L::OFF_U;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem_base + kColH, umma_desc_sw128_mn(kt + kk * 2048, L::SUB),
                      umma_desc_sw128_mn(ud + kk * 2048, L::SUB), kIdescMM, kk > 0);
          umma_commit(bar(B_DH_FULL));
          // MMA2: [U~; P] U  (rows 64..127 = P U)
          const uint32_t ap = stage_base(c3 & 1) + L::TU;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem_base + kColPU + (c3 & 1) * 64, umma_desc_sw128(ap + kk * 32),
                      umma_desc_sw128_mn(u + kk * 2048, L::SUB), kIdescKM, kk > 0);
          umma_commit(bar(B_PU_FULL + (c3 & 1)));
          ++c3;
          prog = true;
        }
        if (prog) {
          spins = 0;
        } else if (__nanosleep(20), (++spins & 255u) == 0) {  // back off: leave issue slots to the warps sharing this SMSP
          const uint64_t now = globaltimer_ns();
          if (*S.abort_flag) break;
          if (spins == 256) last = now;
          else if (now - last > kWaitTimeoutNs) {
            *S.abort_flag = 1;
            report(p.status, GDN_ERR_TIMEOUT, (uint32_t)n, (uint32_t)h, 9);
            break;
          }
        }
      }
      // every issued MMA has completed before tensor memory is released
      if (c3 > 0) {
        mbar_wait_bounded(bar(B_PU_FULL + ((c3 - 1) & 1)), ((c3 - 1) >> 1) & 1, kWaitTimeoutNs);
        mbar_wait_bounded(bar(B_DH_FULL), (c3 - 1) & 1, kWaitTimeoutNs);
      }
      if (c1 > c3) mbar_wait_bounded(bar(B_D1_FULL + ((c1 - 1) & 1)), ((c1 - 1) >> 1) & 1, kWaitTimeoutNs);
      if (cs > 0) mbar_wait_bounded(bar(B_TMEM_FULL + ((cs - 1) & 1)), ((cs - 1) >> 1) & 1, kWaitTimeoutNs);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ prep
    const int ptid = tid;
    float *sTf = reinterpret_cast<float *>(smem + L::OFF_TF);
    __nv_bfloat16 *sTB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_TB);
    __nv_bfloat16 *sMB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_MB);
    const uint32_t TBa = smem_u32(sTB), MBa = smem_u32(sMB);
    int *vote = votes;

    for (int c = 0; c < nc; ++c) {
      const int slot = c % NIN, stage = c & 1;
      const int valid = valid_rows(c);
      GDN_PHASE(0);
      // warps 0,1 drain the P rows of this chunk's [Q; K] K^T accumulator
      bool ok = warp < 2 ? s_epilogue(c) : true;
      // P and A of this chunk are in shared memory; the carry is done with the
      // stage's previous contents (the P drain waited for MMA2 of chunk c-2)
      if (ok) ok = role_wait(bar(B_S_READY + stage), (c >> 1) & 1, S, p, n, h, 2);
      if (ok) ok = role_wait(bar(B_FULL_IN + slot), (c / NIN) & 1, S, p, n, h, 3);
      ok = __all_sync(0xffffffffu, ok) && !*S.abort_flag;
      GDN_PHASE(1);

      const uint32_t sb = slot_base(slot);
      const uint32_t Ws = sb + L::SW, Qs = sb + L::SQ, Ks = sb + L::SK, Vs = sb + L::SV;
      const float *gate = gate_ptr(slot);
      const float *gam = gate + 64, *beta = gate + 192;
      const float *sA = reinterpret_cast<const float *>(smem + L::OFF_A) + stage * 64 * L::A_LD;
      const uint32_t Us = stage_base(stage) + L::TU;

      // rows past the end of the sequence: zero Q, K, V (the Q K^T MMA has read them)
      if (ok && valid < 64) {
        for (int idx = ptid; idx < (64 - valid) * 24; idx += 128) {
          const int row = valid + idx / 24, q = idx % 24;
          const uint32_t a = tile_addr(q < 8 ? Qs : (q < 16 ? Ks : Vs), row, (q & 7) * 8);
          S4(a) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (lane == 0) vote[(c & 1) * 4 + warp] = ok ? 1 : 0;
      named_sync(kBarPrep, 128);
      GDN_PHASE(2);
      {
        const int *v = vote + (c & 1) * 4;
        if (!(v[0] && v[1] && v[2] && v[3])) break;
      }

      // ---- 16x16 diagonal blocks of T = (I + A)^-1 (right-looking, fp32) ----
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
        const float bgj = bj * gam[16 * w + l];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          sTf[(w * 16 + r) * L::TF_LD + l] = x[r];
          sTB[((0 * 4 + w) * 16 + r) * L::TB_LD + l] = __float2bfloat16_rn(x[r] * bgj);
          sTB[((1 * 4 + w) * 16 + r) * L::TB_LD + l] = __float2bfloat16_rn(x[r] * bj);
        }
      }
      GDN_PHASE(3);
      named_sync(kBarPrep, 128);
      GDN_PHASE(4);

      // ---- M_ik = T_ii A_ik (i > k) on tf32 tensor cores, stored negated (bf16) ----
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
      named_sync(kBarPrep, 128);
      GDN_PHASE(6);

      // ---- block forward substitution: X_i = T_ii B_i + sum_k (-M_ik) X_k, X = [W | U~] ----
      {
        constexpr int PPW = 2;  // 16-column pairs per warp: warps 0,1 -> W, warps 2,3 -> U~
        const int arow = lrow + (lmi & 1) * 8, acol = (lmi >> 1) * 8;
        const bool isW = warp < 2;
        const uint32_t xt = isW ? Ws : Us;
        const uint32_t bsrc = isW ? Ks : Vs;
        const int tbv = isW ? 0 : 1;
        float lacc[4][PPW][2][4];
        {
          // T_ii B_i for every block row: all operand loads first, then the products
          uint32_t ta[4][4], tb[4][PPW][4];
#pragma unroll
          for (int lv = 0; lv < 4; ++lv) {
            ldsm_x4(TBa + (((tbv * 4 + lv) * 16 + arow) * L::TB_LD + acol) * 2, ta[lv][0],
                    ta[lv][1], ta[lv][2], ta[lv][3]);
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp) {
              const int col = 32 * (warp & 1) + 16 * pp;
              ldsm_x4_t(tile_addr(bsrc, 16 * lv + lrow + (lmi & 1) * 8, col + (lmi >> 1) * 8),
                        tb[lv][pp][0], tb[lv][pp][1], tb[lv][pp][2], tb[lv][pp][3]);
            }
          }
#pragma unroll
          for (int lv = 0; lv < 4; ++lv)
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) lacc[lv][pp][nt][e] = 0.f;
                mma_bf16(lacc[lv][pp][nt], ta[lv][0], ta[lv][1], ta[lv][2], ta[lv][3],
                         tb[lv][pp][2 * nt], tb[lv][pp][2 * nt + 1]);
              }
        }
#pragma unroll
        for (int lv = 0; lv < 4; ++lv) {
          if (lv > 0) {
            // X_{lv-1} (just written by all prep warps) and every coupling M_{l2, lv-1}
            uint32_t xb[PPW][4], ma[4][4];
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp) {
              const int col = 32 * (warp & 1) + 16 * pp;
              ldsm_x4_t(tile_addr(xt, 16 * (lv - 1) + lrow + (lmi & 1) * 8, col + (lmi >> 1) * 8),
                        xb[pp][0], xb[pp][1], xb[pp][2], xb[pp][3]);
            }
#pragma unroll
            for (int l2 = lv; l2 < 4; ++l2) {
              const int blk = (l2 * (l2 - 1)) / 2 + (lv - 1);
              ldsm_x4(MBa + ((blk * 16 + arow) * L::TB_LD + acol) * 2, ma[l2][0], ma[l2][1],
                      ma[l2][2], ma[l2][3]);
            }
            // the product on the critical path first
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
                mma_bf16(lacc[lv][pp][nt], ma[lv][0], ma[lv][1], ma[lv][2], ma[lv][3],
                         xb[pp][2 * nt], xb[pp][2 * nt + 1]);
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp) {
              const int col = 32 * (warp & 1) + 16 * pp;
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                  S1(tile_addr(xt, 16 * lv + g + 8 * hf, col + 8 * nt + 2 * t)) =
                      pack_bf16(lacc[lv][pp][nt][2 * hf], lacc[lv][pp][nt][2 * hf + 1]);
            }
            // X_{lv-1} terms of the later block rows, while the other warps catch up
#pragma unroll
            for (int l2 = lv + 1; l2 < 4; ++l2)
#pragma unroll
              for (int pp = 0; pp < PPW; ++pp)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                  mma_bf16(lacc[l2][pp][nt], ma[l2][0], ma[l2][1], ma[l2][2], ma[l2][3],
                           xb[pp][2 * nt], xb[pp][2 * nt + 1]);
          } else {
#pragma unroll
            for (int pp = 0; pp < PPW; ++pp) {
              const int col = 32 * (warp & 1) + 16 * pp;
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                  S1(tile_addr(xt, 16 * lv + g + 8 * hf, col + 8 * nt + 2 * t)) =
                      pack_bf16(lacc[lv][pp][nt][2 * hf], lacc[lv][pp][nt][2 * hf + 1]);
            }
          }
          if (lv < 3) named_sync(kBarPrep, 128);
        }
      }
      // W, U~ and the zeroed rows are read by the tensor cores (async proxy)
      fence_proxy_async_smem();
      GDN_PHASE(7);
      mbar_arrive(bar(B_FULL_ST + stage));
    }
  } else {
    // ------------------------------------------------------------ carry / output
    const int cw = warp - 4;             // TMEM lane quarter of this warp
    const int r = 32 * cw + lane;        // TMEM lane = accumulator row
    const bool chain = cw < 2;           // warps 4,5: state chain; warps 6,7: output
    const int row = chain ? r : r - 64;  // key row (chain) or token (output)
    const size_t state_row =
        ((size_t)n * H + h) * (size_t)DK * dv + (size_t)row * dv + col0;
    auto tm = [&](uint32_t col) { return tmem_base + ((uint32_t)(32 * cw) << 16) + col; };

    // the state row of this thread (warps 4,5): H[row][0..63], fp32
    float hrow[64];
    const uint32_t Hs = sbase + L::OFF_H, Ust = sbase + L::OFF_U, Uds = sbase + L::OFF_UD;
    auto store_row_bf16 = [&](uint32_t tilebase, int rr, const float *x) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        S4(tile_addr(tilebase, rr, 8 * q)) =
            make_uint4(pack_bf16(x[8 * q], x[8 * q + 1]), pack_bf16(x[8 * q + 2], x[8 * q + 3]),
                       pack_bf16(x[8 * q + 4], x[8 * q + 5]), pack_bf16(x[8 * q + 6], x[8 * q + 7]));
    };
    if (chain) {
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.s0) v4 = *reinterpret_cast<const float4 *>(p.s0 + state_row + 4 * q);
        hrow[4 * q] = v4.x;
        hrow[4 * q + 1] = v4.y;
        hrow[4 * q + 2] = v4.z;
        hrow[4 * q + 3] = v4.w;
      }
      store_row_bf16(Hs, row, hrow);
      fence_proxy_async_smem();
      mbar_arrive(bar(B_H_READY));
    }

    // chain warps: chunks 0 .. nc-1.  Output warps: chunks -2 .. nc-1, draining
    // the A rows of chunk c+2 after storing O of chunk c.
    bool alive = true;
    for (int c = chain ? 0 : -2; c < nc && alive; ++c) {
      const int slot = (c + NIN) % NIN, buf = c & 1;
      const int valid = valid_rows(c);
      const float *gate = gate_ptr(slot);
      if (chain) {
        // ---- E1: U = U~ - W H (row = token), Ud = U * exp(G_C - G) ----
        GDN_PHASE(0);
        bool ok = role_wait(bar(B_D1_FULL + buf), (c >> 1) & 1, S, p, n, h, 11);
        if (!__all_sync(0xffffffffu, ok)) break;
        GDN_PHASE(1);
        tc_fence_after();
        {
          const uint32_t Ut = stage_base(buf) + L::TU;
          const float dj = gate[128 + row];
          GDN_PHASE(10);
          // compact loop over 16-column slices (keeps this code resident in the
          // instruction cache between chunks)
#pragma unroll 1
          for (int q2 = 0; q2 < 4; ++q2) {
            uint32_t w[16];
            tmem_ld16(tm(kColD1 + buf * 64 + 16 * q2), w);
            const uint4 xa = S4(tile_addr(Ut, row, 16 * q2)), xb = S4(tile_addr(Ut, row, 16 * q2 + 8));
            tmem_wait_ld();
            const uint32_t x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
            uint32_t pu[8], pd[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float u0 = bf16_lo(x[e]) - __uint_as_float(w[2 * e]);
              const float u1 = bf16_hi(x[e]) - __uint_as_float(w[2 * e + 1]);
              pu[e] = pack_bf16(u0, u1);
              pd[e] = pack_bf16(u0 * dj, u1 * dj);
            }
            S4(tile_addr(Ust, row, 16 * q2)) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
            S4(tile_addr(Ust, row, 16 * q2 + 8)) = make_uint4(pu[4], pu[5], pu[6], pu[7]);
            S4(tile_addr(Uds, row, 16 * q2)) = make_uint4(pd[0], pd[1], pd[2], pd[3]);
            S4(tile_addr(Uds, row, 16 * q2 + 8)) = make_uint4(pd[4], pd[5], pd[6], pd[7]);
          }
          tc_fence_before();
          mbar_arrive(bar(B_D1_FREE + buf));
        }
        GDN_PHASE(11);
        fence_proxy_async_smem();
        GDN_PHASE(12);
        mbar_arrive(bar(B_U_READY));
        GDN_PHASE(2);

        // ---- E2a: H <- gamma_C H + K^T Ud (row = key index) ----
        ok = role_wait(bar(B_DH_FULL), c & 1, S, p, n, h, 12);
        if (!__all_sync(0xffffffffu, ok)) break;
        GDN_PHASE(3);
        tc_fence_after();
        {
          const float gC = sgc[slot];
          uint32_t wa[32], wb[32];
          tmem_ld32(tm(kColH), wa);
          tmem_ld32(tm(kColH + 32), wb);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            hrow[j] = fmaf(gC, hrow[j], __uint_as_float(wa[j]));
            hrow[32 + j] = fmaf(gC, hrow[32 + j], __uint_as_float(wb[j]));
          }
        }
        tc_fence_before();
        store_row_bf16(Hs, row, hrow);
        fence_proxy_async_smem();
        mbar_arrive(bar(B_H_READY));
        mbar_arrive(bar(B_EMPTY_IN + slot));
        GDN_PHASE(4);
      } else if (c >= 0) {
        // ---- E2b: O = diag(gamma) (Q H) + P U (row = token), then store ----
        GDN_PHASE(0);
        bool ok = role_wait(bar(B_PU_FULL + buf), (c >> 1) & 1, S, p, n, h, 13);
        if (!__all_sync(0xffffffffu, ok)) break;
        GDN_PHASE(1);
        tc_fence_after();
        // the staging tile must have been read by the previous chunk's store
        if (c > 0) ok = role_wait(bar(B_OST_FREE), (c - 1) & 1, S, p, n, h, 14);
        if (!__all_sync(0xffffffffu, ok)) break;
        {
          const float gi = gate[64 + row];
          const bool full = valid == 64;
          __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.o) +
                                ((size_t)(start + (int64_t)c * 64 + row) * H + h) * dv + col0;
#pragma unroll 1
          for (int q2 = 0; q2 < 4; ++q2) {
            uint32_t a[16], b[16];
            tmem_ld16(tm(kColD1 + buf * 64 + 16 * q2), a);
            tmem_ld16(tm(kColPU + buf * 64 + 16 * q2), b);
            tmem_wait_ld();
            uint32_t w8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w8[e] = pack_bf16(fmaf(gi, __uint_as_float(a[2 * e]), __uint_as_float(b[2 * e])),
                                fmaf(gi, __uint_as_float(a[2 * e + 1]), __uint_as_float(b[2 * e + 1])));
            const uint4 lo = make_uint4(w8[0], w8[1], w8[2], w8[3]);
            const uint4 hi = make_uint4(w8[4], w8[5], w8[6], w8[7]);
            if (full) {
              S4(tile_addr(sbase + L::OFF_OST, row, 16 * q2)) = lo;
              S4(tile_addr(sbase + L::OFF_OST, row, 16 * q2 + 8)) = hi;
            } else if (row < valid) {  // last partial chunk: this thread's row, directly
              *reinterpret_cast<uint4 *>(orow + 16 * q2) = lo;
              *reinterpret_cast<uint4 *>(orow + 16 * q2 + 8) = hi;
            }
          }
          tc_fence_before();
          mbar_arrive(bar(B_D1_FREE + buf));
          mbar_arrive(bar(B_PU_FREE + buf));
          if (full) fence_proxy_async_smem();
          mbar_arrive(bar(B_EMPTY_IN + slot));
          mbar_arrive(bar(B_OST_FULL));
          GDN_PHASE(2);
          if (r == 64) {  // one thread stores the tile and frees it once read
            ok = role_wait(bar(B_OST_FULL), c & 1, S, p, n, h, 15);
            if (ok && full) {
              tma_store_3d(&tmap_o, col0, h, (int)(start + (int64_t)c * 64), sbase + L::OFF_OST);
              bulk_commit();
              bulk_wait_read<0>();
            }
            mbar_arrive(bar(B_OST_FREE));
          }
        }
        GDN_PHASE(3);
      }
      // output warps: the A rows of the accumulator two chunks ahead
      if (!chain && c + 2 < nc) alive = s_epilogue(c + 2);
      GDN_PHASE(7);
    }
    if (r == 64) bulk_wait_all();  // every O store has completed
    if (chain && p.sN && !*S.abort_flag) {
#pragma unroll
      for (int q = 0; q < 16; ++q)
        *reinterpret_cast<float4 *>(p.sN + state_row + 4 * q) =
            make_float4(hrow[4 * q], hrow[4 * q + 1], hrow[4 * q + 2], hrow[4 * q + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fwd_tc64(const FwdParams &p, cudaStream_t stream) {
  using L = L64;
  const int64_t tokens = p.cu ? p.seq_len : (int64_t)p.num_seqs * p.seq_len;
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap(&tq, p.q, DK, p.num_heads, tokens) ||
      !make_tmap(&tk, p.k, DK, p.num_heads, tokens) ||
      !make_tmap(&tv, p.v, p.dv, p.num_heads, tokens) ||
      !make_tmap(&to, p.o, p.dv, p.num_heads, tokens))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(gdn_fwd_tc64_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (err != cudaSuccess) return err;
  const dim3 grid(p.dv / kDvt, p.num_heads, p.num_seqs);
  gdn_fwd_tc64_kernel<<<grid, kThreads64, L::ALLOC, stream>>>(p, tq, tk, tv, to);
  return cudaGetLastError();
}

}  // namespace gdn

#ifdef GDN_PHASE_PROBE
extern "C" int gdn_phase_probe_read(unsigned long long *host) {
  return (int)cudaMemcpyFromSymbol(host, gdn::tc::g_phase_probe, sizeof(gdn::tc::g_phase_probe));
}
#endif
