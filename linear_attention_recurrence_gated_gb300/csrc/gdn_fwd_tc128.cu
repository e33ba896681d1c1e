// Fused chunked forward of the gated delta rule for head_dim_k = 128, with
// every chunk product on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory) -- including the serial state chain.  It is
// the head_dim_k = 64 kernel's design (gdn_fwd_tc64.cu) carried to a key
// dimension of two 64-column groups; the differences are listed below.
//
// One CTA owns one (sequence, head, 64-wide slice of the value dimension) and
// walks that sequence's 64-token chunks in order ("Optimization Quartet",
// Triton GDN kernel section 3.2: intra-chunk parallel work, serial carry of the
// state; chunk size 64 per "v1.0 Architecture & Design Spec" section 2.3).
// The fp32 state never leaves the chip ("Model Architecture Walkthrough",
// section 6.3): it is held in registers by the E2a warps, one key row per
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
//   MMA3  DH  = K^T Ud               all 128 rows (the state increment)
//   MMA2  DPU = [*; P] U             rows 64..127 = P U
//   E2a   H <- gamma_C H + DH  (registers), bf16 copy -> shared for the next MMA1
//   E2b   O = diag(gamma) Q H + P U -> bf16 -> global
// The key dimension comes in two 64-column groups g, and an input slot holds
// [W_g Q_g K_g] for each, so [W_g; Q_g] and [Q_g; K_g] are contiguous M = 128
// operands whose K steps walk the groups, and K^T = [K_0^T; K_1^T] is one
// MN-major M = 128 operand over both groups.  "*" rows are whatever finite
// tile precedes P in shared memory; their products land in rows nobody reads.
//
// Roles (24 warps, one CTA per SM; warp w reaches the TMEM lanes
// 32*(w%4)..+31 and issues on SM sub-partition w%4):
//   warp 16        producer: gate vectors + TMA loads of Q, K (two boxes
//                  each), V (ring of 2 slots of 57 KB), L2 prefetch
//   warp 13        [Q; K] K^T issuer (tcgen05.mma + commit); owns tensor memory
//   warps 8,9      drain the P rows of [Q; K] K^T (masked decay, bf16)
//   warps 18,19    drain the A rows (masked decay and beta, fp32)
//   warps 2,3,14,15,22,23  prep, one team of six on every chunk (with two
//                  slots only one chunk is ahead of the chain): diagonal 16x16
//                  inverses of (I + A) (fp32), couplings (tf32 mma), blocked
//                  substitution for the 192 columns of [W | U~] (bf16 mma), two
//                  16-column pieces per warp
//   warps 4,5,12,17  E1 (U, Ud from W H) on lane quarters 0,1; warp 4 then
//                  issues MMA3 and MMA2
//   warps 0,1,20,21,6,7,10,11  E2a (state update), two warps (value columns
//                  0..31, 32..63) on every lane quarter, the state in
//                  registers; warp 0 then issues the next MMA1; warps 6,7,10,11
//                  (quarters 2, 3) also store the chunk's output (E2b)
// Every wait is bounded; a timeout records GDN_ERR_TIMEOUT and ends the loops.
//
// GDN block parts that gdn_fwd can fuse into the pass, as in the head_dim_k =
// 64 kernel: beta logits in every instance; the q/k L2 normalisation folded
// into fp32 row factors and column vectors (kFL2) and the output epilogue
// (o + D_h v) * gate (kFEpi) in instances of their own, selected by the mask kF.
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

using namespace ptx;
using namespace tc;

constexpr int DK = 128;
// The input-slot ring, the warps and the warp map.
struct Cfg {
  static constexpr int NIN = 2, kWarps = 24, kTeams = 1, kPrepThreads = 192;
  static constexpr int kWarpSIssue = 13, kWarpProducer = 16;
  // the next MMA1 is issued from an E2a warp that stores no output, so that
  // its wait for the next chunk's prep does not hold back this chunk's output
  static constexpr int kWarpE1Issue = 4, kWarpE2aIssue = 0;
  __device__ __forceinline__ static bool is_prep(int w) {
    return w == 2 || w == 3 || w == 14 || w == 15 || w == 22 || w == 23;
  }
  __device__ __forceinline__ static int prep_index(int w) {
    return (w & 3) - 2 + (w >= 22 ? 4 : (w >= 14 ? 2 : 0));
  }
  __device__ __forceinline__ static bool is_drain(int w) { return w == 8 || w == 9 || w == 18 || w == 19; }
  __device__ __forceinline__ static bool is_e1(int w) { return w == 4 || w == 5 || w == 12 || w == 17; }
  __device__ __forceinline__ static bool is_e2a(int w) {
    return w == 0 || w == 1 || w == 20 || w == 21 || w == 6 || w == 7 || w == 10 || w == 11;
  }
  __device__ __forceinline__ static int e2a_col(int w) { return (w >= 10) ? 32 : 0; }
  // E2a threads; those on lane quarters 2, 3 also store the output and free
  // the slot after it
  static constexpr int kE2aThreads = 256, kOutThreads = 128;
};
constexpr uint32_t kBarPrep = 1;  // the prep team's named barrier
constexpr uint32_t kTmemCols = 512;
// TMEM column map: S double buffer, D1 double buffer, DPU double buffer, DH.
constexpr uint32_t kColS = 0, kColD1 = 128, kColPU = 256, kColH = 384;

constexpr uint32_t kIdescS = umma_idesc_bf16(128, 64);           // K-major x K-major
constexpr uint32_t kIdescKM = umma_idesc_bf16(128, 64, 0, 1);    // K-major A, MN-major B
constexpr uint32_t kIdescMM = umma_idesc_bf16(128, 64, 1, 1);    // MN-major A and B

struct Layout {
  static constexpr int NIN = Cfg::NIN, kTeams = Cfg::kTeams;
  static constexpr int SUB = 8192;
  // input slot: per 64-column group g of q/k, W_g (written by prep) | Q_g |
  // K_g, so that [W_g; Q_g] and [Q_g; K_g] are contiguous M = 128 operands;
  // then V (U~ written over it by prep) and the gates
  static constexpr int NG = DK / 64, GSTRIDE = 3 * SUB;
  static constexpr int SW = 0, SQ = SUB, SK = 2 * SUB, SV = NG * GSTRIDE, SG = SV + SUB;
  // gates: G (log2) [0,64), 2^(G_C - G) [64,128), beta [128,192), E [192,256)
  static constexpr int SLOT = SG + 1024;
  static constexpr int OFF_IN = 0;
  static constexpr int OFF_H = OFF_IN + NIN * SLOT;   // state H [dk][dv] bf16
  static constexpr int OFF_U = OFF_H + NG * SUB;      // U  [token][dv] bf16
  static constexpr int OFF_UD = OFF_U + SUB;          // Ud [token][dv] bf16
  // P ring [3][token][token] bf16, right after the Ud tile: the 8 KB tile
  // before P_i completes the M = 128 operand [*; P_i] of MMA2
  static constexpr int OFF_P = OFF_UD + SUB;
  // A, per S buffer: the 10 16x16 blocks on or below the diagonal, block (r, c)
  // at index r (r + 1) / 2 + c, rows of A_LD floats
  static constexpr int A_LD = 20;
  static constexpr int A_BLK = 16 * A_LD;              // floats per block
  static constexpr int A_BUF = 10 * A_BLK;             // floats per buffer
  static constexpr int OFF_A = OFF_P + 3 * SUB;        // f32 [2][10][16][A_LD]
  // per prep team: T_ii diag(beta gamma) and T_ii diag(beta) (bf16,
  // column-major) and the couplings M_ik (bf16).  T_ii itself (fp32,
  // column-major) overwrites the diagonal block A_ii once it has been read.
  static constexpr int TB_LD = 16;
  static constexpr int TB_TEAM = 2 * 4 * 16 * TB_LD * 2;
  static constexpr int OFF_TB = OFF_A + 2 * A_BUF * 4;
  static constexpr int MB_TEAM = 6 * 16 * TB_LD * 2;
  static constexpr int OFF_MB = OFF_TB + kTeams * TB_TEAM;
  static constexpr int OFF_GC = OFF_MB + kTeams * MB_TEAM;
  static constexpr int OFF_VOTE = OFF_GC + 64;
  static constexpr int OFF_TMEM = OFF_VOTE + 64;
  static constexpr int OFF_BAR = OFF_TMEM + 16;
  static constexpr int NBAR = 32;
  static constexpr int OFF_FLAG = OFF_BAR + NBAR * 8;
  // fused instances only: per input slot, fp32 vectors r_q [0,64), r_k
  // [64,128), the output gate [128,192), G - log2 r_k [192,256) and E r_k
  // [256,320); then the two mbarriers that gather the drain threads' norms
  static constexpr int RN_SLOT = 5 * 64;
  static constexpr int OFF_RN = OFF_FLAG + 16;
  static constexpr int OFF_NBAR = OFF_RN + NIN * RN_SLOT * 4;
  static constexpr int BYTES = OFF_NBAR + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(SLOT % 1024 == 0 && OFF_H % 1024 == 0 && OFF_P % 1024 == 0,
                "alignment");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// mbarrier indices
enum : int {
  B_FULL_IN = 0,     // [4]  TMA bytes landed (+ producer arrival)
  B_EMPTY_IN = 4,    // [4]  slot free: MMA3/MMA2 commit + the output threads' reads (129)
  B_FULL_ST = 8,     // [2]  prep wrote W and U~ (192)
  B_TMEM_FULL = 10,  // [2]  Q K^T / K K^T accumulator ready (commit)
  B_TMEM_EMPTY = 12, // [2]  ... drained (128, the drain warps)
  B_S_READY = 14,    // [2]  P and A in shared memory (128, the drain warps)
  B_H_READY = 16,    //      bf16 state written for the next MMA1 (128)
  B_D1_FULL = 17,    // [2]  MMA1 done (commit)
  B_D1_FREE = 19,    // [2]  D1 drained (E1 128 + output 64)
  B_U_READY = 21,    //      U and Ud written (128)
  B_DH_FULL = 22,    //      MMA3 done (commit)
  B_PU_FULL = 23,    // [2]  MMA2 done (commit)
  B_PU_FREE = 25,    // [2]  DPU drained (64)
  B_A_FREE = 27,     // [2]  A buffer read by the prep (inverse, couplings) (192)
  B_P_FREE = 29,     // [3]  P buffer read by MMA2 (commit)
};

// Two fp32 lanes in one 64-bit register: Blackwell's packed FMA/MUL/ADD run two
// ordinary IEEE fp32 operations per instruction (used in the carry drains).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(uint64_t v) {
  float lo, hi;
  upk2(v, lo, hi);
  return pack_bf16(lo, hi);
}

// One thread drains one row i of a 64-column fp32 accumulator of [Q; K] K^T
// (taddr: this warp's TMEM lane quarter at the buffer's first column) into a
// masked, decayed row of P (bf16, swizzled tile at Ps) or of A (fp32, into the blocks at Ablk):
//   P_ij = S_ij 2^(G_i - G_j) (j <= i),   A_ij = beta_i S_ij 2^(G_i - G_j) (j < i)
// with G in log2 units.  The warp owns rows 32*half .. 32*half+31.  Per
// 16-column block: blocks after those rows are zero (no load, no arithmetic);
// blocks before them use two factors that are both <= 1,
// 2^(G_i - G_b) * E_j with E_j = 2^(G_b - G_j) precomputed per token (b the
// block's last token); the two blocks that meet the rows take one exponent
// per element.  One shared (not inlined) copy keeps the instruction footprint
// small.
// The column factors come from Gc (in place of G_j) and Ec (in place of E_j),
// which carry a column scale when the q/k normalisation is folded in; the row
// factor comes in through bi.
__device__ __noinline__ void drain_s_row(uint32_t taddr, const float *G2, const float *Gc,
                                         const float *Ec, int i, int half, bool isP, float bi,
                                         int ilim, bool rowok, uint32_t Ps, float *Ablk,
                                         uint8_t *smem, uint32_t sbase) {
  const float Gi = G2[i];
  // |beta_i| folded into the exponent (log2 0 = -inf gives 0; a negative beta
  // flips the sign afterwards), rows past the end of the sequence by an empty
  // column range
  const float Gb = Gi + __log2f(fabsf(bi));
  const bool neg = bi < 0.f;
  const int jlim = rowok ? ilim : 0;
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
        const float4 x = *reinterpret_cast<const float4 *>((before ? Ec : Gc) + 16 * cb + 4 * q);
        f[4 * q] = x.x;
        f[4 * q + 1] = x.y;
        f[4 * q + 2] = x.z;
        f[4 * q + 3] = x.w;
      }
      const float scale = before ? bi * ex2(Gi - G2[16 * cb + 15]) : bi;
      tmem_wait_ld();
      if (before) {
        const float sc = rowok ? scale : 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) val[e] = __uint_as_float(v[e]) * (sc * f[e]);
      } else {
        const int lim = jlim - 16 * cb;  // columns e < lim are kept
#pragma unroll
        for (int e = 0; e < 16; ++e)
          val[e] = e < lim ? __uint_as_float(v[e]) * ex2(Gb - f[e]) : 0.f;
        if (neg) {
#pragma unroll
          for (int e = 0; e < 16; ++e) val[e] = -val[e];
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
    } else if (cb <= (i >> 4)) {  // blocks on or below the diagonal only
      const int rb = i >> 4;
      float *dst = Ablk + ((rb * (rb + 1)) / 2 + cb) * Layout::A_BLK + (i & 15) * Layout::A_LD;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4 *>(dst + 4 * q) =
            make_float4(val[4 * q], val[4 * q + 1], val[4 * q + 2], val[4 * q + 3]);
    }
  }
}

// kFSeg: one segment of a split sequence (launched only by the split plan);
// kFRank: packed sequences taken longest first (below)
constexpr int kFL2 = 1, kFEpi = 2, kFSeg = 4, kFRank = 8;

// Packed sequences (cu_seqlens): CTAs start in launch order, so the sequence
// of launch index z is the z-th longest (ties by index) rather than the z-th,
// and the longest chains do not start last.  Each thread t < N ranks sequence
// t against all others; up to kRankedSeqs sequences, else launch order.  Runs
// before any other use of shared memory (its first word holds the result).
constexpr int kRankedSeqs = 128;
__device__ __forceinline__ int longest_first(const FwdParams &p, int z, uint8_t *smem) {
  int *pick = reinterpret_cast<int *>(smem);
  const int t = threadIdx.x;
  if (t == 0) *pick = z;
  __syncthreads();
  if (t < p.num_seqs) {
    const int64_t lt = (int64_t)p.cu[t + 1] - p.cu[t];
    int rank = 0;
    for (int u = 0; u < p.num_seqs; ++u) {
      const int64_t lu = (int64_t)p.cu[u + 1] - p.cu[u];
      rank += (lu > lt || (lu == lt && u < t)) ? 1 : 0;
    }
    if (rank == z) *pick = t;
  }
  __syncthreads();
  const int n = *pick;
  __syncthreads();  // every thread has read the word before shared memory is reused
  return n;
}

template <int kF>
__global__ void __launch_bounds__(Cfg::kWarps * 32, 1)
gdn_fwd_tc128_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v) {
  using L = Layout;
  using C = Cfg;
  constexpr int NIN = C::NIN, NG = L::NG;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t *smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, h = blockIdx.y;
  const int H = p.num_heads, dv = p.dv;

  // The unit: a whole sequence, or one segment of a split sequence (dense
  // inputs).  Segments after the first run from zero ("transport" mode) and
  // have dk/64 extra column tiles that carry the identity through the
  // segment's chunks (its state map's M and its per-token reads r).
  constexpr bool segm = (kF & kFSeg) != 0;
  int n = blockIdx.z, seg = 0;
  bool transport = false;
  int64_t start, len;
  if constexpr (segm) {
    // grid z = segment * num_seqs + sequence, so that every sequence's first
    // segment is dispatched first.  The later segments hold seg_len tokens
    // each and end at the last chunk's end; segment 0 takes the chunks they
    // leave at the front.
    n = blockIdx.z % p.num_seqs;
    seg = blockIdx.z / p.num_seqs;
    transport = seg > 0;
    const int64_t first = (p.seq_len + 63) / 64 * 64 - (int64_t)(p.seg_count - 1) * p.seg_len;
    const int64_t s0 = seg == 0 ? 0 : first + (int64_t)(seg - 1) * p.seg_len;
    const int64_t sl = seg == 0 ? first : p.seg_len;
    start = (int64_t)n * p.seq_len + s0;
    const int64_t rest = p.seq_len - s0;  // > 0 by construction
    len = rest < sl ? rest : sl;
  } else {
    if constexpr ((kF & kFRank) != 0) n = longest_first(p, blockIdx.z, smem);
    if (!sequence_bounds(p, n, h, start, len)) return;  // uniform over the CTA
  }
  const bool mtile = segm && tile * kDvt >= dv;  // a transport column tile
  if (mtile && !transport) return;
  // value columns col0.. of v, o and the states, or transport columns col0..
  const int col0 = mtile ? tile * kDvt - dv : tile * kDvt;
  if ((p.flags & GDN_DEBUG_CHECKS) &&
      !debug_ranges_ok(p, n, h, start, len, mtile ? 0 : col0, kDvt, 2, true))
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
  auto slot_base = [&](int s) { return sbase + L::OFF_IN + s * L::SLOT; };
  auto p_base = [&](int s) { return sbase + L::OFF_P + s * L::SUB; };
  auto gate_ptr = [&](int s) {
    return reinterpret_cast<float *>(smem + L::OFF_IN + s * L::SLOT + L::SG);
  };
  auto valid_rows = [&](int c) {
    return (int)(len - (int64_t)c * 64 < 64 ? len - (int64_t)c * 64 : 64);
  };

  if (tid == 0) {
    for (int s = 0; s < NIN; ++s) {
      mbar_init(bar(B_FULL_IN + s), 1);
      mbar_init(bar(B_EMPTY_IN + s), 1 + C::kOutThreads);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_FULL_ST + s), C::kPrepThreads);
      mbar_init(bar(B_TMEM_FULL + s), 1);
      mbar_init(bar(B_TMEM_EMPTY + s), 128);
      mbar_init(bar(B_S_READY + s), 128);
      mbar_init(bar(B_D1_FULL + s), 1);
      mbar_init(bar(B_D1_FREE + s), 128 + C::kOutThreads);
      mbar_init(bar(B_A_FREE + s), C::kPrepThreads);
      mbar_init(bar(B_PU_FULL + s), 1);
      mbar_init(bar(B_PU_FREE + s), C::kOutThreads);
    }
    mbar_init(bar(B_H_READY), C::kE2aThreads);
    mbar_init(bar(B_U_READY), 128);
    for (int s = 0; s < 3; ++s) mbar_init(bar(B_P_FREE + s), 1);
    mbar_init(bar(B_DH_FULL), 1);
    if constexpr ((kF & kFL2) != 0) {
      mbar_init(sbase + L::OFF_NBAR, 128);
      mbar_init(sbase + L::OFF_NBAR + 8, 128);
    }
    *S.abort_flag = 0;
    fence_mbar_init();
  }
  if (mtile) {  // V = 0 on the transport columns (no load ever writes these tiles)
    for (int idx = tid; idx < NIN * (L::SUB / 16); idx += C::kWarps * 32) {
      const int sl = idx / (L::SUB / 16), q = idx % (L::SUB / 16);
      reinterpret_cast<uint4 *>(smem + L::OFF_IN + sl * L::SLOT + L::SV)[q] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (warp == C::kWarpSIssue) tmem_alloc(sbase + L::OFF_TMEM, kTmemCols);
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

  if (warp == C::kWarpProducer) {
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
    const uint32_t kTx = (2 * NG + (mtile ? 0 : 1)) * L::SUB;
    int issued = 0;
    for (int c = 0; c < nc; ++c) {
      const int slot = c % NIN;
      // Gate vectors of chunk c, computed before the slot is free: G (log2
      // units), the decay to the chunk end 2^(G_C - G), beta, and
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
      const float2 vD = make_float2(ex2(Gl - G0), ex2(Gl - G1));
      const float2 vE = make_float2(ex2(Gb - G0), ex2(Gb - G1));
      const float2 vB = make_float2(bv0, bv1);
      const float gC = ex2(Gl);
      const float2 vO = make_float2(og0, og1);
      load_gates(c + 1);
      GDN_PHASE(0);
      bool ok = true;
      if (c >= NIN) ok = role_wait(bar(B_EMPTY_IN + slot), ((c / NIN) - 1) & 1, S, p, n, h, 1);
      GDN_PHASE(1);
      if (!__all_sync(0xffffffffu, ok)) break;
      {
        float *gate = gate_ptr(slot);
        *reinterpret_cast<float2 *>(gate + 2 * lane) = make_float2(G0, G1);
        *reinterpret_cast<float2 *>(gate + 64 + 2 * lane) = vD;
        *reinterpret_cast<float2 *>(gate + 128 + 2 * lane) = vB;
        *reinterpret_cast<float2 *>(gate + 192 + 2 * lane) = vE;
        if (lane == 0) sgc[c & 3] = gC;  // a ring of 4: E2a may read it after the slot is freed
        if constexpr ((kF & kFEpi) != 0)
          *reinterpret_cast<float2 *>(reinterpret_cast<float *>(smem + L::OFF_RN) +
                                      slot * L::RN_SLOT + 128 + 2 * lane) = vO;
      }
      __syncwarp();
      if (lane == 0) {
        const uint32_t sb = slot_base(slot);
        const int row = (int)(start + (int64_t)c * 64);
        mbar_arrive_expect_tx(bar(B_FULL_IN + slot), kTx);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          tma_load_3d(sb + g * L::GSTRIDE + L::SQ, &tmap_q, 64 * g, h, row, bar(B_FULL_IN + slot));
          tma_load_3d(sb + g * L::GSTRIDE + L::SK, &tmap_k, 64 * g, h, row, bar(B_FULL_IN + slot));
        }
        if (!mtile) tma_load_3d(sb + L::SV, &tmap_v, col0, h, row, bar(B_FULL_IN + slot));
        if (c + NIN < nc) {  // warm L2 with the tiles of the chunk that reuses this slot
          const int prow = row + NIN * 64;
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            tma_prefetch_3d(&tmap_q, 64 * g, h, prow);
            tma_prefetch_3d(&tmap_k, 64 * g, h, prow);
          }
          if (!mtile) tma_prefetch_3d(&tmap_v, col0, h, prow);
        }
      }
      GDN_PHASE(2);
      ++issued;
    }
    if (lane == 0)
      for (int c = issued - NIN < 0 ? 0 : issued - NIN; c < issued; ++c)
        mbar_wait_bounded(bar(B_FULL_IN + c % NIN), (c / NIN) & 1, kWaitTimeoutNs);
  } else if (C::is_drain(warp)) {
    // ------------------------------------------------------------ S drains
    // The [Q; K] K^T accumulator of each chunk: lane quarters 0,1 hold the P
    // rows (warps 8,9), quarters 2,3 the A rows (warps 18,19).
    const int wq = warp & 3;
    const bool isP = wq < 2;
    const int i = 32 * (wq & 1) + lane;
    const uint32_t tq = tmem_base + ((uint32_t)(32 * wq) << 16);
    for (int c = 0; c < nc; ++c) {
      const int slot = c % NIN, buf = c & 1;
      GDN_PHASE(8);
      constexpr bool l2 = (kF & kFL2) != 0;
      const float *gate = gate_ptr(slot);
      const float *G2 = gate, *beta = gate + 128, *E = gate + 192;
      float *rn = reinterpret_cast<float *>(smem + L::OFF_RN) + slot * L::RN_SLOT;
      bool ok = true;
      float r = 1.f;
      if constexpr (l2) {
        // This thread's row norm, q_i (P rows) or k_i (A rows), from the input
        // tile as soon as it lands; it is published before the accumulator and
        // buffer waits, so the P drains (which need every r_k as a column
        // factor) do not wait on the A drains' buffer.
        ok = role_wait(bar(B_FULL_IN + slot), (c / NIN) & 1, S, p, n, h, 8);
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint32_t tb = slot_base(slot) + (isP ? L::SQ : L::SK);
        // eight independent partial sums, so that the norm is a short
        // dependent chain on the slot's path
        float ss[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q8 = 0; q8 < DK / 8; ++q8) {
          const uint4 x = S4(swz<L::GSTRIDE>(tb, i, 8 * q8));
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          float a = ss[q8 & 7];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
            a = fmaf(lo, lo, fmaf(hi, hi, a));
          }
          ss[q8 & 7] = a;
        }
        r = rsqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) + ((ss[4] + ss[5]) + (ss[6] + ss[7])) + 1e-6f);
        if (isP) {
          rn[i] = r;
        } else {
          rn[64 + i] = r;
          rn[192 + i] = G2[i] - __log2f(r);  // column j: 2^(G_i - G_j) r_k_j
          rn[256 + i] = E[i] * r;
        }
        mbar_arrive(sbase + L::OFF_NBAR + 8 * (c & 1));
        ok = role_wait(bar(B_TMEM_FULL + buf), (c >> 1) & 1, S, p, n, h, 7);
      } else {
        ok = role_wait(bar(B_TMEM_FULL + buf), (c >> 1) & 1, S, p, n, h, 7);
        if (ok) ok = role_wait(bar(B_FULL_IN + slot), (c / NIN) & 1, S, p, n, h, 8);
      }
      // the P buffer was last read by MMA2 of chunk c-3; the A buffer by the
      // inverse and couplings of chunk c-2
      if (ok && isP && c >= 3)
        ok = role_wait(bar(B_P_FREE + c % 3), ((c / 3) - 1) & 1, S, p, n, h, 10);
      if (ok && !isP && c >= 2)
        ok = role_wait(bar(B_A_FREE + buf), ((c - 2) >> 1) & 1, S, p, n, h, 21);
      if constexpr (l2)
        if (ok) ok = role_wait(sbase + L::OFF_NBAR + 8 * (c & 1), (c >> 1) & 1, S, p, n, h, 30);
      GDN_PHASE(9);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int valid = valid_rows(c);
      const int ilim = isP ? i + 1 : i;  // P keeps j <= i, A keeps j < i
      // row factor: 1, or r_q (P) / beta_i r_k (A) under the normalisation
      const float bi = (isP ? 1.f : beta[i]) * r;
      float *Ablk = reinterpret_cast<float *>(smem + L::OFF_A) + buf * L::A_BUF;
      drain_s_row(tq + kColS + buf * 64, G2, l2 ? rn + 192 : G2, l2 ? rn + 256 : E, i, wq & 1,
                  isP, bi, ilim, i < valid, p_base(c % 3), Ablk, smem, sbase);
      tc_fence_before();
      mbar_arrive(bar(B_TMEM_EMPTY + buf));
      if (isP) fence_proxy_async_smem();  // P is read by MMA2 (async proxy)
      GDN_PHASE(10);
      mbar_arrive(bar(B_S_READY + buf));
    }
  } else if (warp == C::kWarpSIssue) {
    // ------------------------------------------------------------ [Q; K] K^T issuer
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nc; ++c) {
        bool ok = role_wait(bar(B_FULL_IN + c % NIN), (c / NIN) & 1, S, p, n, h, 5);
        if (ok && c >= 2)
          ok = role_wait(bar(B_TMEM_EMPTY + (c & 1)), ((c >> 1) - 1) & 1, S, p, n, h, 6);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a = slot_base(c % NIN) + L::SQ;  // [Q_g; K_g] per column group g
#pragma unroll
        for (int kk = 0; kk < 4 * NG; ++kk) {
          const uint32_t ak = a + (kk >> 2) * L::GSTRIDE + (kk & 3) * 32;
          umma_bf16(tmem_base + kColS + (c & 1) * 64, umma_desc_sw128(ak),
                    umma_desc_sw128(ak + L::SUB), kIdescS, kk > 0);
        }
        umma_commit(bar(B_TMEM_FULL + (c & 1)));
        GDN_PROBE_AT(warp, c, 0, clock64());
        ++issued;
      }
      // the last product has completed before tensor memory is released
      if (issued > 0)
        mbar_wait_bounded(bar(B_TMEM_FULL + ((issued - 1) & 1)), ((issued - 1) >> 1) & 1,
                          kWaitTimeoutNs);
    }
    __syncwarp();
  } else if (C::is_prep(warp)) {
    // ------------------------------------------------------------ prep
    // One team of six warps takes every chunk; pw is the warp within the team.
    const int pw = C::prep_index(warp), ptid = 32 * pw + lane;
    const uint32_t kBar = kBarPrep;
    __nv_bfloat16 *sTB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_TB);
    __nv_bfloat16 *sMB = reinterpret_cast<__nv_bfloat16 *>(smem + L::OFF_MB);
    const uint32_t TBa = smem_u32(sTB), MBa = smem_u32(sMB);
    int *vote = votes;

    for (int c = 0; c < nc; ++c) {
      const int slot = c % NIN, stage = c & 1, vset = c & 1;
      const int valid = valid_rows(c);
      GDN_PHASE(0);
      // P and A of this chunk are in shared memory; the carry is done with the
      // stage's previous contents (the P drain waited for MMA2 of chunk c-2)
      bool ok = role_wait(bar(B_S_READY + stage), (c >> 1) & 1, S, p, n, h, 2);
      if (ok) ok = role_wait(bar(B_FULL_IN + slot), (c / NIN) & 1, S, p, n, h, 3);
      ok = __all_sync(0xffffffffu, ok) && !*S.abort_flag;
      GDN_PHASE(1);

      const uint32_t sb = slot_base(slot);
      const uint32_t Vs = sb + L::SV;
      const float *gate = gate_ptr(slot);
      const float *G2 = gate, *beta = gate + 128;
      float *sA = reinterpret_cast<float *>(smem + L::OFF_A) + stage * L::A_BUF;
      const uint32_t Us = Vs;  // U~ replaces V, block row by block row

      // rows past the end of the sequence: zero Q, K, V (the Q K^T MMA has read them)
      if (ok && valid < 64) {
        constexpr int kPerRow = (2 * NG + 1) * 8;  // 16-byte granules of Q_g, K_g, V
        for (int idx = ptid; idx < (64 - valid) * kPerRow; idx += C::kPrepThreads) {
          const int row = valid + idx / kPerRow, q = idx % kPerRow, t8 = q >> 3;
          const uint32_t tb = t8 == 2 * NG ? Vs : sb + (t8 >> 1) * L::GSTRIDE + ((t8 & 1) ? L::SK : L::SQ);
          S4(tile_addr(tb, row, (q & 7) * 8)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (lane == 0) vote[vset * 8 + pw] = ok ? 1 : 0;
      named_sync(kBar, C::kPrepThreads);
      GDN_PHASE(2);
      {
        const int *v = vote + vset * 8;
        if (!(v[0] && v[1] && v[2] && v[3] && v[4] && v[5])) break;
      }

      // ---- 16x16 diagonal blocks of T = (I + A)^-1 (fp32).  Team warps 4,5 take
      // two blocks each, one per half-warp; lane l builds column l of its block by
      // forward substitution, T_rl = [r == l] - sum_{k<r} A_rk T_kl, reading
      // rows of A as float4 (broadcast within the half-warp).  T is stored
      // column-major: fp32 for the couplings, and as bf16 T diag(beta gamma) and
      // T diag(beta) for the substitution. ----
      if (pw >= 4) {
        const int blk = 2 * (pw - 4) + (lane >> 4), l = lane & 15;
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
        __syncwarp();  // every lane of the half-warp is done reading A_bb
        float *tcol = sA + ((blk * (blk + 1)) / 2 + blk) * L::A_BLK + l * L::A_LD;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4 *>(tcol + 4 * q) =
              make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        const float bj = beta[16 * blk + l];
        float bgj = bj * ex2(G2[16 * blk + l]);  // beta_j gamma_j
        if constexpr ((kF & kFL2) != 0)  // times r_k_j: W = T diag(beta gamma r_k) K
          bgj *= reinterpret_cast<const float *>(smem + L::OFF_RN)[slot * L::RN_SLOT + 64 + 16 * blk + l];
        uint32_t wg[8], wb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          wg[e] = pack_bf16(x[2 * e] * bgj, x[2 * e + 1] * bgj);
          wb[e] = pack_bf16(x[2 * e] * bj, x[2 * e + 1] * bj);
        }
        uint4 *tg = reinterpret_cast<uint4 *>(sTB + ((0 * 4 + blk) * 16 + l) * L::TB_LD);
        uint4 *tb = reinterpret_cast<uint4 *>(sTB + ((1 * 4 + blk) * 16 + l) * L::TB_LD);
        tg[0] = make_uint4(wg[0], wg[1], wg[2], wg[3]);
        tg[1] = make_uint4(wg[4], wg[5], wg[6], wg[7]);
        tb[0] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        tb[1] = make_uint4(wb[4], wb[5], wb[6], wb[7]);
      }
      GDN_PHASE(3);
      named_sync(kBar, C::kPrepThreads);
      GDN_PHASE(4);

      // ---- M_ik = T_ii A_ik (i > k) on tf32 tensor cores, stored negated (bf16) ----
#pragma unroll 1
      for (int blk = pw; blk < 6; blk += 6) {
        const int i = blk == 0 ? 1 : (blk < 3 ? 2 : 3);
        const int k = blk - (i * (i - 1)) / 2;
        // T_ii, column-major in the diagonal block of A: T(row, col) = T[col * A_LD + row]
        const float *T = sA + ((i * (i + 1)) / 2 + i) * L::A_BLK;
        const float *Ak = sA + ((i * (i + 1)) / 2 + k) * L::A_BLK;
        float acc[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint32_t a0 = to_tf32(T[(8 * ks + t) * L::A_LD + g]);
          const uint32_t a1 = to_tf32(T[(8 * ks + t) * L::A_LD + g + 8]);
          const uint32_t a2 = to_tf32(T[(8 * ks + t + 4) * L::A_LD + g]);
          const uint32_t a3 = to_tf32(T[(8 * ks + t + 4) * L::A_LD + g + 8]);
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
      named_sync(kBar, C::kPrepThreads);
      mbar_arrive(bar(B_A_FREE + stage));  // A of this buffer is no longer read
      GDN_PHASE(6);

      // ---- block forward substitution, left-looking (a compact loop):
      // X_i = T_ii B_i + sum_{k<i} (-M_ik) X_k for X = [W | U~], B = [K | V] (the
      // beta, gamma scalings are folded into the T_ii tiles).  The 192 columns of
      // [W | U~] go to the six warps as two 16-column pieces each.  A warp
      // reads back only its own columns of the earlier block rows, so the levels
      // need no CTA-wide barrier. ----
      {
        constexpr int NP = (DK + 64) / 16 / 6;  // 16-column pieces per warp
        const int arow = lrow + (lmi & 1) * 8, acol = (lmi >> 1) * 8;
        const int trow = lrow + (lmi >> 1) * 8, tcol = (lmi & 1) * 8;  // column-major T tiles
        uint32_t xt[NP], bsrc[NP];
        int pcol[NP];
        bool pwW[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          const int gc = 16 * (NP * pw + j);  // column of [W | U~]
          pwW[j] = gc < DK;
          const uint32_t grp = sb + (gc >> 6) * L::GSTRIDE;
          xt[j] = pwW[j] ? grp + L::SW : Us;
          bsrc[j] = pwW[j] ? grp + L::SK : Vs;
          pcol[j] = pwW[j] ? (gc & 63) : gc - DK;
        }
#pragma unroll 1
        for (int lv = 0; lv < 4; ++lv) {
          float acc[NP][2][4];
          {
            uint32_t tw[4], tu[4], tb[NP][4];
            ldsm_x4_t(TBa + (((0 * 4 + lv) * 16 + trow) * L::TB_LD + tcol) * 2, tw[0], tw[1],
                      tw[2], tw[3]);
            ldsm_x4_t(TBa + (((1 * 4 + lv) * 16 + trow) * L::TB_LD + tcol) * 2, tu[0], tu[1],
                      tu[2], tu[3]);
#pragma unroll
            for (int j = 0; j < NP; ++j)
              ldsm_x4_t(tile_addr(bsrc[j], 16 * lv + arow, pcol[j] + acol), tb[j][0], tb[j][1],
                        tb[j][2], tb[j][3]);
#pragma unroll
            for (int j = 0; j < NP; ++j) {
              // T_ii diag(beta gamma) for W pieces, T_ii diag(beta) for U~ pieces
              const uint32_t a0 = pwW[j] ? tw[0] : tu[0], a1 = pwW[j] ? tw[1] : tu[1];
              const uint32_t a2 = pwW[j] ? tw[2] : tu[2], a3 = pwW[j] ? tw[3] : tu[3];
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][nt][e] = 0.f;
                mma_bf16(acc[j][nt], a0, a1, a2, a3, tb[j][2 * nt], tb[j][2 * nt + 1]);
              }
            }
          }
#pragma unroll 1
          for (int k = 0; k < lv; ++k) {
            const int blk = (lv * (lv - 1)) / 2 + k;
            uint32_t ma[4], xb[NP][4];
            ldsm_x4(MBa + ((blk * 16 + arow) * L::TB_LD + acol) * 2, ma[0], ma[1], ma[2], ma[3]);
#pragma unroll
            for (int j = 0; j < NP; ++j)
              ldsm_x4_t(tile_addr(xt[j], 16 * k + arow, pcol[j] + acol), xb[j][0], xb[j][1],
                        xb[j][2], xb[j][3]);
#pragma unroll
            for (int j = 0; j < NP; ++j)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
                mma_bf16(acc[j][nt], ma[0], ma[1], ma[2], ma[3], xb[j][2 * nt], xb[j][2 * nt + 1]);
          }
#pragma unroll
          for (int j = 0; j < NP; ++j)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                S1(tile_addr(xt[j], 16 * lv + g + 8 * hf, pcol[j] + 8 * nt + 2 * t)) =
                    pack_bf16(acc[j][nt][2 * hf], acc[j][nt][2 * hf + 1]);
          __syncwarp();
        }
      }
      // W, U~ and the zeroed rows are read by the tensor cores (async proxy)
      fence_proxy_async_smem();
      GDN_PHASE(7);
      mbar_arrive(bar(B_FULL_ST + stage));
    }
  } else {
    // ------------------------------------------------------------ carry chain / output
    const int wq = warp & 3;                // TMEM lane quarter
    const int row = 32 * (wq & 1) + lane;   // token (E1, output)
    auto tm = [&](uint32_t col) { return tmem_base + ((uint32_t)(32 * wq) << 16) + col; };
    const uint32_t Hs = sbase + L::OFF_H, Ust = sbase + L::OFF_U, Uds = sbase + L::OFF_UD;
    // MMA1 of chunk c: [W; Q] H (rows 0..63 = W H, rows 64..127 = Q H), the
    // key dimension in 64-column groups [W_g; Q_g]
    auto issue_mma1 = [&](int c) {
      const uint32_t a = slot_base(c % NIN) + L::SW;
#pragma unroll
      for (int kk = 0; kk < 4 * NG; ++kk)
        umma_bf16(tmem_base + kColD1 + (c & 1) * 64,
                  umma_desc_sw128(a + (kk >> 2) * L::GSTRIDE + (kk & 3) * 32),
                  umma_desc_sw128_mn(Hs + kk * 2048, L::SUB), kIdescKM, kk > 0);
      umma_commit(bar(B_D1_FULL + (c & 1)));
    };
    // the operands and the accumulator of MMA1(c) are ready (one thread);
    // `pre`: D1_FREE and FULL_ST were already seen complete
    auto mma1_ready = [&](int c, bool pre) {
      bool ok = true;
      if (!pre && c >= 2)
        ok = role_wait(bar(B_D1_FREE + (c & 1)), ((c >> 1) - 1) & 1, S, p, n, h, 18);
      GDN_PROBE_AT(warp, c, 12, clock64());
      if (ok && !pre) ok = role_wait(bar(B_FULL_ST + (c & 1)), (c >> 1) & 1, S, p, n, h, 16);
      GDN_PROBE_AT(warp, c, 8, clock64());
      if (ok) ok = role_wait(bar(B_H_READY), c & 1, S, p, n, h, 17);
      GDN_PROBE_AT(warp, c, 9, clock64());
      return ok;
    };
    auto mma1_pre = [&](int c) {
      return (c < 2 || mbar_test(bar(B_D1_FREE + (c & 1)), ((c >> 1) - 1) & 1)) &&
             mbar_test(bar(B_FULL_ST + (c & 1)), (c >> 1) & 1);
    };
    // E2b for chunk c: the output rows of this warp's lane quarter (2 or 3),
    // value columns ocb .. ocb + 16 nq - 1; then frees D1, DPU and the input
    // slot.  Returns false if a wait gave up.
    constexpr bool epi = (kF & kFEpi) != 0;  // the block epilogue (o + D_h v) * gate
    float dh = 0.f;
    if constexpr (epi)
      if (p.d_skip) dh = p.d_skip[h];
    // gi: gamma_i (times r_q_i under the normalisation) and og: the output gate,
    // both read from the slot before it was released
    auto output_chunk = [&](int c, int ocb, int nq, float gi, float og) -> bool {
        const int buf = c & 1;
        const int valid = valid_rows(c);
        // ---- E2b: O = diag(gamma) (Q H) + P U (row = token); each thread
        // stores its row of O, value columns ocb .. ocb + 16 nq - 1 ----
        const size_t orow_idx = (size_t)(start + (int64_t)c * 64 + row) * H + h;
        const bool st = row < valid;
        const __nv_bfloat16 *vrow = static_cast<const __nv_bfloat16 *>(p.v) + orow_idx * dv + col0;
        if (epi && st) {  // v is reloaded (its tile now holds U~)
          prefetch_l1(vrow + ocb);
          prefetch_l1(vrow + ocb + 16 * nq - 1);
        }
        GDN_PHASE(0);
        bool ok = role_wait(bar(B_PU_FULL + buf), (c >> 1) & 1, S, p, n, h, 13);
        if (!__all_sync(0xffffffffu, ok)) return false;
        GDN_PHASE(1);
        tc_fence_after();
        {
          // o (a later segment's o0), or r on the transport columns
          __nv_bfloat16 *orow =
              mtile ? static_cast<__nv_bfloat16 *>(p.seg_r) + orow_idx * DK + col0
                    : static_cast<__nv_bfloat16 *>(p.o) + orow_idx * dv + col0;
          const uint64_t gi2 = pk2(gi, gi);
#pragma unroll 1
          for (int q2 = ocb / 16; q2 < ocb / 16 + nq; ++q2) {
            uint32_t a[16], b[16];
            tmem_ld16(tm(kColD1 + buf * 64 + 16 * q2), a);
            tmem_ld16(tm(kColPU + buf * 64 + 16 * q2), b);
            tmem_wait_ld();
            uint32_t w8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w8[e] = pack_bf16x2(fma2(gi2, pk2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1])),
                                       pk2(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]))));
            if constexpr (epi) {
              if (st) {
                const uint4 v0 = reinterpret_cast<const uint4 *>(vrow + 16 * q2)[0];
                const uint4 v1 = reinterpret_cast<const uint4 *>(vrow + 16 * q2)[1];
                const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float o0 = fmaf(gi, __uint_as_float(a[2 * e]), __uint_as_float(b[2 * e]));
                  const float o1 =
                      fmaf(gi, __uint_as_float(a[2 * e + 1]), __uint_as_float(b[2 * e + 1]));
                  w8[e] = pack_bf16(block_epilogue(o0, bf16_lo(vw[e]), dh, og),
                                    block_epilogue(o1, bf16_hi(vw[e]), dh, og));
                }
              }
            }
            if (st) {
              reinterpret_cast<uint4 *>(orow + 16 * q2)[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
              reinterpret_cast<uint4 *>(orow + 16 * q2)[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
            }
          }
          tc_fence_before();
          mbar_arrive(bar(B_D1_FREE + buf));
          mbar_arrive(bar(B_PU_FREE + buf));
        }
        return true;
    };
    if (C::is_e1(warp)) {
      // ---- E1 (warps 4,5,12,17): U = U~ - W H (row = token), Ud = U * exp(G_C - G),
      // 32 value columns per warp; warp 4 lane 0 then issues MMA3 and MMA2
      const int cb = warp >= 12 ? 32 : 0;
      int done = 0;
      for (int c = 0; c < nc; ++c) {
        const int slot = c % NIN, buf = c & 1;
        const float *gate = gate_ptr(slot);
        GDN_PHASE(0);
        bool ok = role_wait(bar(B_D1_FULL + buf), (c >> 1) & 1, S, p, n, h, 11);
        // U is overwritten below: MMA2 of chunk c-1 (issued from another
        // thread than MMA1) has finished reading it
        if (ok && c >= 1) ok = role_wait(bar(B_PU_FULL + (buf ^ 1)), ((c - 1) >> 1) & 1, S, p, n, h, 23);
        if (!__all_sync(0xffffffffu, ok)) break;
        GDN_PHASE(1);
        tc_fence_after();
        // the issuing thread looks at the (usually long complete) barrier of
        // MMA2's accumulator now, so that the check overlaps this epilogue
        bool pu_free = true;
        if (warp == C::kWarpE1Issue && lane == 0 && c >= 2)
          pu_free = mbar_test(bar(B_PU_FREE + buf), ((c >> 1) - 1) & 1);
        const uint32_t Ut = slot_base(slot) + L::SV;  // U~ (written over V by prep)
        float dj = gate[64 + row];
        if constexpr ((kF & kFL2) != 0)  // Ud = diag(d r_k) U
          dj *= reinterpret_cast<const float *>(smem + L::OFF_RN)[slot * L::RN_SLOT + 64 + row];
        const uint64_t dj2 = pk2(dj, dj);
        {
          uint32_t w[32];
          tmem_ld32(tm(kColD1 + buf * 64 + cb), w);
          uint4 xu[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) xu[q] = S4(tile_addr(Ut, row, cb + 8 * q));
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t x[4] = {xu[q].x, xu[q].y, xu[q].z, xu[q].w};
            uint32_t pu[4], pd[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint64_t u = sub2(pk2(bf16_lo(x[e]), bf16_hi(x[e])),
                                      pk2(__uint_as_float(w[8 * q + 2 * e]),
                                          __uint_as_float(w[8 * q + 2 * e + 1])));
              pu[e] = pack_bf16x2(u);
              pd[e] = pack_bf16x2(mul2(u, dj2));
            }
            S4(tile_addr(Ust, row, cb + 8 * q)) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
            S4(tile_addr(Uds, row, cb + 8 * q)) = make_uint4(pd[0], pd[1], pd[2], pd[3]);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_D1_FREE + buf));
        fence_proxy_async_smem();
        mbar_arrive(bar(B_U_READY));
        GDN_PHASE(2);
        if (warp == C::kWarpE1Issue) {
          if (lane == 0) {
            GDN_PROBE_AT(warp, c, 6, clock64());
            ok = role_wait(bar(B_U_READY), c & 1, S, p, n, h, 19);
            GDN_PROBE_AT(warp, c, 7, clock64());
            if (ok && !pu_free)
              ok = role_wait(bar(B_PU_FREE + buf), ((c >> 1) - 1) & 1, S, p, n, h, 20);
            GDN_PROBE_AT(warp, c, 8, clock64());
            if (ok) {
              tc_fence_after();
              // MMA3: the state increment [K_0^T; K_1^T] Ud = K^T Ud, an M = 128
              // product of the MN-major views of the two K tiles, in all 128 lanes
              const uint32_t kt = slot_base(slot) + L::SK;
              constexpr uint32_t kMnAtom = L::GSTRIDE;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem_base + kColH, umma_desc_sw128_mn(kt + kk * 2048, kMnAtom),
                          umma_desc_sw128_mn(Uds + kk * 2048, L::SUB), kIdescMM, kk > 0);
              GDN_PROBE_AT(warp, c, 9, clock64());
              umma_commit(bar(B_DH_FULL));
              // MMA3 was the last reader of the slot's tiles (W, Q by MMA1 and
              // U~ by E1 are done before it is issued; MMA2 reads P and U); the
              // output threads' arrivals cover the gate values.  No commit for
              // the last NIN chunks: no slot reload waits on it.
              if (c + NIN < nc) umma_commit(bar(B_EMPTY_IN + slot));
              GDN_PROBE_AT(warp, c, 10, clock64());
              // MMA2: [*; P] U  (rows 64..127 = P U)
              const uint32_t ap = p_base(c % 3) - L::SUB;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem_base + kColPU + buf * 64, umma_desc_sw128(ap + kk * 32),
                          umma_desc_sw128_mn(Ust + kk * 2048, L::SUB), kIdescKM, kk > 0);
              GDN_PROBE_AT(warp, c, 11, clock64());
              umma_commit(bar(B_PU_FULL + buf));
              umma_commit(bar(B_P_FREE + c % 3));
              GDN_PROBE_AT(warp, c, 5, clock64());
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          done = c + 1;
        }
      }
      // the last products have completed before tensor memory is released
      if (warp == C::kWarpE1Issue && lane == 0 && done > 0)
        mbar_wait_bounded(bar(B_PU_FULL + ((done - 1) & 1)), ((done - 1) >> 1) & 1, kWaitTimeoutNs);
    } else if (C::is_e2a(warp)) {
      // ---- E2a: H <- gamma_C H + K^T Ud (krow = key index); this thread's
      // part of the state, H[krow][cb .. cb+31], stays in registers.  Lane 0
      // of warp kWarpE2aIssue then issues MMA1 of the next chunk.  Two warps
      // on every lane quarter; those on quarters 2, 3 then store the chunk's
      // output (E2b) for their 32 value columns.
      const int cb = C::e2a_col(warp);
      const int krow = 32 * wq + lane;
      const bool also_out = wq >= 2;
      const size_t state_row =
          ((size_t)n * H + h) * (size_t)DK * dv + (size_t)krow * dv + col0 + cb;
      // a split sequence's per-segment arrays: [N][seg_count][H][dk][dv or dk]
      const size_t unit = ((size_t)n * p.seg_count + seg) * H + h;
      const size_t seg_row = unit * DK * dv + (size_t)krow * dv + col0 + cb;
      float hrow[32];
      auto store_seg = [&](uint32_t tilebase, const float *x) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          S4(tile_addr(tilebase, krow, cb + 8 * q)) =
              make_uint4(pack_bf16(x[8 * q], x[8 * q + 1]), pack_bf16(x[8 * q + 2], x[8 * q + 3]),
                         pack_bf16(x[8 * q + 4], x[8 * q + 5]), pack_bf16(x[8 * q + 6], x[8 * q + 7]));
      };
      // the initial state: the caller's (whole sequence, first segment), zero
      // (a later segment's value columns) or the identity (its transport
      // columns)
      const float *s_in = transport ? nullptr : p.s0 ? p.s0 + state_row : nullptr;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s_in) v4 = *reinterpret_cast<const float4 *>(s_in + 4 * q);
        hrow[4 * q] = v4.x;
        hrow[4 * q + 1] = v4.y;
        hrow[4 * q + 2] = v4.z;
        hrow[4 * q + 3] = v4.w;
      }
      if (mtile) {
#pragma unroll
        for (int j = 0; j < 32; ++j) hrow[j] = (krow == col0 + cb + j) ? 1.f : 0.f;
      }
      store_seg(Hs, hrow);
      fence_proxy_async_smem();
      mbar_arrive(bar(B_H_READY));
      int issued = 0;  // MMA1 products issued (by lane 0 of warp kWarpE2aIssue)
      bool alive = true;
      if (warp == C::kWarpE2aIssue) {
        if (lane == 0) {
          alive = mma1_ready(0, false);
          if (alive) {
            tc_fence_after();
            issue_mma1(0);
          }
        }
        alive = __shfl_sync(0xffffffffu, alive, 0);
        issued = alive ? 1 : 0;
      }
      for (int c = 0; c < nc && alive; ++c) {
        const int slot = c % NIN;
        // The output threads read their per-token values of chunk c from the
        // slot first and release it: gamma_i (times r_q_i under the
        // normalisation) and the output gate.
        float gi = 1.f, og = 1.f;
        if (also_out) {
          bool okin = role_wait(bar(B_FULL_IN + slot), (c / NIN) & 1, S, p, n, h, 24);
          // r_q comes from the P drains: wait for the chunk's norms
          if constexpr ((kF & kFL2) != 0)
            if (okin) okin = role_wait(sbase + L::OFF_NBAR + 8 * (c & 1), (c >> 1) & 1, S, p, n, h, 25);
          if (!__all_sync(0xffffffffu, okin)) break;
          gi = ex2(gate_ptr(slot)[row]);
          const float *rn = reinterpret_cast<const float *>(smem + L::OFF_RN) + slot * L::RN_SLOT;
          if constexpr ((kF & kFL2) != 0) gi *= rn[row];
          if constexpr (epi) og = rn[128 + row];
          if (c + NIN < nc) mbar_arrive(bar(B_EMPTY_IN + slot));
        }
        GDN_PHASE(3);
        bool ok = role_wait(bar(B_DH_FULL), c & 1, S, p, n, h, 12);
        if (!__all_sync(0xffffffffu, ok)) break;
        GDN_PHASE(4);
        tc_fence_after();
        bool pre = false;
        if (warp == C::kWarpE2aIssue && lane == 0 && c + 1 < nc) pre = mma1_pre(c + 1);
        {
          const float gC = sgc[c & 3];
          uint32_t w[32];
          tmem_ld32(tm(kColH + cb), w);
          tmem_wait_ld();
          const uint64_t gC2 = pk2(gC, gC);
#pragma unroll
          for (int j = 0; j < 32; j += 2)
            upk2(fma2(gC2, pk2(hrow[j], hrow[j + 1]), pk2(__uint_as_float(w[j]), __uint_as_float(w[j + 1]))),
                 hrow[j], hrow[j + 1]);
        }
        tc_fence_before();
        store_seg(Hs, hrow);
        fence_proxy_async_smem();
        mbar_arrive(bar(B_H_READY));
        GDN_PHASE(5);
        if (warp == C::kWarpE2aIssue && c + 1 < nc) {
          if (lane == 0) {
            ok = mma1_ready(c + 1, pre);
            if (ok) {
              tc_fence_after();
              issue_mma1(c + 1);
              GDN_PROBE_AT(warp, c + 1, 6, clock64());
            }
          }
          alive = __shfl_sync(0xffffffffu, ok, 0);
          if (alive) issued = c + 2;
        }
        if (also_out && alive && !output_chunk(c, cb, 2, gi, og)) alive = false;
      }
      // the last MMA1 has completed before tensor memory is released
      if (warp == C::kWarpE2aIssue && lane == 0 && issued > 0)
        mbar_wait_bounded(bar(B_D1_FULL + ((issued - 1) & 1)), ((issued - 1) >> 1) & 1,
                          kWaitTimeoutNs);
      // the final state: the caller's (whole sequence), the state entering
      // segment 1 (segment 0), or a later segment's X / M
      float *s_out = nullptr;
      if (mtile) s_out = p.seg_m + unit * DK * DK + (size_t)krow * DK + col0 + cb;
      else if (transport) s_out = p.seg_x + seg_row;
      else if (segm) s_out = p.seg_state + seg_row + (size_t)H * DK * dv;  // segment 1
      else s_out = p.sN ? p.sN + state_row : nullptr;
      if (s_out && !*S.abort_flag) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4 *>(s_out + 4 * q) =
              make_float4(hrow[4 * q], hrow[4 * q + 1], hrow[4 * q + 2], hrow[4 * q + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpSIssue) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

cudaError_t launch_tc128(const FwdParams &p, cudaStream_t stream) {
  using L = Layout;
  const int64_t tokens = p.cu ? p.seq_len : (int64_t)p.num_seqs * p.seq_len;
  CUtensorMap tq, tk, tv;
  if (!make_tmap(&tq, p.q, DK, p.num_heads, tmap_rows(p, tokens, p.ext.q, DK)) ||
      !make_tmap(&tk, p.k, DK, p.num_heads, tmap_rows(p, tokens, p.ext.k, DK)) ||
      !make_tmap(&tv, p.v, p.dv, p.num_heads, tmap_rows(p, tokens, p.ext.v, p.dv)))
    return cudaErrorInvalidValue;
  // the block parts fused into the pass run in their own instantiation, so
  // the plain pass carries none of their code
  using Kern = decltype(&gdn_fwd_tc128_kernel<0>);
  const Kern inst[12] = {gdn_fwd_tc128_kernel<0>,
                         gdn_fwd_tc128_kernel<kFL2>,
                         gdn_fwd_tc128_kernel<kFEpi>,
                         gdn_fwd_tc128_kernel<kFL2 | kFEpi>,
                         gdn_fwd_tc128_kernel<kFSeg>,
                         gdn_fwd_tc128_kernel<kFSeg | kFL2>,
                         gdn_fwd_tc128_kernel<kFSeg | kFEpi>,
                         gdn_fwd_tc128_kernel<kFSeg | kFL2 | kFEpi>,
                         gdn_fwd_tc128_kernel<kFRank>,
                         gdn_fwd_tc128_kernel<kFRank | kFL2>,
                         gdn_fwd_tc128_kernel<kFRank | kFEpi>,
                         gdn_fwd_tc128_kernel<kFRank | kFL2 | kFEpi>};
  // packed sequences (never split) take the longest-first instances
  const bool rank = p.cu != nullptr && p.num_seqs > 1 && p.num_seqs <= kRankedSeqs;
  const int feat = ((p.flags & GDN_QK_L2NORM) ? kFL2 : 0) | ((p.d_skip || p.out_gate) ? kFEpi : 0);
  const Kern kern = p.seg_len > 0 ? inst[kFSeg | feat] : rank ? inst[8 | feat] : inst[feat];
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (err != cudaSuccess) return err;
  if (p.seg_len == 0) {
    const dim3 grid(p.dv / kDvt, p.num_heads, p.num_seqs);
    kern<<<grid, Cfg::kWarps * 32, L::ALLOC, stream>>>(p, tq, tk, tv);
    return cudaGetLastError();
  }
  // A split sequence (each segment maps its entry state H to M H + X and
  // its outputs o to o0 + r H; "Optimization Quartet", Triton GDN kernel
  // section 3.2, names the inter-chunk carry as the serial part of the
  // chunked form):
  //   1. one launch: segment 0 from the caller's state, writing the state
  //      that enters segment 1; segments 1 .. S-1 from zero (o0, X) and from
  //      the identity on dk extra columns (r, M); the first segments'
  //      CTAs are dispatched first, the longest;
  //   2. the composition H_(s+1) = M_s H_s + X_s for s = 1 .. S-1, in order,
  //      in one launch (the last step gives the caller's final state);
  //   3. the correction o += r H_s over segments 1 .. S-1.
  const int S = p.seg_count;
  const dim3 grid(p.dv / kDvt + DK / kDvt, p.num_heads, p.num_seqs * S);
  kern<<<grid, Cfg::kWarps * 32, L::ALLOC, stream>>>(p, tq, tk, tv);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if ((err = launch_seg_compose(p, 1, stream)) != cudaSuccess) return err;
  return launch_seg_correct(p, stream);
}

}  // namespace

bool tc_supported(int dk, int dv) { return (dk == 64 || dk == 128) && dv % kDvt == 0; }

// the split launch above takes dense dk = 128 calls, up to kMaxSegments segments
int seq_split_segments(const FwdParams &p) {
  return p.dk == DK && p.cu == nullptr ? kMaxSegments : 1;
}

cudaError_t launch_fwd_tc(const FwdParams &p, cudaStream_t stream) {
  switch (p.dk) {
    case 64: return launch_fwd_tc64(p, stream);
    case 128: return launch_tc128(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

#ifdef GDN_PHASE_PROBE
extern "C" int gdn_phase_probe_read_tc128(unsigned long long *host) {
  return (int)cudaMemcpyFromSymbol(host, gdn::tc::g_phase_probe, sizeof(gdn::tc::g_phase_probe));
}
#endif
