// The HyMo pages' own recurrence: a diagonal (per-state-row) decay, write key
// b, read key c, no erase term ("Model Architecture Walkthrough", section
// 5.2.1; "Optimization Quartet", Triton GDN kernel section 3.2):
//
//   h_t = exp(g_t A) (.) h_{t-1} + b_t v_t^T,   o_t = h_t^T c_t,   A = -exp(A_log[head])
//
// with h_t (S x D, fp32), one decay rate A_s per state row s.
//
// Work split.  A CTA of 8 warps owns 128 consecutive tokens of one (batch row,
// head); warp w owns the 16-token chunk w.  With G_i the within-chunk inclusive
// sum of g and alpha_i,s = exp(A_s g_i):
//
//   o_i  = (c_i (.) E_i)^T h_start  +  sum_{j<=i} P_ij v_j,
//   P_ij = sum_s c_i,s b_j,s exp(A_s (G_i - G_j))                 (intra-chunk)
//   h_end = gamma (.) h_start + sum_j (b_j (.) F_j) v_j^T          (state update)
//
// E_i = prod_{v<=i} alpha_v, F_j = prod_{v>j} alpha_v, gamma = prod_v alpha_v: all
// products of factors <= 1, so nothing overflows however fast a head decays.
// The per-row decay of P cannot be split into a row factor times a column
// factor over the whole chunk without overflow (exp(-A_s G_j) is unbounded), so
// P is built level by level: a pair (i > j) whose indices first differ in bit
// l is split at the last index of the lower 2^l-block, and both halves of the
// split decay are products of alphas inside that block.  Each level is one
// rank-32 product X_l X_l^T on the tensor cores, where row i of X_l is c_i
// times a prefix product (i in the upper half of its 2^(l+1)-block) or b_i times
// a suffix product (lower half); the diagonal is c b^T.
//
// Chunk to chunk, and CTA to CTA, the state is an elementwise affine map
// h -> gamma (.) h + dH.  The 8 chunk maps of a CTA are composed in shared
// memory; across CTAs the start state comes from a decoupled look-back: each
// CTA publishes its aggregate map, then walks back over its predecessors'
// published maps until it meets one that published its end state.  CTAs take
// their (head, 128-token block) from a ticket counter in launch order, so a
// CTA only ever waits on CTAs that are already running; every wait is bounded.
//
// bf16 storage: operands are bf16 on mma.sync with fp32 accumulation.  fp32
// storage: every operand is split into bf16 hi + lo and each product takes
// three MMAs (hi*hi + hi*lo + lo*hi), about 2^-16 relative.
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_tc_common.cuh"

namespace gdn {
namespace diag {

using namespace ptx;

constexpr int kS = 32;            // state rows (d_state)
constexpr int kD = 32;            // value columns (head_dim)
constexpr int kCT = 16;           // tokens per warp chunk
constexpr int kNW = 8;            // warps (chunks) per CTA
constexpr int kSC = kCT * kNW;    // tokens per CTA
constexpr int kThreads = 32 * kNW;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kAgg = 1, kIncl = 2;   // flag states (low 2 bits)

// Workspace: [0, 256) status word (first 16 bytes) and counters at byte 64;
// then one flag per (head, block), one aggregate map and one end state.
struct Counters {
  uint32_t ticket, done, epoch, pad;
};
constexpr size_t kCountersOff = 64;
constexpr size_t kAggFloats = kS * kD + kS;   // dH (fragment order) then gamma
constexpr size_t kInclFloats = kS * kD;

struct Workspace {
  size_t flags, agg, incl, total;
};
inline Workspace workspace_layout(int64_t tasks) {
  Workspace w;
  w.flags = kStatusBytes;
  w.agg = (w.flags + (size_t)tasks * 4 + 255) & ~(size_t)255;
  w.incl = w.agg + (size_t)tasks * kAggFloats * 4;
  w.total = w.incl + (size_t)tasks * kInclFloats * 4;
  return w;
}

struct DiagParams {
  const float *g, *A_log, *h0;
  float *hN;
  DeviceStatus *status;
  Counters *ctr;
  uint32_t *flags;
  float *agg, *incl;
  int32_t batch, seq_len, num_heads, nblk;   // nblk = 128-token blocks per sequence
};

// Shared-memory layout for storage type T.
template <typename T>
struct Lay {
  static constexpr bool SPLIT = sizeof(T) == 4;
  static constexpr int NP = SPLIT ? 2 : 1;          // bf16 planes per staged operand
  static constexpr int ROWB = 32 * (int)sizeof(T);  // bytes per input row
  static constexpr int TILE = kSC * ROWB;           // one TMA input tile
  static constexpr int SUB = kCT * ROWB;            // one warp's rows of a tile
  static constexpr int PLANE = kCT * 64;            // 16 rows x 32 bf16
  static constexpr int XCH = 4 * NP * PLANE;        // level planes / dH / H fragments / o
  static constexpr int CTL = NP * PLANE;            // c~ = c (.) E
  static constexpr int BHT = NP * PLANE;            // b^ = b (.) F
  static constexpr int VSP = SPLIT ? 2 * PLANE : 0; // v hi/lo
  static constexpr int DGP = SPLIT ? 4 * PLANE : 0; // c hi/lo, b hi/lo (diagonal)
  static constexpr int WARP = XCH + CTL + BHT + VSP + DGP;
  static constexpr int OFF_V = 0, OFF_B = TILE, OFF_C = 2 * TILE;
  static constexpr int OFF_W = 3 * TILE;
  static constexpr int W_CT = XCH, W_BH = XCH + CTL, W_VS = W_BH + BHT, W_DG = W_VS + VSP;
  static constexpr int OFF_GAM = OFF_W + kNW * WARP;
  static constexpr int OFF_MISC = OFF_GAM + kNW * kS * 4;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;
  static constexpr int MIN_BLOCKS = SPLIT ? 1 : 3;
};

// Rows of 64 bytes (32 bf16) with the 64-byte swizzle: 16-byte granule index
// XOR (row / 2) mod 4, the layout TMA writes with SWIZZLE_64B.
__device__ __forceinline__ uint32_t sw64(uint32_t base, int row, int byte) {
  return base + row * 64 + ((((byte >> 4) ^ (row >> 1)) & 3) << 4) + (byte & 15);
}
// Rows of 128 bytes (32 fp32) with the 128-byte swizzle (granule XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int byte) {
  return base + row * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void sts32f(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// One token's pair of inputs (state rows 2sp, 2sp+1, or value columns) as held
// by a prep lane.
template <typename T> struct Pair;
template <> struct Pair<__nv_bfloat16> {
  uint32_t r;
  __device__ __forceinline__ float x() const { return bf16_lo(r); }
  __device__ __forceinline__ float y() const { return bf16_hi(r); }
};
template <> struct Pair<float> {
  float2 r;
  __device__ __forceinline__ float x() const { return r.x; }
  __device__ __forceinline__ float y() const { return r.y; }
};

template <typename T>
__device__ __forceinline__ Pair<T> load_pair(uint32_t sub, int row, int pair);
template <>
__device__ __forceinline__ Pair<__nv_bfloat16> load_pair<__nv_bfloat16>(uint32_t sub, int row,
                                                                        int pair) {
  return Pair<__nv_bfloat16>{lds32(sw64(sub, row, 4 * pair))};
}
template <>
__device__ __forceinline__ Pair<float> load_pair<float>(uint32_t sub, int row, int pair) {
  return Pair<float>{lds64f(sw128(sub, row, 8 * pair))};
}

// Store (x, y) as bf16 into a staged plane; with NP == 2 also the residual
// (x - bf16(x), y - bf16(y)) into the lo plane one PLANE further.
template <int NP>
__device__ __forceinline__ void put(uint32_t plane, int row, int pair, float x, float y) {
  const uint32_t a = sw64(plane, row, 4 * pair);
  const uint32_t hi = pack_bf16(x, y);
  sts32(a, hi);
  if (NP == 2) sts32(a + kCT * 64, pack_bf16(x - bf16_lo(hi), y - bf16_hi(hi)));
}
template <typename T, int NP>
__device__ __forceinline__ void put_raw(uint32_t plane, int row, int pair, const Pair<T> &v) {
  if constexpr (NP == 1 && sizeof(T) == 2) {
    sts32(sw64(plane, row, 4 * pair), v.r);
  } else {
    put<NP>(plane, row, pair, v.x(), v.y());
  }
}

// ---- warp MMA on (possibly split) bf16 operands ----
template <int NP>
__device__ __forceinline__ void mma_np(float (&d)[4], const uint32_t (&a)[NP][4],
                                       const uint32_t (&b0)[NP], const uint32_t (&b1)[NP]) {
  mma_bf16(d, a[0][0], a[0][1], a[0][2], a[0][3], b0[0], b1[0]);
  if constexpr (NP == 2) {
    mma_bf16(d, a[0][0], a[0][1], a[0][2], a[0][3], b0[1], b1[1]);
    mma_bf16(d, a[1][0], a[1][1], a[1][2], a[1][3], b0[0], b1[0]);
  }
}

// The 16x16 product of two staged [16 rows][32] planes, X_A X_B^T, as two
// 16x8 accumulators (n-tile 0: columns 0-7, n-tile 1: columns 8-15).
template <int NP, bool NT1, bool SAME>
__device__ __forceinline__ void gram16(float (&R)[2][4], uint32_t pa, uint32_t pb, int lane) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int q = 0; q < 4; ++q) R[nt][q] = 0.f;
  const int row = lane & 15, colb = (lane >> 4) * 16;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    uint32_t a[NP][4], b[NP][4];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      ldsm_x4(sw64(pa + p * kCT * 64, row, ks * 32 + colb), a[p][0], a[p][1], a[p][2], a[p][3]);
      if constexpr (SAME) {
#pragma unroll
        for (int e = 0; e < 4; ++e) b[p][e] = a[p][e];
      } else {
        ldsm_x4(sw64(pb + p * kCT * 64, row, ks * 32 + colb), b[p][0], b[p][1], b[p][2],
                b[p][3]);
      }
    }
    uint32_t b0[NP], b1[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) { b0[p] = b[p][0]; b1[p] = b[p][2]; }
    mma_np<NP>(R[0], a, b0, b1);
    if (NT1) {
#pragma unroll
      for (int p = 0; p < NP; ++p) { b0[p] = b[p][1]; b1[p] = b[p][3]; }
      mma_np<NP>(R[1], a, b0, b1);
    }
  }
}

// A fragments of V^T (rows = value columns d, k = tokens j) for m-tile md.
template <int NP>
__device__ __forceinline__ void load_vt(uint32_t (&a)[NP][4], uint32_t vplane, int md, int lane) {
  const int mi = lane >> 3;
  const int row = (lane & 7) + 8 * (mi >> 1), col = 16 * md + 8 * (mi & 1);
#pragma unroll
  for (int p = 0; p < NP; ++p)
    ldsm_x4_t(sw64(vplane + p * kCT * 64, row, 2 * col), a[p][0], a[p][1], a[p][2], a[p][3]);
}

__device__ __forceinline__ bool spin_flag(const uint32_t *f, uint32_t tag, uint32_t &state) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    const uint32_t v = ld_acquire_gpu(f);
    if ((v & ~3u) == tag && (v & 3u) != 0) {
      state = v & 3u;
      return true;
    }
    if ((it & 15u) == 15u) {
      if (globaltimer_ns() - t0 > kWaitNs) return false;
      __nanosleep(64);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, Lay<T>::MIN_BLOCKS)
gdn_diag_kernel(const DiagParams p, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                const __grid_constant__ CUtensorMap tm_o) {
  using L = Lay<T>;
  constexpr int NP = L::NP;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char *sptr = smem_raw + (sbase - smem_u32(smem_raw));
  uint32_t *misc = reinterpret_cast<uint32_t *>(sptr + L::OFF_MISC);
  const uint32_t bar = sbase + L::OFF_MISC;        // mbarrier (8 bytes)
  // misc[2]: ticket, misc[3]: epoch tag, misc[4..5]: look-back flag broadcast

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int heads_total = p.batch * p.num_heads;
  const int64_t tasks = (int64_t)heads_total * p.nblk;

  if (tid == 0) {
    const uint32_t ep = *reinterpret_cast<volatile uint32_t *>(&p.ctr->epoch);
    const uint32_t t = atomicAdd(&p.ctr->ticket, 1u);
    misc[2] = t;
    misc[3] = (ep & 0x3fffffffu) << 2;
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t ticket = misc[2], tag = misc[3];
  const bool valid = (int64_t)ticket < tasks;
  const int blk = valid ? (int)(ticket / (uint32_t)heads_total) : 0;
  const int head = valid ? (int)(ticket % (uint32_t)heads_total) : 0;
  const int bb = head / p.num_heads, hd = head % p.num_heads;
  const int t0 = blk * kSC;
  const int64_t task = (int64_t)head * p.nblk + blk;
  if (!valid && tid == 0) report(p.status, GDN_ERR_DEVICE_CHECK, 0u, 0u, ticket);

  if (tid == 0 && valid) {
    mbar_arrive_expect_tx(bar, 3 * L::TILE);
    tma_load_4d(sbase + L::OFF_V, &tm_v, 0, hd, t0, bb, bar);
    tma_load_4d(sbase + L::OFF_B, &tm_b, 0, hd, t0, bb, bar);
    tma_load_4d(sbase + L::OFF_C, &tm_c, 0, hd, t0, bb, bar);
  }

  // gate of token (16 warp + lane) for lanes 0..15 (0 past the end: no decay)
  const int tok_w = t0 + kCT * warp;
  float gtok = 0.f;
  if (lane < kCT && tok_w + lane < p.seq_len)
    gtok = __ldg(p.g + ((int64_t)bb * p.seq_len + tok_w + lane) * p.num_heads + hd);
  // scaled decay rates A_s log2(e) of this lane's state rows 2sp, 2sp+1
  const int sp = lane & 15, hh = lane >> 4;
  const float ah0 = -__expf(__ldg(p.A_log + hd * kS + 2 * sp)) * kLog2e;
  const float ah1 = -__expf(__ldg(p.A_log + hd * kS + 2 * sp + 1)) * kLog2e;

  if (valid && !mbar_wait_bounded(bar, 0, kWaitNs))
    report(p.status, GDN_ERR_TIMEOUT, (uint32_t)bb, (uint32_t)hd, 1u);

  const uint32_t wbase = sbase + L::OFF_W + warp * L::WARP;
  const uint32_t xch = wbase, ctl = wbase + L::W_CT, bht = wbase + L::W_BH;
  const uint32_t subv = sbase + L::OFF_V + warp * L::SUB;
  const uint32_t subb = sbase + L::OFF_B + warp * L::SUB;
  const uint32_t subc = sbase + L::OFF_C + warp * L::SUB;
  const uint32_t vplane = L::SPLIT ? wbase + L::W_VS : subv;
  const uint32_t cdiag = L::SPLIT ? wbase + L::W_DG : subc;
  const uint32_t bdiag = L::SPLIT ? wbase + L::W_DG + 2 * L::PLANE : subb;
  float *gam = reinterpret_cast<float *>(sptr + L::OFF_GAM);

  // =================== step 1: the chunk of this warp ===================
  // ---- prep: lane (sp, hh) owns state rows 2sp, 2sp+1 of tokens 8hh..8hh+7 ----
  {
    Pair<T> cr[8], br[8];
    float a0[8], a1[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = 8 * hh + u;
      cr[u] = load_pair<T>(subc, r, sp);
      br[u] = load_pair<T>(subb, r, sp);
      const float gu = __shfl_sync(0xffffffffu, gtok, r);
      a0[u] = exp2f(ah0 * gu);
      a1[u] = exp2f(ah1 * gu);
    }
    if constexpr (L::SPLIT) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int r = 8 * hh + u;
        const Pair<T> vv = load_pair<T>(subv, r, sp);
        put<2>(vplane, r, sp, vv.x(), vv.y());
        put<2>(cdiag, r, sp, cr[u].x(), cr[u].y());
        put<2>(bdiag, r, sp, br[u].x(), br[u].y());
      }
    }
    const uint32_t X0 = xch, X1 = xch + NP * L::PLANE, X2 = xch + 2 * NP * L::PLANE,
                   X3 = xch + 3 * NP * L::PLANE;
    // level 0: pairs (2m+1, 2m); upper (odd) rows c alpha, lower rows b
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = 8 * hh + u;
      if (u & 1) put<NP>(X0, r, sp, cr[u].x() * a0[u], cr[u].y() * a1[u]);
      else put_raw<T, NP>(X0, r, sp, br[u]);
    }
    // level 1: blocks {0,1 | 2,3} within each 4-block
    {
      const float p23x = a0[2] * a0[3], p23y = a1[2] * a1[3];
      const float p67x = a0[6] * a0[7], p67y = a1[6] * a1[7];
      put<NP>(X1, 8 * hh + 0, sp, br[0].x() * a0[1], br[0].y() * a1[1]);
      put_raw<T, NP>(X1, 8 * hh + 1, sp, br[1]);
      put<NP>(X1, 8 * hh + 2, sp, cr[2].x() * a0[2], cr[2].y() * a1[2]);
      put<NP>(X1, 8 * hh + 3, sp, cr[3].x() * p23x, cr[3].y() * p23y);
      put<NP>(X1, 8 * hh + 4, sp, br[4].x() * a0[5], br[4].y() * a1[5]);
      put_raw<T, NP>(X1, 8 * hh + 5, sp, br[5]);
      put<NP>(X1, 8 * hh + 6, sp, cr[6].x() * a0[6], cr[6].y() * a1[6]);
      put<NP>(X1, 8 * hh + 7, sp, cr[7].x() * p67x, cr[7].y() * p67y);
    }
    // level 2: blocks {0..3 | 4..7}; up2 = prefix from 4, lo2 = suffix to 3
    float up2x[8], up2y[8], lo2x[4], lo2y[4];
    up2x[4] = a0[4]; up2y[4] = a1[4];
#pragma unroll
    for (int u = 5; u < 8; ++u) { up2x[u] = up2x[u - 1] * a0[u]; up2y[u] = up2y[u - 1] * a1[u]; }
    lo2x[3] = 1.f; lo2y[3] = 1.f;
#pragma unroll
    for (int u = 2; u >= 0; --u) { lo2x[u] = lo2x[u + 1] * a0[u + 1]; lo2y[u] = lo2y[u + 1] * a1[u + 1]; }
#pragma unroll
    for (int u = 0; u < 3; ++u) put<NP>(X2, 8 * hh + u, sp, br[u].x() * lo2x[u], br[u].y() * lo2y[u]);
    put_raw<T, NP>(X2, 8 * hh + 3, sp, br[3]);
#pragma unroll
    for (int u = 4; u < 8; ++u) put<NP>(X2, 8 * hh + u, sp, cr[u].x() * up2x[u], cr[u].y() * up2y[u]);
    // prefix (inclusive) and suffix (exclusive) products over this half
    float prex[8], prey[8], sufx[8], sufy[8];
    prex[0] = a0[0]; prey[0] = a1[0];
#pragma unroll
    for (int u = 1; u < 4; ++u) { prex[u] = prex[u - 1] * a0[u]; prey[u] = prey[u - 1] * a1[u]; }
#pragma unroll
    for (int u = 4; u < 8; ++u) { prex[u] = prex[3] * up2x[u]; prey[u] = prey[3] * up2y[u]; }
    sufx[7] = 1.f; sufy[7] = 1.f;
#pragma unroll
    for (int u = 6; u >= 4; --u) { sufx[u] = sufx[u + 1] * a0[u + 1]; sufy[u] = sufy[u + 1] * a1[u + 1]; }
#pragma unroll
    for (int u = 0; u < 4; ++u) { sufx[u] = lo2x[u] * up2x[7]; sufy[u] = lo2y[u] * up2y[7]; }
    // level 3: the two halves; upper half c prefix, lower half b suffix
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = 8 * hh + u;
      if (hh) put<NP>(X3, r, sp, cr[u].x() * prex[u], cr[u].y() * prey[u]);
      else put<NP>(X3, r, sp, br[u].x() * sufx[u], br[u].y() * sufy[u]);
    }
    // whole-chunk prefix E and suffix F: the other half's total product
    const float ox = __shfl_xor_sync(0xffffffffu, prex[7], 16);
    const float oy = __shfl_xor_sync(0xffffffffu, prey[7], 16);
    const float ex = hh ? ox : 1.f, ey = hh ? oy : 1.f;   // E = ex * pre
    const float fx = hh ? 1.f : ox, fy = hh ? 1.f : oy;   // F = fx * suf
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = 8 * hh + u;
      put<NP>(ctl, r, sp, cr[u].x() * (ex * prex[u]), cr[u].y() * (ey * prey[u]));
      put<NP>(bht, r, sp, br[u].x() * (fx * sufx[u]), br[u].y() * (fy * sufy[u]));
    }
    if (hh) {   // gamma = E of the last token
      gam[warp * kS + 2 * sp] = ex * prex[7];
      gam[warp * kS + 2 * sp + 1] = ey * prey[7];
    }
  }
  __syncwarp();

  // ---- P (16 x 16, lower triangle) level by level ----
  // Element (nt, q) of a 16x8 accumulator is (row g + 8 (q >> 1), col 8 nt + 2t + (q & 1)).
  const int g = lane >> 2, tq = lane & 3;
  int lev[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = 2 * tq + e;
    lev[e] = g > j ? 31 - __clz(g ^ j) : (g == j ? 4 : 5);
  }
  float p00 = 0.f, p01 = 0.f, p02, p03, p12 = 0.f, p13 = 0.f;
  {
    float R[2][4];
    gram16<NP, false, true>(R, xch + 3 * NP * L::PLANE, xch + 3 * NP * L::PLANE, lane);
    p02 = R[0][2];
    p03 = R[0][3];
#pragma unroll
    for (int l = 0; l < 3; ++l) {
      gram16<NP, true, true>(R, xch + l * NP * L::PLANE, xch + l * NP * L::PLANE, lane);
      if (lev[0] == l) { p00 = R[0][0]; p12 = R[1][2]; }
      if (lev[1] == l) { p01 = R[0][1]; p13 = R[1][3]; }
    }
    gram16<NP, true, false>(R, cdiag, bdiag, lane);
    if (lev[0] == 4) { p00 = R[0][0]; p12 = R[1][2]; }
    if (lev[1] == 4) { p01 = R[0][1]; p13 = R[1][3]; }
  }
  // P^T as B fragments (k = key token j, n = query token i), per 8-row block ni
  uint32_t pb0[NP][2], pb1[NP][2];
  {
    pb0[0][0] = pack_bf16(p00, p01);
    pb0[0][1] = 0u;
    pb1[0][0] = pack_bf16(p02, p03);
    pb1[0][1] = pack_bf16(p12, p13);
    if constexpr (NP == 2) {
      pb0[1][0] = pack_bf16(p00 - bf16_lo(pb0[0][0]), p01 - bf16_hi(pb0[0][0]));
      pb0[1][1] = 0u;
      pb1[1][0] = pack_bf16(p02 - bf16_lo(pb1[0][0]), p03 - bf16_hi(pb1[0][0]));
      pb1[1][1] = pack_bf16(p12 - bf16_lo(pb1[0][1]), p13 - bf16_hi(pb1[0][1]));
    }
  }

  // ---- dH^T (d x s) = V^T b^ ----
  {
    float dH[2][4][4];
#pragma unroll
    for (int md = 0; md < 2; ++md)
#pragma unroll
      for (int ns = 0; ns < 4; ++ns)
#pragma unroll
        for (int q = 0; q < 4; ++q) dH[md][ns][q] = 0.f;
    uint32_t va[2][NP][4];
    load_vt<NP>(va[0], vplane, 0, lane);
    load_vt<NP>(va[1], vplane, 1, lane);
    const int mi = lane >> 3;
#pragma unroll
    for (int nsp = 0; nsp < 2; ++nsp) {
      uint32_t bq[NP][4];
      const int row = (lane & 7) + 8 * (mi & 1), col = 8 * (2 * nsp + (mi >> 1));
#pragma unroll
      for (int pp = 0; pp < NP; ++pp)
        ldsm_x4_t(sw64(bht + pp * L::PLANE, row, 2 * col), bq[pp][0], bq[pp][1], bq[pp][2],
                  bq[pp][3]);
      uint32_t b0[NP], b1[NP], b2[NP], b3[NP];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        b0[pp] = bq[pp][0]; b1[pp] = bq[pp][1]; b2[pp] = bq[pp][2]; b3[pp] = bq[pp][3];
      }
#pragma unroll
      for (int md = 0; md < 2; ++md) {
        mma_np<NP>(dH[md][2 * nsp], va[md], b0, b1);
        mma_np<NP>(dH[md][2 * nsp + 1], va[md], b2, b3);
      }
    }
    __syncwarp();   // every lane is done reading the level planes
#pragma unroll
    for (int md = 0; md < 2; ++md)
#pragma unroll
      for (int ns = 0; ns < 4; ++ns) {
        float4 *dst = reinterpret_cast<float4 *>(sptr + (xch - sbase)) + ((md * 4 + ns) * 32 + lane);
        *dst = make_float4(dH[md][ns][0], dH[md][ns][1], dH[md][ns][2], dH[md][ns][3]);
      }
  }
  __syncthreads();

  // =================== step 2: compose the chunk maps (all threads) ===================
  // Thread (warp rg, lane l) owns fragment block rg = 4 md + ns of every chunk:
  // state elements (d, s) = (16 md + g + 8 (q >> 1), 8 ns + 2 tq + (q & 1)).
  const int md = warp >> 2, ns = warp & 3;
  const int s0 = 8 * ns + 2 * tq, d0 = 16 * md + g;
  auto dH_at = [&](int w) {
    return *reinterpret_cast<const float4 *>(sptr + L::OFF_W + w * L::WARP +
                                             ((warp * 32 + lane) << 4));
  };
  auto gam_at = [&](int w) { return *reinterpret_cast<const float2 *>(gam + w * kS + s0); };
  float4 agg = make_float4(0.f, 0.f, 0.f, 0.f);
  float2 G = make_float2(1.f, 1.f);
#pragma unroll
  for (int w = 0; w < kNW; ++w) {
    const float4 x = dH_at(w);
    const float2 gm = gam_at(w);
    agg.x = fmaf(gm.x, agg.x, x.x);
    agg.y = fmaf(gm.y, agg.y, x.y);
    agg.z = fmaf(gm.x, agg.z, x.z);
    agg.w = fmaf(gm.y, agg.w, x.w);
    G.x *= gm.x;
    G.y *= gm.y;
  }
  const int64_t head_task0 = (int64_t)head * p.nblk;
  const uint32_t fidx = (warp * 32 + lane) * 4;   // fragment-order float index
  if (valid && blk > 0) {
    float *ag = p.agg + task * kAggFloats;
    __stcg(reinterpret_cast<float4 *>(ag + fidx), agg);
    if (md == 0 && g == 0) __stcg(reinterpret_cast<float2 *>(ag + kS * kD + s0), G);
    __threadfence();
  }
  __syncthreads();
  if (tid == 0 && valid && blk > 0) st_release_gpu(p.flags + task, tag | kAgg);

  // ---- look-back: start state of this block ----
  auto init_at = [&]() {
    float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.h0) {
      const float *h0 = p.h0 + (int64_t)head * kS * kD;
      h.x = h0[s0 * kD + d0];
      h.y = h0[(s0 + 1) * kD + d0];
      h.z = h0[s0 * kD + d0 + 8];
      h.w = h0[(s0 + 1) * kD + d0 + 8];
    }
    return h;
  };
  float4 hs;
  {
    float4 dF = make_float4(0.f, 0.f, 0.f, 0.f);
    float2 gF = make_float2(1.f, 1.f);
    int j = blk - 1;
    int par = 0;
    bool done = j < 0 || !valid;
    hs = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < 0 && valid) hs = init_at();
    while (!done) {
      if (tid == 0) {
        uint32_t st = 0;
        if (!spin_flag(p.flags + head_task0 + j, tag, st)) {
          report(p.status, GDN_ERR_TIMEOUT, (uint32_t)bb, (uint32_t)hd, 2u);
          st = 3;
        }
        misc[4 + par] = st;
      }
      __syncthreads();
      const uint32_t st = misc[4 + par];
      par ^= 1;
      if (st == kIncl) {
        const float4 x = __ldcg(reinterpret_cast<const float4 *>(p.incl + (head_task0 + j) * kInclFloats + fidx));
        hs.x = fmaf(gF.x, x.x, dF.x);
        hs.y = fmaf(gF.y, x.y, dF.y);
        hs.z = fmaf(gF.x, x.z, dF.z);
        hs.w = fmaf(gF.y, x.w, dF.w);
        done = true;
      } else if (st == kAgg) {
        const float *ag = p.agg + (head_task0 + j) * kAggFloats;
        const float4 x = __ldcg(reinterpret_cast<const float4 *>(ag + fidx));
        const float2 gj = __ldcg(reinterpret_cast<const float2 *>(ag + kS * kD + s0));
        dF.x = fmaf(gF.x, x.x, dF.x);
        dF.y = fmaf(gF.y, x.y, dF.y);
        dF.z = fmaf(gF.x, x.z, dF.z);
        dF.w = fmaf(gF.y, x.w, dF.w);
        gF.x *= gj.x;
        gF.y *= gj.y;
        if (--j < 0) {
          const float4 x0 = init_at();
          hs.x = fmaf(gF.x, x0.x, dF.x);
          hs.y = fmaf(gF.y, x0.y, dF.y);
          hs.z = fmaf(gF.x, x0.z, dF.z);
          hs.w = fmaf(gF.y, x0.w, dF.w);
          done = true;
        }
      } else {   // timed out: carry on with what was composed so far
        hs = dF;
        done = true;
      }
    }
  }
  // ---- publish the end state of this block ----
  {
    float4 he;
    he.x = fmaf(G.x, hs.x, agg.x);
    he.y = fmaf(G.y, hs.y, agg.y);
    he.z = fmaf(G.x, hs.z, agg.z);
    he.w = fmaf(G.y, hs.w, agg.w);
    if (valid) {
      __stcg(reinterpret_cast<float4 *>(p.incl + task * kInclFloats + fidx), he);
      __threadfence();
      if (blk == p.nblk - 1 && p.hN) {
        float *hn = p.hN + (int64_t)head * kS * kD;
        hn[s0 * kD + d0] = he.x;
        hn[(s0 + 1) * kD + d0] = he.y;
        hn[s0 * kD + d0 + 8] = he.z;
        hn[(s0 + 1) * kD + d0 + 8] = he.w;
      }
    }
  }
  __syncthreads();
  if (tid == 0 && valid) st_release_gpu(p.flags + task, tag | kIncl);

  // ---- start state of every chunk, as bf16 A fragments of H^T ----
  uint32_t hf[kNW][NP][2];
  {
    float4 h = hs;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
      hf[w][0][0] = pack_bf16(h.x, h.y);
      hf[w][0][1] = pack_bf16(h.z, h.w);
      if constexpr (NP == 2) {
        hf[w][1][0] = pack_bf16(h.x - bf16_lo(hf[w][0][0]), h.y - bf16_hi(hf[w][0][0]));
        hf[w][1][1] = pack_bf16(h.z - bf16_lo(hf[w][0][1]), h.w - bf16_hi(hf[w][0][1]));
      }
      const float4 x = dH_at(w);
      const float2 gm = gam_at(w);
      h.x = fmaf(gm.x, h.x, x.x);
      h.y = fmaf(gm.y, h.y, x.y);
      h.z = fmaf(gm.x, h.z, x.z);
      h.w = fmaf(gm.y, h.w, x.w);
    }
  }
  __syncthreads();   // all reads of dH done
  {
    // block (md, ns): k-step ks = ns / 2; a-register 0/1 (k low) or 2/3 (k high)
    const int ks = ns >> 1, a_lo = (ns & 1) ? 2 : 0;
    const int i0 = (md * 2 + ks) * 4 + a_lo, i1 = i0 + 1;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
      uint32_t *dst = reinterpret_cast<uint32_t *>(sptr + L::OFF_W + w * L::WARP);
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        dst[pp * 512 + i0 * 32 + lane] = hf[w][pp][0];
        dst[pp * 512 + i1 * 32 + lane] = hf[w][pp][1];
      }
    }
  }
  __syncthreads();

  // =================== step 3: outputs of this warp's chunk ===================
  {
    float O[2][2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int q = 0; q < 4; ++q) O[a][b][q] = 0.f;
    const uint32_t *hsrc = reinterpret_cast<const uint32_t *>(sptr + (xch - sbase));
    // inter-chunk: O^T += H^T (c (.) E)^T
    const int row = lane & 15, colb = (lane >> 4) * 16;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t cb[NP][4];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp)
        ldsm_x4(sw64(ctl + pp * L::PLANE, row, ks * 32 + colb), cb[pp][0], cb[pp][1], cb[pp][2],
                cb[pp][3]);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        uint32_t a[NP][4];
#pragma unroll
        for (int pp = 0; pp < NP; ++pp)
#pragma unroll
          for (int e = 0; e < 4; ++e) a[pp][e] = hsrc[pp * 512 + ((m * 2 + ks) * 4 + e) * 32 + lane];
        uint32_t b0[NP], b1[NP];
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) { b0[pp] = cb[pp][0]; b1[pp] = cb[pp][2]; }
        mma_np<NP>(O[m][0], a, b0, b1);
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) { b0[pp] = cb[pp][1]; b1[pp] = cb[pp][3]; }
        mma_np<NP>(O[m][1], a, b0, b1);
      }
    }
    // intra-chunk: O^T += V^T P^T
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      uint32_t va[NP][4];
      load_vt<NP>(va, vplane, m, lane);
      uint32_t b0[NP], b1[NP];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) { b0[pp] = pb0[pp][0]; b1[pp] = pb0[pp][1]; }
      mma_np<NP>(O[m][0], va, b0, b1);
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) { b0[pp] = pb1[pp][0]; b1[pp] = pb1[pp][1]; }
      mma_np<NP>(O[m][1], va, b0, b1);
    }
    __syncwarp();   // H fragments consumed: the exchange slot becomes the o tile
    // o tile [16 tokens][32 columns] in the storage type, row-major
    if constexpr (sizeof(T) == 2) {
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) {
        const uint32_t addr = xch + (8 * ni + (lane & 7)) * 64 + (lane >> 3) * 16;
        stsm_x4_t(addr, pack_bf16(O[0][ni][0], O[0][ni][1]), pack_bf16(O[0][ni][2], O[0][ni][3]),
                  pack_bf16(O[1][ni][0], O[1][ni][1]), pack_bf16(O[1][ni][2], O[1][ni][3]));
      }
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int ni = 0; ni < 2; ++ni)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int d = 16 * m + g + 8 * (q >> 1), i = 8 * ni + 2 * tq + (q & 1);
            sts32f(xch + i * 128 + d * 4, O[m][ni][q]);
          }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && valid && tok_w < p.seq_len) {
      tma_store_4d(&tm_o, 0, hd, tok_w, bb, xch);
      bulk_commit();
      bulk_wait_read<0>();
    }
  }

  // ---- launch bookkeeping: the last CTA resets the ticket and advances the epoch ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t d = atomicAdd(&p.ctr->done, 1u);
    if ((int64_t)d == tasks - 1) {
      p.ctr->ticket = 0u;
      p.ctr->done = 0u;
      atomicAdd(&p.ctr->epoch, 1u);
      __threadfence();
    }
  }
}

namespace {

// [B][T][H][32] tensor of the storage type viewed as 4-D (32, H, T, B).
bool make_tmap4(CUtensorMap *m, const void *ptr, bool f32, int H, int T, int B, int box_t,
                bool swizzle) {
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc) return false;
  const cuuint64_t e = f32 ? 4 : 2;
  const cuuint64_t dims[4] = {32, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {32 * e, 32 * e * H, 32 * e * H * (cuuint64_t)T};
  const cuuint32_t box[4] = {32, 1, (cuuint32_t)box_t, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = !swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE
                                         : (f32 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                : CU_TENSOR_MAP_SWIZZLE_64B);
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
cudaError_t launch_t(const DiagParams &p, const void *v, const void *b, const void *c, void *o,
                     int64_t tasks, cudaStream_t stream) {
  using L = Lay<T>;
  const bool f32 = sizeof(T) == 4;
  CUtensorMap tv, tb, tc_, to;
  if (!make_tmap4(&tv, v, f32, p.num_heads, p.seq_len, p.batch, kSC, true) ||
      !make_tmap4(&tb, b, f32, p.num_heads, p.seq_len, p.batch, kSC, true) ||
      !make_tmap4(&tc_, c, f32, p.num_heads, p.seq_len, p.batch, kSC, true) ||
      !make_tmap4(&to, o, f32, p.num_heads, p.seq_len, p.batch, kCT, false))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(gdn_diag_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (err != cudaSuccess) return err;
  gdn_diag_kernel<T><<<(unsigned)tasks, kThreads, L::ALLOC, stream>>>(p, tv, tb, tc_, to);
  return cudaGetLastError();
}

bool aligned16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace diag
}  // namespace gdn

extern "C" size_t gdn_diag_workspace_size(int32_t batch, int32_t seq_len, int32_t num_heads,
                                          int32_t d_state, int32_t head_dim) {
  using namespace gdn::diag;
  if (batch <= 0 || seq_len <= 0 || num_heads <= 0 || d_state <= 0 || head_dim <= 0) return 0;
  const int64_t nblk = ((int64_t)seq_len + kSC - 1) / kSC;
  return workspace_layout((int64_t)batch * num_heads * nblk).total;
}

extern "C" gdn_status gdn_diag_fwd(const void *v, const void *b, const void *c, const float *g,
                                   const float *A_log, const float *initial_state, void *o,
                                   float *final_state, int32_t batch, int32_t seq_len,
                                   int32_t num_heads, int32_t d_state, int32_t head_dim,
                                   gdn_dtype dtype, uint32_t flags, void *workspace,
                                   size_t workspace_bytes, void *stream) {
  using namespace gdn;
  using namespace gdn::diag;
  if (batch <= 0 || seq_len <= 0 || num_heads <= 0 || d_state <= 0 || head_dim <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (flags != 0u) return GDN_ERR_INVALID_ARG;
  if (d_state != kS || head_dim != kD) return GDN_ERR_UNSUPPORTED;
  const int64_t nblk = ((int64_t)seq_len + kSC - 1) / kSC;
  const int64_t tasks = (int64_t)batch * num_heads * nblk;
  if (tasks > 0x7fffffffLL || (int64_t)batch * num_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (!v || !b || !c || !g || !A_log || !o) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {v, b, c, g, A_log, initial_state, o, final_state};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  if (!workspace) return GDN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GDN_ERR_INVALID_ARG;
  const Workspace wl = workspace_layout(tasks);
  if (workspace_bytes < wl.total) return GDN_ERR_WORKSPACE;

  const size_t e = dtype == GDN_F32 ? 4 : 2;
  const size_t rows = (size_t)batch * (size_t)seq_len * (size_t)num_heads;
  const size_t b_v = rows * kD * e, b_bc = rows * kS * e, b_g = rows * 4;
  const size_t b_A = (size_t)num_heads * kS * 4;
  const size_t b_state = (size_t)batch * num_heads * kS * kD * 4;
  struct Range { const void *p; size_t n; };
  const Range inputs[] = {{v, b_v}, {b, b_bc}, {c, b_bc}, {g, b_g}, {A_log, b_A},
                          {workspace, workspace_bytes}};
  for (const Range &r : inputs) {
    if (overlaps(o, b_v, r.p, r.n)) return GDN_ERR_INVALID_ARG;
    if (overlaps(final_state, b_state, r.p, r.n)) return GDN_ERR_INVALID_ARG;
  }
  if (overlaps(o, b_v, initial_state, b_state) || overlaps(o, b_v, final_state, b_state))
    return GDN_ERR_INVALID_ARG;
  if (initial_state && final_state && initial_state != final_state &&
      overlaps(initial_state, b_state, final_state, b_state))
    return GDN_ERR_INVALID_ARG;
  if (overlaps(workspace, workspace_bytes, initial_state, b_state)) return GDN_ERR_INVALID_ARG;

  unsigned char *ws = static_cast<unsigned char *>(workspace);
  DiagParams p;
  p.g = g; p.A_log = A_log; p.h0 = initial_state; p.hN = final_state;
  p.status = reinterpret_cast<DeviceStatus *>(ws);
  p.ctr = reinterpret_cast<Counters *>(ws + kCountersOff);
  p.flags = reinterpret_cast<uint32_t *>(ws + wl.flags);
  p.agg = reinterpret_cast<float *>(ws + wl.agg);
  p.incl = reinterpret_cast<float *>(ws + wl.incl);
  p.batch = batch; p.seq_len = seq_len; p.num_heads = num_heads; p.nblk = (int32_t)nblk;
  const cudaError_t err =
      dtype == GDN_F32 ? launch_t<float>(p, v, b, c, o, tasks, (cudaStream_t)stream)
                       : launch_t<__nv_bfloat16>(p, v, b, c, o, tasks, (cudaStream_t)stream);
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
