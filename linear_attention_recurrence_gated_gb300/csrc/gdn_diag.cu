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

#ifdef GDN_DIAG_PROBE
// Phase-timing build only: globaltimer stamps of thread 0, [ticket][phase].
static __device__ unsigned long long g_diag_probe[8192 * 12];
#define GDN_DPROBE(k)                                                   \
  do {                                                                  \
    if (threadIdx.x == 0 && probe_id < 8192u)                           \
      ::gdn::diag::g_diag_probe[probe_id * 12u + (k)] = globaltimer_ns(); \
  } while (0)
#else
#define GDN_DPROBE(k) \
  do {                \
  } while (0)
#endif

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
  const float *D_skip, *out_gate;   // block epilogue (NULL = off)
  uint32_t opts;                    // GDN_GATE_SIGMOID
  float *hN;
  void *o;
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
__device__ __forceinline__ void sts32f(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// (x, y) as bf16 at plane + off; with NP == 2 also the residual into the lo
// plane one PLANE further.
template <int NP>
__device__ __forceinline__ void put2(unsigned char *plane, int off, float2 v) {
  const uint32_t hi = pack_bf16(v.x, v.y);
  *reinterpret_cast<uint32_t *>(plane + off) = hi;
  if constexpr (NP == 2)
    *reinterpret_cast<uint32_t *>(plane + off + kCT * 64) =
        pack_bf16(v.x - bf16_lo(hi), v.y - bf16_hi(hi));
}

// Two fp32 products in one packed instruction.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
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

template <typename T>
__global__ void __launch_bounds__(kThreads, Lay<T>::MIN_BLOCKS)
gdn_diag_kernel(const DiagParams p, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c) {
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

#ifdef GDN_DIAG_PROBE
  uint32_t probe_id = 0xffffffffu;
#endif
  if (tid == 0) {
    const uint32_t ep = *reinterpret_cast<volatile uint32_t *>(&p.ctr->epoch);
    misc[2] = atomicAdd(&p.ctr->ticket, 1u);
    misc[3] = (ep & 0x3fffffffu) << 2;
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t tag = misc[3];
  uint32_t ticket = misc[2];

  // Inputs of block `t`: v, b, c tiles by TMA (one thread), and the gates of
  // this warp's 16 tokens into lanes 0..15 (0 past the end: no decay).
  auto issue_tiles = [&](uint32_t t) {
    const int hdx = (int)(t % (uint32_t)heads_total);
    const int blk_ = (int)(t / (uint32_t)heads_total);
    const int b_ = hdx / p.num_heads, h_ = hdx % p.num_heads;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, 3 * L::TILE);
    tma_load_4d(sbase + L::OFF_V, &tm_v, 0, h_, blk_ * kSC, b_, bar);
    tma_load_4d(sbase + L::OFF_B, &tm_b, 0, h_, blk_ * kSC, b_, bar);
    tma_load_4d(sbase + L::OFF_C, &tm_c, 0, h_, blk_ * kSC, b_, bar);
  };
  auto load_gate = [&](uint32_t t) {
    float x = 0.f;
    if ((int64_t)t < tasks && lane < kCT) {
      const int hdx = (int)(t % (uint32_t)heads_total);
      const int tok = (int)(t / (uint32_t)heads_total) * kSC + kCT * warp + lane;
      const int b_ = hdx / p.num_heads, h_ = hdx % p.num_heads;
      if (tok < p.seq_len) {
        x = __ldg(p.g + ((int64_t)b_ * p.seq_len + tok) * p.num_heads + h_);
        if (p.opts & GDN_GATE_SIGMOID) x = 1.f / (1.f + __expf(-x));
      }
    }
    return x;
  };
  if (tid == 0 && (int64_t)ticket < tasks) issue_tiles(ticket);
  float gtok = load_gate(ticket);
  const int sp = lane & 15, hh = lane >> 4;
  uint32_t phase = 0;

  // Persistent loop: one 128-token block per iteration.  The next block's
  // ticket and tiles are taken as soon as this block's tiles are consumed.
  while ((int64_t)ticket < tasks) {
#ifdef GDN_DIAG_PROBE
  probe_id = ticket;
#endif
  GDN_DPROBE(0);
  const bool valid = true;
  const int blk = (int)(ticket / (uint32_t)heads_total);
  const int head = (int)(ticket % (uint32_t)heads_total);
  const int bb = head / p.num_heads, hd = head % p.num_heads;
  const int t0 = blk * kSC;
  const int64_t task = (int64_t)head * p.nblk + blk;
  const int tok_w = t0 + kCT * warp;
  // output gate of token (16 warp + lane) for lanes 0..15 (block epilogue)
  float ogate = 1.f;
  if (p.out_gate && lane < kCT && tok_w + lane < p.seq_len)
    ogate = __ldg(p.out_gate + ((int64_t)bb * p.seq_len + tok_w + lane) * p.num_heads + hd);
  // scaled decay rates A_s log2(e) of this lane's state rows 2sp, 2sp+1
  const float ah0 = -__expf(__ldg(p.A_log + hd * kS + 2 * sp)) * kLog2e;
  const float ah1 = -__expf(__ldg(p.A_log + hd * kS + 2 * sp + 1)) * kLog2e;
  __syncwarp();   // this warp's previous o tile is copied out of its exchange slot

  if (!mbar_wait_bounded(bar, phase, kWaitNs))
    report(p.status, GDN_ERR_TIMEOUT, (uint32_t)bb, (uint32_t)hd, 1u);
  GDN_DPROBE(2);

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
    // Byte offset of (row 8hh + u, pair sp) in a plane of 64-byte rows with the
    // 64-byte swizzle is o64[(u >> 1) & 3] + 64 u; in a tile of 128-byte fp32
    // rows with the 128-byte swizzle it is o128[u] + 128 u.
    int o64[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) o64[k] = hh * 512 + ((((sp >> 2) ^ k) & 3) << 4) + (sp & 3) * 4;
    unsigned char *const wp = sptr + (wbase - sbase);
    unsigned char *const tb = sptr + L::OFF_B + warp * L::SUB;
    unsigned char *const tcp = sptr + L::OFF_C + warp * L::SUB;
    auto off = [&](int u) { return o64[(u >> 1) & 3] + 64 * u; };

    float2 cf[8], bfv[8];
    uint32_t braw[8];
    if constexpr (!L::SPLIT) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t rc = *reinterpret_cast<const uint32_t *>(tcp + off(u));
        braw[u] = *reinterpret_cast<const uint32_t *>(tb + off(u));
        cf[u] = make_float2(bf16_lo(rc), bf16_hi(rc));
        bfv[u] = make_float2(bf16_lo(braw[u]), bf16_hi(braw[u]));
      }
    } else {
      int o128[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) o128[u] = hh * 1024 + (((sp >> 1) ^ u) << 4) + (sp & 1) * 8;
      unsigned char *const tv = sptr + L::OFF_V + warp * L::SUB;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int a = o128[u] + 128 * u;
        cf[u] = *reinterpret_cast<const float2 *>(tcp + a);
        bfv[u] = *reinterpret_cast<const float2 *>(tb + a);
        const float2 vv = *reinterpret_cast<const float2 *>(tv + a);
        put2<2>(wp + L::W_VS, off(u), vv);
        put2<2>(wp + L::W_DG, off(u), cf[u]);
        put2<2>(wp + L::W_DG + 2 * L::PLANE, off(u), bfv[u]);
        braw[u] = 0u;
      }
    }
    // per-token decay factors alpha_u = 2^(A_s log2(e) g_u)
    float2 al[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float gu = __shfl_sync(0xffffffffu, gtok, 8 * hh + u);
      const float2 e = mul2(make_float2(ah0, ah1), make_float2(gu, gu));
      al[u] = make_float2(ex2(e.x), ex2(e.y));
    }
    auto raw_b = [&](unsigned char *plane, int u) {
      if constexpr (!L::SPLIT) *reinterpret_cast<uint32_t *>(plane + off(u)) = braw[u];
      else put2<2>(plane, off(u), bfv[u]);
    };
    unsigned char *const X0 = wp, *const X1 = wp + NP * L::PLANE,
                  *const X2 = wp + 2 * NP * L::PLANE, *const X3 = wp + 3 * NP * L::PLANE;
    // level 0: pairs (2m+1, 2m); upper (odd) rows c alpha, lower rows b
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u & 1) put2<NP>(X0, off(u), mul2(cf[u], al[u]));
      else raw_b(X0, u);
    }
    // level 1: blocks {0,1 | 2,3} within each 4-block
    const float2 p23 = mul2(al[2], al[3]), p67 = mul2(al[6], al[7]);
    put2<NP>(X1, off(0), mul2(bfv[0], al[1]));
    raw_b(X1, 1);
    put2<NP>(X1, off(2), mul2(cf[2], al[2]));
    put2<NP>(X1, off(3), mul2(cf[3], p23));
    put2<NP>(X1, off(4), mul2(bfv[4], al[5]));
    raw_b(X1, 5);
    put2<NP>(X1, off(6), mul2(cf[6], al[6]));
    put2<NP>(X1, off(7), mul2(cf[7], p67));
    // level 2: blocks {0..3 | 4..7}; up2 = prefix from 4, lo2 = suffix to 3
    float2 up2[8], lo2[4];
    up2[4] = al[4];
    up2[5] = mul2(up2[4], al[5]);
    up2[6] = mul2(up2[5], al[6]);
    up2[7] = mul2(up2[6], al[7]);
    lo2[2] = al[3];
    lo2[1] = p23;
    lo2[0] = mul2(p23, al[1]);
#pragma unroll
    for (int u = 0; u < 3; ++u) put2<NP>(X2, off(u), mul2(bfv[u], lo2[u]));
    raw_b(X2, 3);
#pragma unroll
    for (int u = 4; u < 8; ++u) put2<NP>(X2, off(u), mul2(cf[u], up2[u]));
    // prefix (inclusive) and suffix (exclusive) products over this half
    float2 pre[8], suf[8];
    pre[0] = al[0];
#pragma unroll
    for (int u = 1; u < 4; ++u) pre[u] = mul2(pre[u - 1], al[u]);
#pragma unroll
    for (int u = 4; u < 8; ++u) pre[u] = mul2(pre[3], up2[u]);
    suf[7] = make_float2(1.f, 1.f);
    suf[6] = al[7];
    suf[5] = p67;
    suf[4] = mul2(p67, al[5]);
    suf[3] = up2[7];
#pragma unroll
    for (int u = 0; u < 3; ++u) suf[u] = mul2(lo2[u], up2[7]);
    // level 3: the two halves; upper half c prefix, lower half b suffix
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float2 x = hh ? cf[u] : bfv[u];
      const float2 f = hh ? pre[u] : suf[u];
      put2<NP>(X3, off(u), mul2(x, f));
    }
    // whole-chunk prefix E and suffix F: the other half's total product
    const float2 ot = make_float2(__shfl_xor_sync(0xffffffffu, pre[7].x, 16),
                                  __shfl_xor_sync(0xffffffffu, pre[7].y, 16));
    const float2 one = make_float2(1.f, 1.f);
    const float2 ex = hh ? ot : one;   // E = ex * pre
    const float2 fx = hh ? one : ot;   // F = fx * suf
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      put2<NP>(wp + L::W_CT, off(u), mul2(cf[u], mul2(ex, pre[u])));
      put2<NP>(wp + L::W_BH, off(u), mul2(bfv[u], mul2(fx, suf[u])));
    }
    if (hh) {   // gamma = E of the last token
      const float2 gm = mul2(ex, pre[7]);
      *reinterpret_cast<float2 *>(gam + warp * kS + 2 * sp) = gm;
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
  // (the V^T fragments are kept for the intra-chunk output: the tiles are
  // refilled with the next block while this one finishes)
  uint32_t va[2][NP][4];
  {
    float dH[2][4][4];
#pragma unroll
    for (int md = 0; md < 2; ++md)
#pragma unroll
      for (int ns = 0; ns < 4; ++ns)
#pragma unroll
        for (int q = 0; q < 4; ++q) dH[md][ns][q] = 0.f;
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
  // every read of this block's tiles is done: take the next block
  if (warp == 2 && lane == 0) {
    const uint32_t nt = atomicAdd(&p.ctr->ticket, 1u);
    misc[6] = nt;
    if ((int64_t)nt < tasks) issue_tiles(nt);
  }

  GDN_DPROBE(3);
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
  }
  __syncthreads();
  if (tid == 0 && valid && blk > 0) st_release_gpu(p.flags + task, tag | kAgg);
  GDN_DPROBE(4);

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
  float4 hs = make_float4(0.f, 0.f, 0.f, 0.f);
  {
    float4 dF = make_float4(0.f, 0.f, 0.f, 0.f);
    float2 gF = make_float2(1.f, 1.f);
    int j = blk - 1;   // nearest predecessor not yet composed
    int par = 0;
    bool done = !valid;
    while (!done) {
      // warp 1 reads the flags of predecessors j, j-1, ..., j-31 at once and
      // finds the nearest that published its end state (before the start of
      // the sequence counts as one: the initial state); all nearer ones must
      // have published their aggregate maps.  (Warp 0 may still be in the
      // release store of this block's aggregate.)
      if (warp == 1) {
        const int jl = j - lane;
        uint32_t st = jl < 0 ? kIncl : 0u;
        int m = 33;
        const uint64_t t_start = globaltimer_ns();
        for (uint32_t it = 0;; ++it) {
          if (st != kIncl) {
            const uint32_t v = ld_acquire_gpu(p.flags + head_task0 + jl);
            if ((v & ~3u) == tag && (v & 3u) != 0) st = v & 3u;
          }
          const uint32_t incl = __ballot_sync(0xffffffffu, st == kIncl);
          const uint32_t ready = __ballot_sync(0xffffffffu, st != 0u);
          const int first = incl ? __ffs(incl) - 1 : 32;
          const uint32_t need = first == 32 ? 0xffffffffu : ((1u << first) - 1u);
          if ((ready & need) == need) { m = first; break; }
          if ((it & 15u) == 15u) {
            if (globaltimer_ns() - t_start > kWaitNs) break;
            __nanosleep(64);
          }
        }
        if (lane == 0) {
          if (m > 32) report(p.status, GDN_ERR_TIMEOUT, (uint32_t)bb, (uint32_t)hd, 2u);
          misc[4 + par] = (uint32_t)m;
        }
      }
      __syncthreads();
      const int m = (int)misc[4 + par];
      par ^= 1;
      if (m > 32) {   // timed out: carry on with what was composed so far
        hs = dF;
        break;
      }
      // compose the aggregate maps of j, j-1, ..., j-m+1 (nearest first)
      for (int l = 0; l < m; l += 4) {
        float4 x[4];
        float2 gj[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (l + e < m) {
            const float *ag = p.agg + (head_task0 + j - l - e) * kAggFloats;
            x[e] = __ldcg(reinterpret_cast<const float4 *>(ag + fidx));
            gj[e] = __ldcg(reinterpret_cast<const float2 *>(ag + kS * kD + s0));
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (l + e < m) {
            dF.x = fmaf(gF.x, x[e].x, dF.x);
            dF.y = fmaf(gF.y, x[e].y, dF.y);
            dF.z = fmaf(gF.x, x[e].z, dF.z);
            dF.w = fmaf(gF.y, x[e].w, dF.w);
            gF.x *= gj[e].x;
            gF.y *= gj[e].y;
          }
        }
      }
      if (m < 32) {
        const int jm = j - m;
        const float4 x = jm < 0 ? init_at()
                                : __ldcg(reinterpret_cast<const float4 *>(
                                      p.incl + (head_task0 + jm) * kInclFloats + fidx));
        hs.x = fmaf(gF.x, x.x, dF.x);
        hs.y = fmaf(gF.y, x.y, dF.y);
        hs.z = fmaf(gF.x, x.z, dF.z);
        hs.w = fmaf(gF.y, x.w, dF.w);
        done = true;
      } else {
        j -= 32;
      }
    }
  }
  GDN_DPROBE(5);
  // ---- publish the end state of this block ----
  {
    float4 he;
    he.x = fmaf(G.x, hs.x, agg.x);
    he.y = fmaf(G.y, hs.y, agg.y);
    he.z = fmaf(G.x, hs.z, agg.z);
    he.w = fmaf(G.y, hs.w, agg.w);
    if (valid) {
      __stcg(reinterpret_cast<float4 *>(p.incl + task * kInclFloats + fidx), he);
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
  const uint32_t next_ticket = misc[6];   // written by warp 2 before the barrier above
  const float gnext = load_gate(next_ticket);
  GDN_DPROBE(6);

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

  GDN_DPROBE(7);
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
      uint32_t b0[NP], b1[NP];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) { b0[pp] = pb0[pp][0]; b1[pp] = pb0[pp][1]; }
      mma_np<NP>(O[m][0], va[m], b0, b1);
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) { b0[pp] = pb1[pp][0]; b1[pp] = pb1[pp][1]; }
      mma_np<NP>(O[m][1], va[m], b0, b1);
    }
    // block epilogue: o <- (o + D_h v) * g_gate.  The V^T A fragments of m-tile
    // m sit at the positions of the O^T accumulators: register 2 ni + (q >> 1)
    // holds v at (d, i) = (16 m + g + 8 (q >> 1), 8 ni + 2 tq + (q & 1)).
    if (p.D_skip || p.out_gate) {
      const float Dh = p.D_skip ? __ldg(p.D_skip + hd) : 0.f;
      float gt[2][2];
#pragma unroll
      for (int ni = 0; ni < 2; ++ni)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) gt[ni][e2] = __shfl_sync(0xffffffffu, ogate, 8 * ni + 2 * tq + e2);
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int ni = 0; ni < 2; ++ni)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = 2 * ni + (q >> 1);
            float vv = (q & 1) ? bf16_hi(va[m][0][r]) : bf16_lo(va[m][0][r]);
            if constexpr (NP == 2) vv += (q & 1) ? bf16_hi(va[m][1][r]) : bf16_lo(va[m][1][r]);
            O[m][ni][q] = fmaf(Dh, vv, O[m][ni][q]) * gt[ni][q & 1];
          }
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
    __syncwarp();
    // coalesced 16-byte stores of the tile's rows that are inside the sequence
    if (valid) {
      constexpr int kChunks = kCT * kD * (int)sizeof(T) / 16;   // 16-byte pieces of the tile
      constexpr int kPerRow = kD * (int)sizeof(T) / 16;
      const unsigned char *src = sptr + (xch - sbase);
#pragma unroll
      for (int c = lane; c < kChunks; c += 32) {
        const int i = c / kPerRow;
        if (tok_w + i < p.seq_len) {
          const int64_t row = ((int64_t)bb * p.seq_len + tok_w + i) * p.num_heads + hd;
          *reinterpret_cast<uint4 *>(static_cast<unsigned char *>(p.o) + row * kD * sizeof(T) +
                                     (c % kPerRow) * 16) =
              *reinterpret_cast<const uint4 *>(src + c * 16);
        }
      }
    }
  }

  GDN_DPROBE(9);
#ifdef GDN_DIAG_PROBE
  if (tid == 0 && probe_id < 8192u) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_diag_probe[probe_id * 12u + 10] = smid;
  }
#endif
  ticket = next_ticket;
  gtok = gnext;
  phase ^= 1u;
  }   // persistent loop

  // ---- launch bookkeeping: the last CTA out resets the ticket and advances the epoch ----
  if (tid == 0) {
    const uint32_t d = atomicAdd(&p.ctr->done, 1u);
    if (d == gridDim.x - 1) {
      // every CTA of the launch has drawn its last ticket and read the epoch
      p.ctr->ticket = 0u;
      p.ctr->done = 0u;
      atomicAdd(&p.ctr->epoch, 1u);
    }
  }
}

namespace {

// [B][T][H][32] tensor of the storage type viewed as 4-D (32, H, T, B).
bool make_tmap4(CUtensorMap *m, const void *ptr, bool f32, int H, int T, int B, int box_t) {
  tc::EncodeTiledFn enc = tc::encode_fn();
  if (!enc) return false;
  const cuuint64_t e = f32 ? 4 : 2;
  const cuuint64_t dims[4] = {32, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {32 * e, 32 * e * H, 32 * e * H * (cuuint64_t)T};
  const cuuint32_t box[4] = {32, 1, (cuuint32_t)box_t, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
cudaError_t launch_t(const DiagParams &p, const void *v, const void *b, const void *c,
                     int64_t tasks, cudaStream_t stream) {
  using L = Lay<T>;
  const bool f32 = sizeof(T) == 4;
  CUtensorMap tv, tb, tc_;
  if (!make_tmap4(&tv, v, f32, p.num_heads, p.seq_len, p.batch, kSC) ||
      !make_tmap4(&tb, b, f32, p.num_heads, p.seq_len, p.batch, kSC) ||
      !make_tmap4(&tc_, c, f32, p.num_heads, p.seq_len, p.batch, kSC))
    return cudaErrorInvalidValue;
  // persistent CTAs: as many as fit on the device at once (cached per device)
  static int resident[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident[dev] == 0) {
    err = cudaFuncSetAttribute(gdn_diag_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               L::ALLOC);
    if (err != cudaSuccess) return err;
    int per_sm = 0, sms = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gdn_diag_kernel<T>, kThreads,
                                                        L::ALLOC);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    resident[dev] = per_sm > 0 && sms > 0 ? per_sm * sms : 1;
  }
  const int64_t grid = tasks < resident[dev] ? tasks : resident[dev];
  gdn_diag_kernel<T><<<(unsigned)grid, kThreads, L::ALLOC, stream>>>(p, tv, tb, tc_);
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

#ifdef GDN_DIAG_PROBE
extern "C" int gdn_diag_probe_read(unsigned long long *host) {
  return (int)cudaMemcpyFromSymbol(host, gdn::diag::g_diag_probe, sizeof(gdn::diag::g_diag_probe));
}
#endif

extern "C" size_t gdn_diag_workspace_size(int32_t batch, int32_t seq_len, int32_t num_heads,
                                          int32_t d_state, int32_t head_dim) {
  using namespace gdn::diag;
  if (batch <= 0 || seq_len <= 0 || num_heads <= 0 || d_state <= 0 || head_dim <= 0) return 0;
  const int64_t nblk = ((int64_t)seq_len + kSC - 1) / kSC;
  return workspace_layout((int64_t)batch * num_heads * nblk).total;
}

extern "C" gdn_status gdn_diag_fwd(const void *v, const void *b, const void *c, const float *g,
                                   const float *A_log, const float *D_skip,
                                   const float *out_gate, const float *initial_state, void *o,
                                   float *final_state, int32_t batch, int32_t seq_len,
                                   int32_t num_heads, int32_t d_state, int32_t head_dim,
                                   gdn_dtype dtype, uint32_t flags, void *workspace,
                                   size_t workspace_bytes, void *stream) {
  using namespace gdn;
  using namespace gdn::diag;
  if (batch <= 0 || seq_len <= 0 || num_heads <= 0 || d_state <= 0 || head_dim <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)GDN_GATE_SIGMOID) return GDN_ERR_INVALID_ARG;
  if (d_state != kS || head_dim != kD) return GDN_ERR_UNSUPPORTED;
  const int64_t nblk = ((int64_t)seq_len + kSC - 1) / kSC;
  const int64_t tasks = (int64_t)batch * num_heads * nblk;
  if (tasks > 0x7fffffffLL || (int64_t)batch * num_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (!v || !b || !c || !g || !A_log || !o) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {v, b, c, g, A_log, D_skip, out_gate, initial_state, o, final_state};
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
  const size_t b_D = (size_t)num_heads * 4;
  const Range inputs[] = {{v, b_v}, {b, b_bc}, {c, b_bc}, {g, b_g}, {A_log, b_A},
                          {D_skip, b_D}, {out_gate, b_g}, {workspace, workspace_bytes}};
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
  p.g = g; p.A_log = A_log; p.h0 = initial_state; p.hN = final_state; p.o = o;
  p.D_skip = D_skip; p.out_gate = out_gate; p.opts = flags;
  p.status = reinterpret_cast<DeviceStatus *>(ws);
  p.ctr = reinterpret_cast<Counters *>(ws + kCountersOff);
  p.flags = reinterpret_cast<uint32_t *>(ws + wl.flags);
  p.agg = reinterpret_cast<float *>(ws + wl.agg);
  p.incl = reinterpret_cast<float *>(ws + wl.incl);
  p.batch = batch; p.seq_len = seq_len; p.num_heads = num_heads; p.nblk = (int32_t)nblk;
  const cudaError_t err =
      dtype == GDN_F32 ? launch_t<float>(p, v, b, c, tasks, (cudaStream_t)stream)
                       : launch_t<__nv_bfloat16>(p, v, b, c, tasks, (cudaStream_t)stream);
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
