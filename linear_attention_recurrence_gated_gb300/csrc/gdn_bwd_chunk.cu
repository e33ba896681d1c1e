// Chunked backward of the gated delta rule for bf16 storage (head_dim_k and
// head_dim_v in {32, 64, 128}), on warp-level bf16 tensor-core products with
// fp32 accumulation.  The pages' kernel ships a recompute-style backward
// ("Optimization Quartet", Triton GDN kernel section 3.4); this one works in
// the chunked WY form of the forward (chunk size 64, "v1.0 Architecture &
// Design Spec" section 2.3), so that everything but two short state chains is
// parallel over chunks.
//
// Per chunk, with H the state entering it (dk x dv, H = S^T), G the chunk-local
// prefix sum of the log-gates, gamma = exp(G), Gamma_ij = exp(G_i - G_j),
// dec_i = exp(G_C - G_i), K~ = diag(dec) K and T = (I + A)^-1:
//   A  = strictly_lower(diag(beta) K K^T (.) Gamma)     P = (Q K^T (.) Gamma)_{i>=j}
//   W  = T diag(beta gamma) K      U~ = T diag(beta) V      U = U~ - W H
//   O  = diag(gamma) Q H + P U     H' = gamma_C H + K~^T U
// Its reverse, with dH' the gradient of the state leaving the chunk:
//   dU = P^T dO + K~ dH'           dH = gamma_C dH' + Q^T diag(gamma) dO - W^T dU
//   dP = (dO U^T)_{i>=j}           dQ = diag(gamma) dO H^T + (dP (.) Gamma) K
//   dK~ = U dH'^T                  dW = -dU H^T
//   dR_W = T^T dW,  dR_U = T^T dU  (R_W = diag(beta gamma) K, R_U = diag(beta) V)
//   dV = diag(beta) dR_U           dA = -(dR_W W^T + dR_U U~^T), strictly lower
//   dK = diag(dec) dK~ + diag(beta gamma) dR_W + S K + (dP (.) Gamma)^T Q,
//        S = diag(beta) D + D^T diag(beta),  D = dA (.) Gamma
// and the gate gradient collects, per token, the terms through gamma, Gamma,
// dec and gamma_C, then sums them over later tokens of the chunk (G is a
// prefix sum).
//
// Four kernels:
//   prep   (per chunk and head)  A, T (fp32 substitution), W, U~, K~, and the
//          state-free products dO^T P and dO^T diag(gamma) Q of the reverse chain;
//   chain  (per sequence and head, forward)  H at every chunk start;
//   chain  (per sequence and head, reverse)  dH' at every chunk end and the
//          gradient of the initial state;
//   grad   (per chunk and head)  dq, dk, dv, dg, dbeta of the chunk.
// dU and dW enter T^T dU and T^T dW as bf16 operands, and what rounding them
// left out is added back on the diagonal of T (exactly 1), so that dR_U and
// dR_W, over which dbeta and dv sum, keep it.
// The chains keep their state in the MMA accumulator registers of the warps
// (16 value columns per warp, transposed, so that an accumulator is directly
// the A operand of the next product).  No kernel waits on another CTA.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;          // tokens per chunk
constexpr int kThreads = 128;   // 4 warps; warp w owns rows 16w..16w+15 of a chunk product
constexpr int kLdC = kC + 8;    // bf16 row stride of C x C tiles

// ---- fragment loads for mma.m16n8k16 (bf16 operands from shared memory) ----
// A(16 x 16) of a matrix stored row-major as (m, k)
__device__ __forceinline__ void lda_row(const bf16 *base, int ld, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31;
  const bf16 *p = base + (m0 + (l & 7) + ((l >> 3) & 1) * 8) * ld + k0 + (l >> 4) * 8;
  ldsm_x4(smem_u32(p), a[0], a[1], a[2], a[3]);
}
// A(16 x 16) of a matrix stored as (k, m): element (m, k) at base[k * ld + m]
__device__ __forceinline__ void lda_tr(const bf16 *base, int ld, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31, i = l >> 3;
  const bf16 *p = base + (k0 + (i >> 1) * 8 + (l & 7)) * ld + m0 + (i & 1) * 8;
  ldsm_x4_t(smem_u32(p), a[0], a[1], a[2], a[3]);
}
// B(16 x 8) for the n-tiles n0 and n0 + 8 of a matrix stored row-major as (k, n)
__device__ __forceinline__ void ldb_kn(const bf16 *base, int ld, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, i = l >> 3;
  const bf16 *p = base + (k0 + (i & 1) * 8 + (l & 7)) * ld + n0 + (i >> 1) * 8;
  ldsm_x4_t(smem_u32(p), b[0], b[1], b[2], b[3]);
}
// the same for a matrix stored as (n, k): element (k, n) at base[n * ld + k]
__device__ __forceinline__ void ldb_nk(const bf16 *base, int ld, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, i = l >> 3;
  const bf16 *p = base + (n0 + (i >> 1) * 8 + (l & 7)) * ld + k0 + (i & 1) * 8;
  ldsm_x4(smem_u32(p), b[0], b[1], b[2], b[3]);
}

// acc(16 x 8 NT) += A(16 x K) B(K x 8 NT); A rows m0.., B columns n0..
template <int NT, bool A_TR, bool B_NK>
__device__ __forceinline__ void wmma(float (&acc)[NT][4], const bf16 *A, int lda, int m0,
                                     const bf16 *B, int ldb, int n0, int K) {
  static_assert(NT % 2 == 0, "n-tiles come in pairs");
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a[4];
    if (A_TR) lda_tr(A, lda, m0, k0, a);
    else lda_row(A, lda, m0, k0, a);
#pragma unroll
    for (int p = 0; p < NT / 2; ++p) {
      uint32_t b[4];
      if (B_NK) ldb_nk(B, ldb, k0, n0 + 16 * p, b);
      else ldb_kn(B, ldb, k0, n0 + 16 * p, b);
      mma_bf16(acc[2 * p], a[0], a[1], a[2], a[3], b[0], b[1]);
      mma_bf16(acc[2 * p + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
}

// Visit the accumulator elements: f(row, col, value&) with row in m0.., col in n0..
template <int NT, typename F>
__device__ __forceinline__ void each(float (&acc)[NT][4], int m0, int n0, F &&f) {
  const int l = threadIdx.x & 31, r = m0 + (l >> 2), c = n0 + 2 * (l & 3);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    f(r, c + 8 * t, acc[t][0]);
    f(r, c + 8 * t + 1, acc[t][1]);
    f(r + 8, c + 8 * t, acc[t][2]);
    f(r + 8, c + 8 * t + 1, acc[t][3]);
  }
}

// Sum of a per-row partial over the 4 lanes that share a row of the fragment.
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

__device__ __forceinline__ void cp16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// rows x (cols elements of `bytes_per` bytes) from a dense global matrix into a padded tile
template <int ROWS, int ROW_BYTES, int NTH = kThreads>
__device__ __forceinline__ void cp_rows(void *dst, int ld_bytes, const void *src,
                                        size_t src_stride = ROW_BYTES) {
  constexpr int V = ROW_BYTES / 16;
  for (int idx = threadIdx.x; idx < ROWS * V; idx += NTH) {
    const int r = idx / V, c = (idx % V) * 16;
    cp16(static_cast<uint8_t *>(dst) + r * ld_bytes + c,
         static_cast<const uint8_t *>(src) + (size_t)r * src_stride + c);
  }
}

// rows [0, ROWS) of a bf16 matrix with COLS columns (global row stride gstride
// elements) into a padded shared tile with cp.async; rows >= valid are zero.
template <int ROWS, int COLS, int NTH = kThreads>
__device__ __forceinline__ void cp_tile(bf16 *dst, int ld, const bf16 *src, size_t gstride,
                                        int valid) {
  constexpr int V = COLS / 8;  // 16-byte pieces per row
  for (int idx = threadIdx.x; idx < ROWS * V; idx += NTH) {
    const int r = idx / V, c = (idx % V) * 8;
    const bool ok = r < valid;
    const bf16 *g = src + (ok ? (size_t)r * gstride + c : 0);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + r * ld + c)),
                 "l"(g), "r"(ok ? 16 : 0)
                 : "memory");
  }
}

// Chunk gates for tokens i < 64 (threads 0..63): G (inclusive prefix sum of g in
// fp32, the same order in every kernel), G log2(e), gamma, dec and beta.  Tokens
// past the chunk's end have g = 0 and beta = 0.  Needs a __syncthreads() after.
__device__ __forceinline__ void chunk_gates(const float *g, const bf16 *beta, int64_t tok0,
                                            int H, int h, int valid, float *sG, float *sGl,
                                            float *sGam, float *sDec, float *sBeta,
                                            float *sTmp) {
  const int i = threadIdx.x, lane = i & 31;
  float x = 0.f, b = 0.f;
  if (i < kC && i < valid) {
    const size_t off = (size_t)(tok0 + i) * H + h;
    x = g[off];
    b = __bfloat162float(beta[off]);
  }
  if (i < kC) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (i == 31) sTmp[0] = x;
  }
  __syncthreads();
  if (i < kC) {
    if (i >= 32) x += sTmp[0];
    sG[i] = x;
    sGl[i] = x * 1.4426950408889634f;
    sBeta[i] = b;
    sGam[i] = expf(x);
  }
  __syncthreads();
  if (i < kC) sDec[i] = expf(sG[kC - 1] - sG[i]);
}

// The sequence and chunk of a chunk slot (see ckpt_first_slot); false when the
// slot holds no chunk or the sequence bounds are bad.
__device__ __forceinline__ bool slot_chunk(const FwdParams &p, int64_t slot, int h, int &n,
                                           int64_t &tok0, int &valid) {
  int64_t start, len, c;
  if (p.cu == nullptr) {
    const int64_t nck = (p.seq_len + kC - 1) / kC;
    n = (int)(slot / nck);
    c = slot - (int64_t)n * nck;
    if (n >= p.num_seqs) return false;
  } else {
    int lo = 0, hi = p.num_seqs - 1;   // last n with cu[n] / 64 + n <= slot
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)p.cu[mid] / kC + mid <= slot) lo = mid;
      else hi = mid - 1;
    }
    n = lo;
    c = slot - ((int64_t)p.cu[n] / kC + n);
    if (c < 0) return false;
  }
  if (!sequence_bounds(p, n, h, start, len)) return false;
  if (c * kC >= len) return false;
  tok0 = start + c * kC;
  valid = (int)(len - c * kC < kC ? len - c * kC : kC);
  return true;
}

// Per (chunk slot, head) records of the workspace.
template <int DK, int DV>
struct ChunkWs {
  bf16 *W, *Ut, *T, *Kt;     // [64][DK], [64][DV], [64][64], [64][DK]
  bf16 *Hb, *dHb;            // [DK][DV]: state entering / gradient leaving the chunk
  float *X1t, *X2t;          // [DV][64] = dO^T P,  [DV][DK] = dO^T diag(gamma) Q
  float *gC;                 // [4]: gamma_C, the gradient of gamma_C, 0, 0
  static constexpr size_t kW = 64 * DK, kUt = 64 * DV, kT = 64 * 64, kKt = 64 * DK;
  static constexpr size_t kX1 = (size_t)DV * 64, kX2 = (size_t)DV * DK, kH = (size_t)DK * DV;
  static size_t bytes(int64_t units) {
    return (size_t)units * (2 * (kW + kUt + kT + kKt + 2 * kH) + 4 * (kX1 + kX2 + 4));
  }
  __host__ __device__ void carve(void *base, int64_t units) {
    uint8_t *b = static_cast<uint8_t *>(base);
    W = reinterpret_cast<bf16 *>(b);   b += units * kW * 2;
    Ut = reinterpret_cast<bf16 *>(b);  b += units * kUt * 2;
    T = reinterpret_cast<bf16 *>(b);   b += units * kT * 2;
    Kt = reinterpret_cast<bf16 *>(b);  b += units * kKt * 2;
    Hb = reinterpret_cast<bf16 *>(b);  b += units * kH * 2;
    dHb = reinterpret_cast<bf16 *>(b); b += units * kH * 2;
    X1t = reinterpret_cast<float *>(b); b += units * kX1 * 4;
    X2t = reinterpret_cast<float *>(b); b += units * kX2 * 4;
    gC = reinterpret_cast<float *>(b);
  }
};

struct ChunkBwdParams {
  FwdParams f;
  const bf16 *dO;
  const float *dHN;
  float *dq, *dk, *dv, *dg, *dbeta, *dh0;
  void *ws;            // ChunkWs arrays
  int64_t slots;       // chunk slots per head
};

// Pairs of adjacent accumulator elements: f(row, col, x0, x1) with col even.
template <int NT, typename F>
__device__ __forceinline__ void each2(float (&acc)[NT][4], int m0, int n0, F &&f) {
  const int l = threadIdx.x & 31, r = m0 + (l >> 2), c = n0 + 2 * (l & 3);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    f(r, c + 8 * t, acc[t][0], acc[t][1]);
    f(r + 8, c + 8 * t, acc[t][2], acc[t][3]);
  }
}

__device__ __forceinline__ float bf(const bf16 &x) { return __bfloat162float(x); }
// Gamma_ij = exp(G_i - G_j) <= 1 is taken as 2^(G_i log2 e - G_j log2 e) with the
// hardware exp2 (decays below 2^-126 flush to zero).
__device__ __forceinline__ float rbf(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ void st_bf2(bf16 *p, float a, float b) {
  *reinterpret_cast<uint32_t *>(p) = pack_bf16(a, b);
}

// ---------------------------------------------------------------- prep ----
// 8 warps: warp w owns rows 16 (w % 4).. of a chunk product and half of its columns.
constexpr int kPrepThreads = 256;

template <int DK, int DV>
struct PrepSmem {
  static constexpr int LK = DK + 8, LV = DV + 8, LA = 68, LB = 17;
  bf16 q[64 * LK], k[64 * LK], rw[64 * LK];   // rw: diag(beta gamma) K, then diag(gamma) Q
  bf16 v[64 * LV], o[64 * LV], ru[64 * LV];
  bf16 P[64 * kLdC], T[64 * kLdC];
  float A[64 * LA];            // A; its diagonal 16 x 16 blocks become T's
  float Toff[6][16 * LB];      // T's blocks below the diagonal, (i, j) at i (i - 1) / 2 + j
  float X[3][16 * LB];         // scratch of the block substitution
  float G[64], Gl[64], gam[64], dec[64], beta[64], tmp[4];
};

// T = (I + A)^-1 of a strictly lower A (fp32), in 16 x 16 blocks: the diagonal
// blocks by forward substitution (in place over A's), then the blocks below by
// diagonals, T_ij = -T_ii sum_{j <= m < i} A_im T_mj.
template <int DK, int DV>
__device__ __forceinline__ void block_inverse(PrepSmem<DK, DV> &s) {
  constexpr int LA = PrepSmem<DK, DV>::LA, LB = PrepSmem<DK, DV>::LB;
  const int tid = threadIdx.x, b = tid >> 4, j = tid & 15;
  float t[16];
  if (tid < kC) {
    const float *Ab = s.A + 16 * b * LA + 16 * b;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a = 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) a = fmaf(Ab[i * LA + m], t[m], a);
      t[i] = i < j ? 0.f : (i == j ? 1.f : -a);
    }
  }
  __syncthreads();   // every column has read its A block
  if (tid < kC) {
    float *Tb = s.A + 16 * b * LA + 16 * b;
#pragma unroll
    for (int i = 0; i < 16; ++i) Tb[i * LA + j] = t[i];
  }
  __syncthreads();
  // Each thread forms four rows (4rq .. 4rq + 3) of one column c of a block, so
  // that the column loads serve four rows.
  for (int L = 1; L < 4; ++L) {
    const int nb = 4 - L;   // blocks (j + L, j), j = 0..nb-1
    for (int e = tid; e < nb * 64; e += kPrepThreads) {
      const int j = e >> 6, rq = (e >> 4) & 3, c = e & 15, i = j + L;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kb = j; kb < i; ++kb) {   // T_{kb, j}: the diagonal block (in A) or one below it
        const bool diag = kb == j;
        const float *Tc = diag ? s.A + 16 * j * LA + 16 * j + c : s.Toff[kb * (kb - 1) / 2 + j] + c;
        const int ld = diag ? LA : LB;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const float t0 = Tc[(4 * m4) * ld], t1 = Tc[(4 * m4 + 1) * ld];
          const float t2 = Tc[(4 * m4 + 2) * ld], t3 = Tc[(4 * m4 + 3) * ld];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const float4 a = *reinterpret_cast<const float4 *>(
                s.A + (16 * i + 4 * rq + rr) * LA + 16 * kb + 4 * m4);
            x[rr] = fmaf(a.x, t0, fmaf(a.y, t1, fmaf(a.z, t2, fmaf(a.w, t3, x[rr]))));
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) s.X[j][(4 * rq + rr) * LB + c] = x[rr];
    }
    __syncthreads();
    for (int e = tid; e < nb * 64; e += kPrepThreads) {
      const int j = e >> 6, rq = (e >> 4) & 3, c = e & 15, i = j + L;
      const float *Xc = s.X[j] + c;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int m4 = 0; m4 < 4; ++m4) {
        const float t0 = Xc[(4 * m4) * LB], t1 = Xc[(4 * m4 + 1) * LB];
        const float t2 = Xc[(4 * m4 + 2) * LB], t3 = Xc[(4 * m4 + 3) * LB];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {   // T_ii, lower triangular
          const float4 a = *reinterpret_cast<const float4 *>(
              s.A + (16 * i + 4 * rq + rr) * LA + 16 * i + 4 * m4);
          x[rr] = fmaf(a.x, t0, fmaf(a.y, t1, fmaf(a.z, t2, fmaf(a.w, t3, x[rr]))));
        }
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) s.Toff[i * (i - 1) / 2 + j][(4 * rq + rr) * LB + c] = -x[rr];
    }
    __syncthreads();
  }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kPrepThreads) gdn_bwdc_prep_kernel(const ChunkBwdParams P) {
  using S = PrepSmem<DK, DV>;
  using WS = ChunkWs<DK, DV>;
  constexpr int LK = S::LK, LV = S::LV, LA = S::LA, LB = S::LB;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  S &s = *reinterpret_cast<S *>(smem_raw);
  const FwdParams &p = P.f;
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  int n, valid;
  int64_t tok0;
  if (!slot_chunk(p, slot, h, n, tok0, valid)) return;
  const int H = p.num_heads, tid = threadIdx.x, warp = tid >> 5, m0 = 16 * (warp & 3);
  const int half = warp >> 2;   // column half of the products
  const size_t unit = (size_t)slot * H + h;
  WS ws;
  ws.carve(P.ws, P.slots * H);

  const size_t rq = ((size_t)tok0 * H + h) * DK, rv = ((size_t)tok0 * H + h) * DV;
  cp_tile<64, DK, kPrepThreads>(s.q, LK, static_cast<const bf16 *>(p.q) + rq, (size_t)H * DK, valid);
  cp_tile<64, DK, kPrepThreads>(s.k, LK, static_cast<const bf16 *>(p.k) + rq, (size_t)H * DK, valid);
  cp_tile<64, DV, kPrepThreads>(s.v, LV, static_cast<const bf16 *>(p.v) + rv, (size_t)H * DV, valid);
  cp_tile<64, DV, kPrepThreads>(s.o, LV, P.dO + rv, (size_t)H * DV, valid);
  cp_commit();
  chunk_gates(p.g, static_cast<const bf16 *>(p.beta), tok0, H, h, valid, s.G, s.Gl, s.gam,
              s.dec, s.beta, s.tmp);
  cp_wait<0>();
  __syncthreads();

  // scaled operands (bf16): beta gamma k, beta v; K~ = dec k to the workspace
  for (int idx = tid; idx < 64 * DK / 2; idx += kPrepThreads) {
    const int i = idx / (DK / 2), d = 2 * (idx % (DK / 2));
    const float k0 = bf(s.k[i * LK + d]), k1 = bf(s.k[i * LK + d + 1]);
    const float bg = s.beta[i] * s.gam[i], de = s.dec[i];
    st_bf2(&s.rw[i * LK + d], bg * k0, bg * k1);
    st_bf2(ws.Kt + unit * WS::kKt + i * DK + d, de * k0, de * k1);
  }
  for (int idx = tid; idx < 64 * DV / 2; idx += kPrepThreads) {
    const int i = idx / (DV / 2), c = 2 * (idx % (DV / 2));
    const float b = s.beta[i];
    st_bf2(&s.ru[i * LV + c], b * bf(s.v[i * LV + c]), b * bf(s.v[i * LV + c + 1]));
  }
  if (tid == 0)   // gamma_C; the reverse chain adds the gradient of gamma_C into slot 1
    *reinterpret_cast<float4 *>(ws.gC + unit * 4) = make_float4(s.gam[kC - 1], 0.f, 0.f, 0.f);

  // A = strictly_lower(diag(beta) K K^T (.) Gamma) in fp32; P = (Q K^T (.) Gamma)_{i>=j}
  {
    float acc[4][4];
    zero(acc);
    wmma<4, false, true>(acc, s.k, LK, m0, s.k, LK, 32 * half, DK);
    each(acc, m0, 32 * half, [&](int i, int j, float &x) {
      s.A[i * LA + j] = i > j ? s.beta[i] * x * ex2(s.Gl[i] - s.Gl[j]) : 0.f;
    });
    zero(acc);
    wmma<4, false, true>(acc, s.q, LK, m0, s.k, LK, 32 * half, DK);
    each2(acc, m0, 32 * half, [&](int i, int j, float &x0, float &x1) {
      const float p0 = i >= j ? x0 * ex2(s.Gl[i] - s.Gl[j]) : 0.f;
      const float p1 = i >= j + 1 ? x1 * ex2(s.Gl[i] - s.Gl[j + 1]) : 0.f;
      st_bf2(&s.P[i * kLdC + j], p0, p1);
    });
  }
  __syncthreads();
  block_inverse(s);
  // T to bf16 (shared tile and workspace)
  for (int idx = tid; idx < 64 * 32; idx += kPrepThreads) {
    const int i = idx >> 5, j = 2 * (idx & 31), bi = i >> 4, bj = j >> 4;
    float t0 = 0.f, t1 = 0.f;
    if (bi == bj) {
      t0 = s.A[i * LA + j];
      t1 = s.A[i * LA + j + 1];
    } else if (bi > bj) {
      const float *Tb = s.Toff[bi * (bi - 1) / 2 + bj] + (i & 15) * LB + (j & 15);
      t0 = Tb[0];
      t1 = Tb[1];
    }
    st_bf2(&s.T[i * kLdC + j], t0, t1);
    st_bf2(ws.T + unit * WS::kT + i * kC + j, t0, t1);
  }
  __syncthreads();

  // W = T diag(beta gamma) K, U~ = T diag(beta) V (bf16 to the workspace)
  {
    float acc[DK / 16][4];
    zero(acc);
    wmma<DK / 16, false, false>(acc, s.T, kLdC, m0, s.rw, LK, DK / 2 * half, kC);
    bf16 *W = ws.W + unit * WS::kW;
    each2(acc, m0, DK / 2 * half, [&](int i, int d, float &x0, float &x1) { st_bf2(W + i * DK + d, x0, x1); });
  }
  {
    float acc[DV / 16][4];
    zero(acc);
    wmma<DV / 16, false, false>(acc, s.T, kLdC, m0, s.ru, LV, DV / 2 * half, kC);
    bf16 *Ut = ws.Ut + unit * WS::kUt;
    each2(acc, m0, DV / 2 * half, [&](int i, int c, float &x0, float &x1) { st_bf2(Ut + i * DV + c, x0, x1); });
  }
  // the state-free products of the reverse chain: dO^T P and dO^T diag(gamma) Q (fp32)
  __syncthreads();   // W is done with diag(beta gamma) K
  for (int idx = tid; idx < 64 * DK / 2; idx += kPrepThreads) {
    const int i = idx / (DK / 2), d = 2 * (idx % (DK / 2));
    const float ga = s.gam[i];
    st_bf2(&s.rw[i * LK + d], ga * bf(s.q[i * LK + d]), ga * bf(s.q[i * LK + d + 1]));
  }
  __syncthreads();
  for (int mt = warp & 3; mt < DV / 16; mt += 4) {
    float acc[4][4];
    zero(acc);
    wmma<4, true, false>(acc, s.o, LV, 16 * mt, s.P, kLdC, 32 * half, kC);
    float *X1 = ws.X1t + unit * WS::kX1;
    each2(acc, 16 * mt, 32 * half, [&](int c, int j, float &x0, float &x1) {
      *reinterpret_cast<float2 *>(X1 + c * kC + j) = make_float2(x0, x1);
    });
    float acc2[DK / 16][4];
    zero(acc2);
    wmma<DK / 16, true, false>(acc2, s.o, LV, 16 * mt, s.rw, LK, DK / 2 * half, kC);
    float *X2 = ws.X2t + unit * WS::kX2;
    each2(acc2, 16 * mt, DK / 2 * half, [&](int c, int d, float &x0, float &x1) {
      *reinterpret_cast<float2 *>(X2 + c * DK + d) = make_float2(x0, x1);
    });
  }
}

// --------------------------------------------------------------- chains ----
// A chain CTA owns a slice of SW = min(DV, 64) value columns (4 warps x 16).
template <int DK, int DV, bool REV>
struct ChainSmem {
  static constexpr int SW = DV < 64 ? DV : 64;
  static constexpr int LK = DK + 8, LS = SW + 8, LX1 = kC + 4, LX2 = DK + 4;
  bf16 W[2][64 * LK], Kt[2][64 * LK];
  bf16 Ut[REV ? 1 : 2][REV ? 8 : 64 * LS];    // the slice's columns of U~
  float X1[REV ? 2 : 1][REV ? SW * LX1 : 4];  // the slice's rows of dO^T P
  float X2[REV ? 2 : 1][REV ? SW * LX2 : 4];  // ... and of dO^T diag(gamma) Q
  bf16 Hb[REV ? 2 : 1][REV ? DK * LS : 8];    // the state entering the chunk (slice)
  float gC[2][4];
};

// A operand (16 x 16, k-step kk) from a 16 x K fp32 accumulator, times `sc`.
template <int NT>
__device__ __forceinline__ void acc_to_a(const float (&acc)[NT][4], int kk, float sc,
                                         uint32_t (&a)[4]) {
  a[0] = pack_bf16(sc * acc[2 * kk][0], sc * acc[2 * kk][1]);
  a[1] = pack_bf16(sc * acc[2 * kk][2], sc * acc[2 * kk][3]);
  a[2] = pack_bf16(sc * acc[2 * kk + 1][0], sc * acc[2 * kk + 1][1]);
  a[3] = pack_bf16(sc * acc[2 * kk + 1][2], sc * acc[2 * kk + 1][3]);
}
// acc(16 x 8 NT) += (sc * X)(16 x 8 KT) B, X an accumulator, B in shared memory
template <int NT, int KT, bool B_NK>
__device__ __forceinline__ void wmma_ra(float (&acc)[NT][4], const float (&X)[KT][4], float sc,
                                        const bf16 *B, int ldb) {
#pragma unroll
  for (int kk = 0; kk < KT / 2; ++kk) {
    uint32_t a[4];
    acc_to_a(X, kk, sc, a);
#pragma unroll
    for (int p = 0; p < NT / 2; ++p) {
      uint32_t b[4];
      if (B_NK) ldb_nk(B, ldb, 16 * kk, 16 * p, b);
      else ldb_kn(B, ldb, 16 * kk, 16 * p, b);
      mma_bf16(acc[2 * p], a[0], a[1], a[2], a[3], b[0], b[1]);
      mma_bf16(acc[2 * p + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
    }
  }
}

// Forward (REV = false): H at every chunk start, from the initial state.
//   U^T = U~^T - H^T W^T,   H'^T = gamma_C H^T + U^T K~
// Reverse (REV = true): dH' at every chunk end, from d_final_state, and the
// gradient of the initial state.
//   dU^T = (dO^T P) + dH'^T K~^T,   dH^T = gamma_C dH'^T + (dO^T diag(gamma) Q) - dU^T W
// A CTA takes one slice of up to 64 value columns; its warp w keeps the
// transposed state of 16 of them (16 x DK) in its accumulators.  The next
// chunk's operands are staged while it works.
template <int DK, int DV, bool REV>
__global__ void __launch_bounds__(kThreads) gdn_bwdc_chain_kernel(const ChunkBwdParams P) {
  using S = ChainSmem<DK, DV, REV>;
  using WS = ChunkWs<DK, DV>;
  constexpr int LK = S::LK, LS = S::LS, SW = S::SW, LX1 = S::LX1, LX2 = S::LX2;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  S &s = *reinterpret_cast<S *>(smem_raw);
  const FwdParams &p = P.f;
  const int h = blockIdx.x, n = blockIdx.y, cs = SW * blockIdx.z;  // first column of the slice
  int64_t start, len;
  if (!sequence_bounds(p, n, h, start, len)) return;
  const int H = p.num_heads, warp = threadIdx.x >> 5;
  const int c0 = cs + 16 * warp;   // this warp's value columns c0..c0+15
  const bool active = 16 * warp < SW;
  const int64_t ck0 = ckpt_first_slot(n, start, p.seq_len, p.cu != nullptr);
  const int nck = (int)((len + kC - 1) / kC);
  WS ws;
  ws.carve(P.ws, P.slots * H);

  auto stage = [&](int buf, int cc) {
    const size_t unit = (size_t)(ck0 + cc) * H + h;
    cp_rows<64, DK * 2>(s.W[buf], LK * 2, ws.W + unit * WS::kW);
    cp_rows<64, DK * 2>(s.Kt[buf], LK * 2, ws.Kt + unit * WS::kKt);
    if (REV) {
      cp_rows<SW, kC * 4>(s.X1[buf], LX1 * 4, ws.X1t + unit * WS::kX1 + (size_t)cs * kC);
      cp_rows<SW, DK * 4>(s.X2[buf], LX2 * 4, ws.X2t + unit * WS::kX2 + (size_t)cs * DK);
      cp_rows<DK, SW * 2>(s.Hb[buf], LS * 2, ws.Hb + unit * WS::kH + cs, (size_t)DV * 2);
    } else {
      cp_rows<64, SW * 2>(s.Ut[buf], LS * 2, ws.Ut + unit * WS::kUt + cs, (size_t)DV * 2);
    }
    if (threadIdx.x == 0) cp16(s.gC[buf], ws.gC + unit * 4);
    cp_commit();
  };

  // state^T: row = value column c0 + (lane/4) (+8), column = key row d
  float st[DK / 8][4];
  const size_t sbase = ((size_t)n * H + h) * DK * DV;
  {
    const float *src = REV ? P.dHN : p.s0;
    each(st, c0, 0, [&](int c, int d, float &x) {
      x = (src != nullptr && active) ? src[sbase + (size_t)d * DV + c] : 0.f;
    });
  }
  stage(0, REV ? nck - 1 : 0);
  for (int it = 0; it < nck; ++it) {
    const int cc = REV ? nck - 1 - it : it, buf = it & 1;
    if (it + 1 < nck) {
      stage(buf ^ 1, REV ? cc - 1 : cc + 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const size_t unit = (size_t)(ck0 + cc) * H + h;
    bf16 *out = (REV ? ws.dHb : ws.Hb) + unit * WS::kH;
    const float gC = s.gC[buf][0];
    if (active) {
      float dot = 0.f;   // reverse: <dH', H>, the gradient of gamma_C
      each2(st, c0, 0, [&](int c, int d, float &x0, float &x1) {
        out[(size_t)d * DV + c] = __float2bfloat16_rn(x0);
        out[(size_t)(d + 1) * DV + c] = __float2bfloat16_rn(x1);
        if (REV)
          dot += x0 * bf(s.Hb[buf][d * LS + c - cs]) + x1 * bf(s.Hb[buf][(d + 1) * LS + c - cs]);
      });
      if (REV) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if ((threadIdx.x & 31) == 0) atomicAdd(ws.gC + unit * 4 + 1, dot);
      }
      float u[8][4];   // 16 value columns x 64 tokens
      if (!REV) {
        zero(u);
        wmma_ra<8, DK / 8, true>(u, st, 1.f, s.W[buf], LK);   // H^T W^T
        each(u, c0, 0, [&](int c, int i, float &x) { x = bf(s.Ut[buf][i * LS + c - cs]) - x; });
#pragma unroll
        for (int t = 0; t < DK / 8; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) st[t][e] *= gC;
        wmma_ra<DK / 8, 8, false>(st, u, 1.f, s.Kt[buf], LK);  // + U^T K~
      } else {
        each(u, c0, 0, [&](int c, int i, float &x) { x = s.X1[buf][(c - cs) * LX1 + i]; });
        wmma_ra<8, DK / 8, true>(u, st, 1.f, s.Kt[buf], LK);   // + dH'^T K~^T
        each(st, c0, 0, [&](int c, int d, float &x) { x = gC * x + s.X2[buf][(c - cs) * LX2 + d]; });
        wmma_ra<DK / 8, 8, false>(st, u, -1.f, s.W[buf], LK);  // - dU^T W
      }
    }
    __syncthreads();   // buffer `buf` is restaged two iterations on
  }
  if (REV && P.dh0 != nullptr && active)
    each(st, c0, 0, [&](int c, int d, float &x) { P.dh0[sbase + (size_t)d * DV + c] = x; });
}

// ----------------------------------------------------------------- grad ----
// NS = 1: 4 warps, warp w owns rows 16w.. of every chunk product.  NS = 2 (a
// head dim of 128): 8 warps, warp w owns rows 16 (w % 4).. and half of the
// columns, so that the per-warp accumulators stay within the registers.
template <int DK, int DV>
struct GradSmem {
  static constexpr int LK = DK + 8, LV = DV + 8, LO = LV > kLdC ? LV : kLdC;
  static constexpr int R1 = (DK * LV > 64 * LK ? DK * LV : 64 * LK);  // H, then dR_W
  static constexpr int R2 = (DK * LV > 64 * LV ? DK * LV : 64 * LV);  // dH', then dR_U
  bf16 q[64 * LK], k[64 * LK], W[64 * LK], KtDW[64 * LK];  // K~, then dW
  bf16 UU[64 * LV];    // U~, U over it, then U~ again
  bf16 dU[64 * LV];
  bf16 oD[64 * LO];    // dO (row stride LV), then v (LV), then diag(beta) D (kLdC)
  bf16 T[64 * kLdC], PDP[64 * kLdC];  // P, then dP (.) Gamma
  bf16 r1[R1], r2[R2];
  float G[64], Gl[64], gam[64], dec[64], beta[64];
  float dgam[64], dbg[64], ddec[64], dB[64], Erow[64], Ecol[64], dG[64];
  float tmp[4];
};

template <int DK, int DV>
__host__ __device__ constexpr int grad_split() { return (DK > 64 || DV > 64) ? 2 : 1; }

// Column sums over the warp's 16 rows of a 16 x 8NT accumulator at columns
// n0.., added into col[].
template <int NT>
__device__ __forceinline__ void add_col_sums(const float (&e)[NT][4], int n0, float *col) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float c0 = e[t][0] + e[t][2], c1 = e[t][1] + e[t][3];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      c0 += __shfl_xor_sync(0xffffffffu, c0, o);
      c1 += __shfl_xor_sync(0xffffffffu, c1, o);
    }
    if (l < 4) {
      atomicAdd(col + n0 + 8 * t + 2 * l, c0);
      atomicAdd(col + n0 + 8 * t + 2 * l + 1, c1);
    }
  }
}

// Per-row partials of rows r0 and r0 + 8 (one per lane), summed over the quad
// and, with column-split warps, over the two warps of a row block.
template <int NS>
__device__ __forceinline__ void put_rows(float *arr, int r0, float p0, float p1) {
  p0 = quad_sum(p0);
  p1 = quad_sum(p1);
  if ((threadIdx.x & 3) == 0) {
    if (NS == 1) {
      arr[r0] = p0;
      arr[r0 + 8] = p1;
    } else {
      atomicAdd(arr + r0, p0);
      atomicAdd(arr + r0 + 8, p1);
    }
  }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads * grad_split<DK, DV>())
gdn_bwdc_grad_kernel(const ChunkBwdParams P) {
  constexpr int NS = grad_split<DK, DV>(), NTH = kThreads * NS;
  constexpr int NC = 8 / NS, NK = DK / 8 / NS, NV = DV / 8 / NS;  // n-tiles per warp
  using S = GradSmem<DK, DV>;
  using WS = ChunkWs<DK, DV>;
  constexpr int LK = S::LK, LV = S::LV;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  S &s = *reinterpret_cast<S *>(smem_raw);
  const FwdParams &p = P.f;
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  int n, valid;
  int64_t tok0;
  if (!slot_chunk(p, slot, h, n, tok0, valid)) return;
  const int H = p.num_heads, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = 16 * (warp & 3), r0 = m0 + (lane >> 2), hf = warp >> 2;
  const int nc0 = hf * (kC / NS), nk0 = hf * (DK / NS), nv0 = hf * (DV / NS);  // column offsets
  const size_t unit = (size_t)slot * H + h;
  WS ws;
  ws.carve(P.ws, P.slots * H);
  bf16 *sH = s.r1, *sDRW = s.r1, *sDH = s.r2, *sDRU = s.r2;

  // ---- loads: every tile in flight at once ----
  const size_t rq = ((size_t)tok0 * H + h) * DK, rv = ((size_t)tok0 * H + h) * DV;
  cp_tile<64, DK, NTH>(s.q, LK, static_cast<const bf16 *>(p.q) + rq, (size_t)H * DK, valid);
  cp_tile<64, DK, NTH>(s.k, LK, static_cast<const bf16 *>(p.k) + rq, (size_t)H * DK, valid);
  cp_tile<64, DV, NTH>(s.oD, LV, P.dO + rv, (size_t)H * DV, valid);
  cp_tile<64, DK, NTH>(s.W, LK, ws.W + unit * WS::kW, DK, kC);
  cp_tile<64, DK, NTH>(s.KtDW, LK, ws.Kt + unit * WS::kKt, DK, kC);
  cp_tile<64, DV, NTH>(s.UU, LV, ws.Ut + unit * WS::kUt, DV, kC);
  cp_tile<64, kC, NTH>(s.T, kLdC, ws.T + unit * WS::kT, kC, kC);
  cp_tile<DK, DV, NTH>(sH, LV, ws.Hb + unit * WS::kH, DV, DK);
  cp_tile<DK, DV, NTH>(sDH, LV, ws.dHb + unit * WS::kH, DV, DK);
  cp_commit();
  if (tid < kC) {
    s.Ecol[tid] = 0.f;
    if (NS > 1) s.dgam[tid] = s.dbg[tid] = s.ddec[tid] = s.dB[tid] = s.Erow[tid] = 0.f;
  }
  chunk_gates(p.g, static_cast<const bf16 *>(p.beta), tok0, H, h, valid, s.G, s.Gl, s.gam,
              s.dec, s.beta, s.tmp);
  const float4 gcv = *reinterpret_cast<const float4 *>(ws.gC + unit * 4);
  const float gC = gcv.x, dgC = gcv.y;
  cp_wait<0>();
  __syncthreads();

  // ---- P, U = U~ - W H ----
  {
    float acc[NC][4];
    zero(acc);
    wmma<NC, false, true>(acc, s.q, LK, m0, s.k, LK, nc0, DK);
    each2(acc, m0, nc0, [&](int i, int j, float &x0, float &x1) {
      const float p0 = i >= j ? x0 * ex2(s.Gl[i] - s.Gl[j]) : 0.f;
      const float p1 = i >= j + 1 ? x1 * ex2(s.Gl[i] - s.Gl[j + 1]) : 0.f;
      st_bf2(&s.PDP[i * kLdC + j], p0, p1);
    });
  }
  {
    float acc[NV][4];
    zero(acc);
    wmma<NV, false, false>(acc, s.W, LK, m0, sH, LV, nv0, DK);
    each2(acc, m0, nv0, [&](int i, int c, float &x0, float &x1) {   // U over U~, in place
      st_bf2(&s.UU[i * LV + c], bf(s.UU[i * LV + c]) - x0, bf(s.UU[i * LV + c + 1]) - x1);
    });
  }
  __syncthreads();
  // dU = P^T dO + K~ dH'; what rounding it to bf16 leaves out stays in registers
  uint32_t dUr[NV][2], dWr[NK][2];
  {
    float acc[NV][4];
    zero(acc);
    wmma<NV, true, false>(acc, s.PDP, kLdC, m0, s.oD, LV, nv0, kC);
    wmma<NV, false, false>(acc, s.KtDW, LK, m0, sDH, LV, nv0, DK);
    each2(acc, m0, nv0, [&](int i, int c, float &x0, float &x1) { st_bf2(&s.dU[i * LV + c], x0, x1); });
#pragma unroll
    for (int t = 0; t < NV; ++t) {
      dUr[t][0] = pack_bf16(acc[t][0] - rbf(acc[t][0]), acc[t][1] - rbf(acc[t][1]));
      dUr[t][1] = pack_bf16(acc[t][2] - rbf(acc[t][2]), acc[t][3] - rbf(acc[t][3]));
    }
  }
  __syncthreads();

  // ---- dP (.) Gamma and its gate terms, dW, dK~, dO H^T ----
  float erow0 = 0.f, erow1 = 0.f;   // row sums of the gate terms E (rows r0, r0 + 8)
  {
    float acc[NC][4], qk[NC][4];
    zero(acc);
    wmma<NC, false, true>(acc, s.oD, LV, m0, s.UU, LV, nc0, DV);
    zero(qk);
    wmma<NC, false, true>(qk, s.q, LK, m0, s.k, LK, nc0, DK);
    // E = dP (.) Gamma (.) Q K^T on and below the diagonal
#pragma unroll
    for (int t = 0; t < NC; ++t) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = r0 + (e >= 2 ? 8 : 0), j = nc0 + 8 * t + 2 * (lane & 3) + (e & 1);
        const float d = i >= j ? acc[t][e] * ex2(s.Gl[i] - s.Gl[j]) : 0.f;
        acc[t][e] = d;
        qk[t][e] *= d;
        if (e < 2) erow0 += qk[t][e]; else erow1 += qk[t][e];
      }
    }
    each2(acc, m0, nc0, [&](int i, int j, float &x0, float &x1) { st_bf2(&s.PDP[i * kLdC + j], x0, x1); });
    add_col_sums(qk, nc0, s.Ecol);
  }
  {
    float acc[NK][4];
    zero(acc);
    wmma<NK, false, true>(acc, s.dU, LV, m0, sH, LV, nk0, DV);
    each2(acc, m0, nk0, [&](int i, int d, float &x0, float &x1) { st_bf2(&s.KtDW[i * LK + d], -x0, -x1); });
#pragma unroll
    for (int t = 0; t < NK; ++t) {
      dWr[t][0] = pack_bf16(rbf(acc[t][0]) - acc[t][0], rbf(acc[t][1]) - acc[t][1]);
      dWr[t][1] = pack_bf16(rbf(acc[t][2]) - acc[t][2], rbf(acc[t][3]) - acc[t][3]);
    }
  }
  float dK[NK][4], dQ[NK][4];
  {
    zero(dK);
    wmma<NK, false, true>(dK, s.UU, LV, m0, sDH, LV, nk0, DV);   // dK~ = U dH'^T
    float p0 = 0.f, p1 = 0.f;
    each2(dK, m0, nk0, [&](int i, int d, float &x0, float &x1) {
      const float e = x0 * bf(s.k[i * LK + d]) + x1 * bf(s.k[i * LK + d + 1]);
      if (i == r0) p0 += e; else p1 += e;
      x0 *= s.dec[i];
      x1 *= s.dec[i];
    });
    put_rows<NS>(s.ddec, r0, p0, p1);
    zero(dQ);
    wmma<NK, false, true>(dQ, s.oD, LV, m0, sH, LV, nk0, DV);   // dO H^T
    p0 = p1 = 0.f;
    each2(dQ, m0, nk0, [&](int i, int d, float &x0, float &x1) {
      const float e = x0 * bf(s.q[i * LK + d]) + x1 * bf(s.q[i * LK + d + 1]);
      if (i == r0) p0 += e; else p1 += e;
      x0 *= s.gam[i];
      x1 *= s.gam[i];
    });
    put_rows<NS>(s.dgam, r0, p0, p1);
  }
  __syncthreads();

  // ---- dR_W = T^T dW, dR_U = T^T dU, dV, dQ ----
  // U and dO are spent: U~ comes back for dA, v takes dO's place
  cp_tile<64, DV, NTH>(s.UU, LV, ws.Ut + unit * WS::kUt, DV, kC);
  cp_tile<64, DV, NTH>(s.oD, LV, static_cast<const bf16 *>(p.v) + rv, (size_t)H * DV, valid);
  cp_commit();
  {
    float acc[NK][4];
    zero(acc);
    wmma<NK, true, false>(acc, s.T, kLdC, m0, s.KtDW, LK, nk0, kC);
#pragma unroll
    for (int t = 0; t < NK; ++t) {   // T's diagonal is 1: the rounding remainder of dW
      acc[t][0] += bf16_lo(dWr[t][0]); acc[t][1] += bf16_hi(dWr[t][0]);
      acc[t][2] += bf16_lo(dWr[t][1]); acc[t][3] += bf16_hi(dWr[t][1]);
    }
    float p0 = 0.f, p1 = 0.f;
    each2(acc, m0, nk0, [&](int i, int d, float &x0, float &x1) {
      const float e = x0 * bf(s.k[i * LK + d]) + x1 * bf(s.k[i * LK + d + 1]);
      if (i == r0) p0 += e; else p1 += e;
      st_bf2(&sDRW[i * LK + d], x0, x1);
    });
    const float bg0 = s.beta[r0] * s.gam[r0], bg1 = s.beta[r0 + 8] * s.gam[r0 + 8];
#pragma unroll
    for (int t = 0; t < NK; ++t) {
      dK[t][0] = fmaf(bg0, acc[t][0], dK[t][0]);
      dK[t][1] = fmaf(bg0, acc[t][1], dK[t][1]);
      dK[t][2] = fmaf(bg1, acc[t][2], dK[t][2]);
      dK[t][3] = fmaf(bg1, acc[t][3], dK[t][3]);
    }
    put_rows<NS>(s.dbg, r0, p0, p1);
  }
  {
    float acc[NV][4];
    zero(acc);
    wmma<NV, true, false>(acc, s.T, kLdC, m0, s.dU, LV, nv0, kC);
#pragma unroll
    for (int t = 0; t < NV; ++t) {
      acc[t][0] += bf16_lo(dUr[t][0]); acc[t][1] += bf16_hi(dUr[t][0]);
      acc[t][2] += bf16_lo(dUr[t][1]); acc[t][3] += bf16_hi(dUr[t][1]);
    }
    cp_wait<0>();
    __syncthreads();   // v and U~ landed
    float p0 = 0.f, p1 = 0.f;
    each2(acc, m0, nv0, [&](int i, int c, float &x0, float &x1) {
      const float e = x0 * bf(s.oD[i * LV + c]) + x1 * bf(s.oD[i * LV + c + 1]);
      if (i == r0) p0 += e; else p1 += e;
      st_bf2(&sDRU[i * LV + c], x0, x1);
      if (i < valid)
        *reinterpret_cast<float2 *>(P.dv + ((size_t)(tok0 + i) * H + h) * DV + c) =
            make_float2(s.beta[i] * x0, s.beta[i] * x1);
    });
    if (NS == 1) {
      p0 = quad_sum(p0);
      p1 = quad_sum(p1);
      if ((lane & 3) == 0) { s.dB[r0] = p0; s.dB[r0 + 8] = p1; }
    } else {
      put_rows<NS>(s.dB, r0, p0, p1);
    }
  }
  wmma<NK, false, false>(dQ, s.PDP, kLdC, m0, s.k, LK, nk0, kC);   // + (dP (.) Gamma) K
  each2(dQ, m0, nk0, [&](int i, int d, float &x0, float &x1) {
    if (i < valid)
      *reinterpret_cast<float2 *>(P.dq + ((size_t)(tok0 + i) * H + h) * DK + d) = make_float2(x0, x1);
  });
  __syncthreads();

  // ---- dA = -(dR_W W^T + dR_U U~^T), D = dA (.) Gamma below the diagonal ----
  {
    float acc[NC][4], kk[NC][4];
    zero(acc);
    wmma<NC, false, true>(acc, sDRW, LK, m0, s.W, LK, nc0, DK);
    wmma<NC, false, true>(acc, sDRU, LV, m0, s.UU, LV, nc0, DV);
    zero(kk);
    wmma<NC, false, true>(kk, s.k, LK, m0, s.k, LK, nc0, DK);
    float p0 = 0.f, p1 = 0.f;
#pragma unroll
    for (int t = 0; t < NC; ++t) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = r0 + (e >= 2 ? 8 : 0), j = nc0 + 8 * t + 2 * (lane & 3) + (e & 1);
        const float D = i > j ? -acc[t][e] * ex2(s.Gl[i] - s.Gl[j]) : 0.f;
        const float dk = D * kk[t][e];            // the dbeta term; beta_i times it is E
        if (e < 2) { p0 += dk; erow0 += s.beta[i] * dk; } else { p1 += dk; erow1 += s.beta[i] * dk; }
        kk[t][e] = s.beta[i] * dk;
        acc[t][e] = s.beta[i] * D;                // diag(beta) D
      }
    }
    add_col_sums(kk, nc0, s.Ecol);
    each2(acc, m0, nc0, [&](int i, int j, float &x0, float &x1) { st_bf2(&s.oD[i * kLdC + j], x0, x1); });
    if (NS == 1) {
      p0 = quad_sum(p0);
      p1 = quad_sum(p1);
      if ((lane & 3) == 0) { s.dB[r0] += p0; s.dB[r0 + 8] += p1; }
    } else {
      put_rows<NS>(s.dB, r0, p0, p1);
    }
    put_rows<NS>(s.Erow, r0, erow0, erow1);
  }
  __syncthreads();

  // ---- dK += (diag(beta) D) K + (diag(beta) D)^T K + (dP (.) Gamma)^T Q ----
  wmma<NK, false, false>(dK, s.oD, kLdC, m0, s.k, LK, nk0, kC);
  wmma<NK, true, false>(dK, s.oD, kLdC, m0, s.k, LK, nk0, kC);
  wmma<NK, true, false>(dK, s.PDP, kLdC, m0, s.q, LK, nk0, kC);
  each2(dK, m0, nk0, [&](int i, int d, float &x0, float &x1) {
    if (i < valid)
      *reinterpret_cast<float2 *>(P.dk + ((size_t)(tok0 + i) * H + h) * DK + d) = make_float2(x0, x1);
  });

  // ---- gates: dG per token, then dg = its sum over later tokens of the chunk ----
  if (tid < kC) {
    const int i = tid;
    const float dgt = s.dgam[i] + s.beta[i] * s.dbg[i];
    s.dG[i] = s.Erow[i] - s.Ecol[i] + s.gam[i] * dgt - s.dec[i] * s.ddec[i];
    s.dB[i] += s.gam[i] * s.dbg[i];
    float xdec = s.dec[i] * s.ddec[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) xdec += __shfl_xor_sync(0xffffffffu, xdec, o);
    if (lane == 0) s.tmp[2 + warp] = xdec;
  }
  __syncthreads();
  if (tid < kC) {
    // suffix sums: thread t takes token 63 - t
    const int t = tid, i = kC - 1 - t;
    float x = s.dG[i];
    if (i == kC - 1) x += gC * dgC + s.tmp[2] + s.tmp[3];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (t == 31) s.tmp[1] = x;
    s.dG[i] = x;
  }
  __syncthreads();
  if (tid < kC) {
    const int t = tid, i = kC - 1 - t;
    const float x = s.dG[i] + (t >= 32 ? s.tmp[1] : 0.f);
    if (i < valid) {
      const size_t off = (size_t)(tok0 + i) * H + h;
      P.dg[off] = x;
      P.dbeta[off] = s.dB[i];
    }
  }
}

// ----------------------------------------------------------------- host ----
template <typename K>
cudaError_t smem_attr(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DK, int DV>
cudaError_t launch_dims(const ChunkBwdParams &P, cudaStream_t s) {
  auto prep = gdn_bwdc_prep_kernel<DK, DV>;
  auto fwd = gdn_bwdc_chain_kernel<DK, DV, false>;
  auto rev = gdn_bwdc_chain_kernel<DK, DV, true>;
  auto grad = gdn_bwdc_grad_kernel<DK, DV>;
  const size_t sp = sizeof(PrepSmem<DK, DV>), sf = sizeof(ChainSmem<DK, DV, false>);
  const size_t sr = sizeof(ChainSmem<DK, DV, true>), sg = sizeof(GradSmem<DK, DV>);
  cudaError_t e;
  if ((e = smem_attr(prep, sp)) != cudaSuccess || (e = smem_attr(fwd, sf)) != cudaSuccess ||
      (e = smem_attr(rev, sr)) != cudaSuccess || (e = smem_attr(grad, sg)) != cudaSuccess)
    return e;
  const dim3 per_chunk((unsigned)P.slots, (unsigned)P.f.num_heads);
  const dim3 per_seq((unsigned)P.f.num_heads, (unsigned)P.f.num_seqs,
                     (unsigned)(DV / ChainSmem<DK, DV, false>::SW));
  prep<<<per_chunk, kPrepThreads, sp, s>>>(P);
  fwd<<<per_seq, kThreads, sf, s>>>(P);
  rev<<<per_seq, kThreads, sr, s>>>(P);
  grad<<<per_chunk, kThreads * grad_split<DK, DV>(), sg, s>>>(P);
  return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const ChunkBwdParams &P, cudaStream_t s) {
  switch (P.f.dv) {
    case 32: return launch_dims<DK, 32>(P, s);
    case 64: return launch_dims<DK, 64>(P, s);
    case 128: return launch_dims<DK, 128>(P, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int DK>
size_t ws_dk(int64_t units, int dv) {
  switch (dv) {
    case 32: return ChunkWs<DK, 32>::bytes(units);
    case 64: return ChunkWs<DK, 64>::bytes(units);
    default: return ChunkWs<DK, 128>::bytes(units);
  }
}

}  // namespace

bool bwd_chunked_supported(int dk, int dv) {
  return (dk == 32 || dk == 64 || dk == 128) && (dv == 32 || dv == 64 || dv == 128);
}

size_t bwd_chunked_ws_bytes(int64_t units, int dk, int dv) {
  if (dk == 32) return ws_dk<32>(units, dv);
  if (dk == 64) return ws_dk<64>(units, dv);
  return ws_dk<128>(units, dv);
}

cudaError_t launch_bwd_chunked(const FwdParams &f, const void *dO, const float *dHN, float *dq,
                               float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                               void *ws, int64_t slots, cudaStream_t s) {
  ChunkBwdParams P;
  P.f = f;
  P.dO = static_cast<const bf16 *>(dO);
  P.dHN = dHN;
  P.dq = dq; P.dk = dk; P.dv = dv; P.dg = dg; P.dbeta = dbeta; P.dh0 = dh0;
  P.ws = ws;
  P.slots = slots;
  if (f.dk == 32) return launch_dk<32>(P, s);
  if (f.dk == 64) return launch_dk<64>(P, s);
  return launch_dk<128>(P, s);
}

}  // namespace gdn
