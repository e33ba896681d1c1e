// Fused chunked forward of the gated delta rule on fp32 CUDA cores.
//
// One CTA owns one (sequence, head, 32-wide slice of the value dimension) and
// walks that sequence's chunks of C tokens (C = 32, 64 or 128; 64 is the
// pages' default) in order, keeping its slice of the
// fp32 state H = S^T (dk x 32) in shared memory for the whole sequence (state
// kept on chip: "Model Architecture Walkthrough", section 6.3; chunked with a
// serial inter-chunk carry: "Optimization Quartet", Triton GDN kernel
// section 3.2).  Columns of H evolve independently of one another, so slices
// of the value dimension need no communication.
//
// Per chunk, with G the chunk-local inclusive prefix sum of g, gamma = exp(G),
// Gamma_ij = exp(G_i - G_j) (i >= j) -- the unrolled decay weight of "Model
// Architecture Walkthrough", section 5.3.1 -- and H0 the state entering the
// chunk, the gated delta rule of Yang et al. (arXiv 2412.06464) becomes
//
//   A = strictly_lower(diag(beta) K K^T (.) Gamma)
//   (I + A) U = diag(beta) V - diag(beta * gamma) K H0        (forward substitution)
//   O   = diag(gamma) Q H0 + (Q K^T (.) Gamma, i >= j) U
//   H_C = gamma_C H0 + (diag(exp(G_C - G)) K)^T U
//
// Exponentials are only ever taken of differences G_i - G_j with i >= j (<= 0
// for non-positive gates), never of G alone negated, so nothing overflows.
// This kernel is the precision path (fp32 storage) and the reference GPU path
// for every configuration; it is simple rather than fast.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kDvTile = 32;

template <int DK, int C>
struct SimtSmem {
  static constexpr int QK_LD = DK + 1;      // padded rows: conflict-free column walks
  static constexpr int U_LD = kDvTile + 1;
  static constexpr int A_LD = C + 1;
  static constexpr int kFloats = 2 * C * QK_LD + C * U_LD + C * kDvTile + DK * kDvTile +
                                 C * A_LD + 4 * C;
  static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int DK, int C, typename Tin>
__global__ void __launch_bounds__(kThreads)
gdn_fwd_simt_kernel(const FwdParams p) {
  using L = SimtSmem<DK, C>;
  constexpr int DVT = kDvTile;
  constexpr int PER_LANE = C / 32;       // gates per lane in the prefix sum
  extern __shared__ float smem[];
  float *sQ = smem;                      // [C][QK_LD]
  float *sK = sQ + C * L::QK_LD;         // [C][QK_LD]
  float *sU = sK + C * L::QK_LD;         // [C][U_LD]   V -> R -> U
  float *sO = sU + C * L::U_LD;          // [C][DVT]    diag(gamma) Q H0
  float *sH = sO + C * DVT;              // [DK][DVT]   the state slice
  float *sA = sH + DK * DVT;             // [C][A_LD]   A, then P (after the substitution)
  float *sG = sA + C * L::A_LD;          // [C] cumulative log-gate
  float *sB = sG + C;                    // [C] beta
  float *sGam = sB + C;                  // [C] exp(G_i)
  float *sDec = sGam + C;                // [C] exp(G_last - G_j)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv;
  const int col0 = tile * DVT;

  int64_t start, len;
  if (!sequence_bounds(p, n, h, start, len)) return;
  if ((p.flags & GDN_DEBUG_CHECKS) &&
      !debug_ranges_ok(p, n, h, start, len, col0, DVT, (int)sizeof(Tin), false))
    return;  // recorded; nothing was accessed
  if (len == 0) {   // an empty sequence: the state passes through
    pass_state_through(p, n, h, col0, DVT);
    return;
  }

  const Tin *q = static_cast<const Tin *>(p.q);
  const Tin *k = static_cast<const Tin *>(p.k);
  const Tin *v = static_cast<const Tin *>(p.v);
  const Tin *beta = static_cast<const Tin *>(p.beta);
  Tin *o = static_cast<Tin *>(p.o);
  const size_t state_base = ((size_t)n * H + h) * (size_t)DK * dv + col0;

  for (int idx = tid; idx < DK * DVT; idx += kThreads) {
    const int d = idx / DVT, c = idx % DVT;
    sH[idx] = p.s0 ? p.s0[state_base + (size_t)d * dv + c] : 0.f;
  }

  for (int64_t c0 = 0; c0 < len; c0 += C) {
    const int rows = (int)(len - c0 < C ? len - c0 : C);
    __syncthreads();  // previous chunk finished with every buffer

    // ---- load the chunk (rows past the end are zero: no effect on H) ----
    for (int idx = tid; idx < C * DK; idx += kThreads) {
      const int r = idx / DK, d = idx % DK;
      float qv = 0.f, kv = 0.f;
      if (r < rows) {
        const size_t off = ((size_t)(start + c0 + r) * H + h) * DK + d;
        qv = to_f32(q[off]);
        kv = to_f32(k[off]);
      }
      sQ[r * L::QK_LD + d] = qv;
      sK[r * L::QK_LD + d] = kv;
    }
    for (int idx = tid; idx < C * DVT; idx += kThreads) {
      const int r = idx / DVT, c = idx % DVT;
      float vv = 0.f;
      if (r < rows) vv = to_f32(v[((size_t)(start + c0 + r) * H + h) * dv + col0 + c]);
      sU[r * L::U_LD + c] = vv;
    }
    if (tid < C) {
      float gg = 0.f, bb = 0.f;
      if (tid < rows) {
        const size_t off = (size_t)(start + c0 + tid) * H + h;
        gg = p.g[off];
        bb = beta_value(to_f32(beta[off]), p.flags);
      }
      sG[tid] = gg;
      sB[tid] = bb;
    }
    __syncthreads();

    // ---- optional q/k L2 normalisation: x / sqrt(sum x^2 + 1e-6) ----
    if (p.flags & GDN_QK_L2NORM) {
      for (int row = warp; row < 2 * C; row += kThreads / 32) {
        float *x = (row < C ? sQ + row * L::QK_LD : sK + (row - C) * L::QK_LD);
        float ss = 0.f;
        for (int d = lane; d < DK; d += 32) ss += x[d] * x[d];
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss + 1e-6f);
        for (int d = lane; d < DK; d += 32) x[d] *= inv;
      }
    }

    // ---- chunk-local inclusive prefix sum of the log-gates ----
    if (warp == 0) {
      float part[PER_LANE];
      float run = 0.f;
#pragma unroll
      for (int e = 0; e < PER_LANE; ++e) {
        run += sG[PER_LANE * lane + e];
        part[e] = run;
      }
      float s = run;
      for (int off = 1; off < 32; off <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += t;
      }
      const float excl = s - run;
#pragma unroll
      for (int e = 0; e < PER_LANE; ++e) sG[PER_LANE * lane + e] = excl + part[e];
    }
    __syncthreads();
    if (tid < C) {
      sGam[tid] = expf(sG[tid]);
      sDec[tid] = expf(sG[C - 1] - sG[tid]);
    }

    // ---- A = strictly_lower(diag(beta) K K^T (.) Gamma) ----
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int i = idx / C, j = idx % C;
      float a = 0.f;
      if (j < i) {
        const float *ki = sK + i * L::QK_LD, *kj = sK + j * L::QK_LD;
        float dkk = 0.f;
#pragma unroll 8
        for (int d = 0; d < DK; ++d) dkk = fmaf(ki[d], kj[d], dkk);
        a = sB[i] * dkk * expf(sG[i] - sG[j]);
      }
      sA[i * L::A_LD + j] = a;
    }
    __syncthreads();

    // ---- R = diag(beta)(V - diag(gamma) K H0) into sU; sO = diag(gamma) Q H0 ----
    for (int idx = tid; idx < C * DVT; idx += kThreads) {
      const int i = idx / DVT, c = idx % DVT;
      const float *qi = sQ + i * L::QK_LD, *ki = sK + i * L::QK_LD;
      float kh = 0.f, qh = 0.f;
#pragma unroll 8
      for (int d = 0; d < DK; ++d) {
        const float hv = sH[d * DVT + c];
        kh = fmaf(ki[d], hv, kh);
        qh = fmaf(qi[d], hv, qh);
      }
      sU[i * L::U_LD + c] = sB[i] * (sU[i * L::U_LD + c] - sGam[i] * kh);
      sO[i * DVT + c] = sGam[i] * qh;
    }
    __syncthreads();

    // ---- (I + A) U = R by forward substitution; one thread per column ----
    if (tid < DVT) {
      const int c = tid;
      for (int i = 1; i < rows; ++i) {
        const float *ai = sA + i * L::A_LD;
        float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
        int j = 0;
        for (; j + 3 < i; j += 4) {
          acc0 = fmaf(ai[j], sU[j * L::U_LD + c], acc0);
          acc1 = fmaf(ai[j + 1], sU[(j + 1) * L::U_LD + c], acc1);
          acc2 = fmaf(ai[j + 2], sU[(j + 2) * L::U_LD + c], acc2);
          acc3 = fmaf(ai[j + 3], sU[(j + 3) * L::U_LD + c], acc3);
        }
        for (; j < i; ++j) acc0 = fmaf(ai[j], sU[j * L::U_LD + c], acc0);
        sU[i * L::U_LD + c] -= (acc0 + acc1) + (acc2 + acc3);
      }
    }
    __syncthreads();

    // ---- P = Q K^T (.) Gamma (i >= j), into A's buffer (A is no longer needed) ----
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int i = idx / C, j = idx % C;
      float pp = 0.f;
      if (j <= i) {
        const float *qi = sQ + i * L::QK_LD, *kj = sK + j * L::QK_LD;
        float dqk = 0.f;
#pragma unroll 8
        for (int d = 0; d < DK; ++d) dqk = fmaf(qi[d], kj[d], dqk);
        pp = dqk * expf(sG[i] - sG[j]);
      }
      sA[i * L::A_LD + j] = pp;
    }
    __syncthreads();

    // ---- O = sO + P U (stored); H_C = gamma_C H0 + (diag(dec) K)^T U ----
    for (int idx = tid; idx < C * DVT; idx += kThreads) {
      const int i = idx / DVT, c = idx % DVT;
      if (i < rows && o) {
        const float *pi = sA + i * L::A_LD;
        float acc = sO[i * DVT + c];
        for (int j = 0; j <= i; ++j) acc = fmaf(pi[j], sU[j * L::U_LD + c], acc);
        const size_t orow = (size_t)(start + c0 + i) * H + h;
        if (p.d_skip || p.out_gate)  // block epilogue (o + D_h v) * gate
          acc = block_epilogue(acc, to_f32(v[orow * dv + col0 + c]), p.d_skip ? p.d_skip[h] : 0.f,
                               p.out_gate ? p.out_gate[orow] : 1.f);
        store_out(o + orow * dv + col0 + c, acc);
      }
    }
    const float gam_last = sGam[C - 1];
    for (int idx = tid; idx < DK * DVT; idx += kThreads) {
      const int d = idx / DVT, c = idx % DVT;
      float acc = gam_last * sH[idx];
      for (int j = 0; j < rows; ++j)
        acc = fmaf(sK[j * L::QK_LD + d] * sDec[j], sU[j * L::U_LD + c], acc);
      sH[idx] = acc;
    }
  }
  __syncthreads();
  if (p.sN)
    for (int idx = tid; idx < DK * DVT; idx += kThreads) {
      const int d = idx / DVT, c = idx % DVT;
      p.sN[state_base + (size_t)d * dv + c] = sH[idx];
    }
}

template <int DK, int C, typename Tin>
cudaError_t launch_simt_dk(const FwdParams &p, cudaStream_t stream) {
  auto kern = gdn_fwd_simt_kernel<DK, C, Tin>;
  const size_t smem = SimtSmem<DK, C>::kBytes;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const dim3 grid(p.dv / kDvTile, p.num_heads, p.num_seqs);
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int C, typename Tin>
cudaError_t launch_simt_c(const FwdParams &p, cudaStream_t stream) {
  switch (p.dk) {
    case 32: return launch_simt_dk<32, C, Tin>(p, stream);
    case 64: return launch_simt_dk<64, C, Tin>(p, stream);
    case 128:
      if constexpr (C <= 64) return launch_simt_dk<128, C, Tin>(p, stream);
      return cudaErrorInvalidValue;   // 128-token chunks with dk = 128 exceed shared memory
    default: return cudaErrorInvalidValue;
  }
}

template <typename Tin>
cudaError_t launch_simt_t(const FwdParams &p, int chunk, cudaStream_t stream) {
  switch (chunk) {
    case 32: return launch_simt_c<32, Tin>(p, stream);
    case 64: return launch_simt_c<64, Tin>(p, stream);
    case 128: return launch_simt_c<128, Tin>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool simt_chunk_supported(int chunk, int dk) {
  return (chunk == 32 || chunk == 64 || chunk == 128) && !(chunk == 128 && dk == 128);
}

cudaError_t launch_fwd_simt(const FwdParams &p, gdn_dtype dtype, int chunk, cudaStream_t stream) {
  return dtype == GDN_F32 ? launch_simt_t<float>(p, chunk, stream)
                          : launch_simt_t<__nv_bfloat16>(p, chunk, stream);
}

}  // namespace gdn
