// Backward pass of the gated delta rule (recompute style: "Optimization
// Quartet", Triton GDN kernel section 3.4 -- the pages' kernel recomputes
// what it needs from the inputs; "Model Architecture Walkthrough", section
// 6.5 -- the backward is a recurrence run backwards in time).
//
// Forward, per (sequence, head), with H = S^T (dk x dv) and alpha = exp(g):
//
//   s_t = H_{t-1}^T k_t,   u_t = beta_t (v_t - alpha_t s_t),
//   H_t = alpha_t H_{t-1} + k_t u_t^T,   o_t = H_t^T q_t.
//
// Backward, t = T..1, with dH the gradient of the state (dH = dH_N at t = T):
//
//   dH   += q_t do_t^T                          dq_t = H_t do_t
//   du    = dH^T k_t,   w = beta_t du          dv_t = w
//   dbeta_t = <du, v_t - alpha_t s_t>
//   dalpha_t = <dH, H_{t-1}> - <w, s_t>         dg_t = alpha_t dalpha_t
//   dk_t  = dH u_t - alpha_t H_{t-1} w
//   dH   <- alpha_t (dH - k_t w^T)              (dH_0 = d initial state)
//
// Columns of H evolve independently, so a CTA owns 32 value columns of one
// (sequence, head) and each of its 8 warps owns 4 of them, rows spread over
// the lanes: the serial chain (du, the dH update, and in the recompute the
// s_t reduction) needs warp shuffles only.  States are recomputed from
// checkpoints (one per 64-token chunk, written by a token-serial fp32 scan of
// the forward with the same layout): once per chunk to the start of each
// 8-token sub-chunk, then per sub-chunk into shared memory.  The sums
// over columns (dq, dk, dbeta, dalpha) gather in shared memory per sub-chunk
// and are added to the fp32 outputs with atomics (several CTAs share a head
// when dv > 32).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kBT = 256;    // threads per CTA: 8 warps x 4 value columns
constexpr int kCols = 32;   // value columns per CTA
constexpr int kSub = 8;     // tokens per recomputed sub-chunk
constexpr int kCk = 64;     // checkpoint interval (the forward's chunk)

struct BwdParams {
  FwdParams f;
  const void *dO;
  const float *dHN;
  const float *ckpt;
  float *scratch;           // per CTA: the sub-chunk start states of one chunk
  int sub_ckpt;             // checkpoints per 64-token chunk: 8 (every sub-chunk) or 1
  float *dq, *dk, *dv, *dg, *dbeta, *dh0;
};

template <int DK>
struct BwdSmem {
  static constexpr int NR = DK / 32;                       // rows per lane
  static constexpr int EL = NR * 4;                        // state elements per thread
  static constexpr int TRAJ = (kSub + 1) * EL * kBT;       // thread-private trajectory
  static constexpr int kFloats = TRAJ + 2 * kSub * DK      // q, k
                                 + 4 * kSub * kCols        // v, do, s, u
                                 + 2 * kSub * DK + 2 * kSub  // dq, dk, dalpha, dbeta sums
                                 + 2 * kSub;               // alpha, beta
  static constexpr size_t kBytes = kFloats * sizeof(float);
};

// Column sums of four values over the warp; every lane gets all four.
__device__ __forceinline__ void reduce4(const float (&a)[4], float (&out)[4], int lane) {
  const bool hi16 = lane & 16, hi8 = lane & 8;
  const float r0 = __shfl_xor_sync(0xffffffffu, hi16 ? a[0] : a[2], 16);
  const float r1 = __shfl_xor_sync(0xffffffffu, hi16 ? a[1] : a[3], 16);
  const float k0 = (hi16 ? a[2] : a[0]) + r0, k1 = (hi16 ? a[3] : a[1]) + r1;
  float x = (hi8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  // lane 0: column 0, lane 8: 1, lane 16: 2, lane 24: 3
#pragma unroll
  for (int j = 0; j < 4; ++j) out[j] = __shfl_sync(0xffffffffu, x, 8 * j);
}

template <int DK, typename Tin>
__global__ void __launch_bounds__(kBT)
gdn_bwd_kernel(const BwdParams P) {
  using L = BwdSmem<DK>;
  constexpr int NR = L::NR;
  extern __shared__ float sm[];
  float *traj = sm;                          // [kSub+1][EL][kBT], thread-private
  float *sQ = traj + L::TRAJ;                // [kSub][DK]
  float *sK = sQ + kSub * DK;                // [kSub][DK]
  float *sV = sK + kSub * DK;                // [kSub][kCols]
  float *sDO = sV + kSub * kCols;            // [kSub][kCols]
  float *sS = sDO + kSub * kCols;            // [kSub][kCols]  s_t
  float *sU = sS + kSub * kCols;             // [kSub][kCols]  u_t
  float *aQ = sU + kSub * kCols;             // [kSub][DK]     dq sums
  float *aK = aQ + kSub * DK;                // [kSub][DK]     dk sums
  float *aA = aK + kSub * DK;                // [kSub]         dalpha sums
  float *aB = aA + kSub;                     // [kSub]         dbeta sums
  float *sAl = aB + kSub;                    // [kSub]         alpha
  float *sBe = sAl + kSub;                   // [kSub]         beta

  const FwdParams &p = P.f;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv;
  const int col0 = tile * kCols, cw = 4 * warp;
  int64_t start, len;
  if (!sequence_bounds(p, n, h, start, len)) return;

  const Tin *q = static_cast<const Tin *>(p.q);
  const Tin *k = static_cast<const Tin *>(p.k);
  const Tin *v = static_cast<const Tin *>(p.v);
  const Tin *beta = static_cast<const Tin *>(p.beta);
  const Tin *dO = static_cast<const Tin *>(P.dO);
  const size_t state_base = ((size_t)n * H + h) * (size_t)DK * dv + col0 + cw;

  // gradient of the state, element (row lane + 32 i, column cw + j)
  float dH[NR][4];
#pragma unroll
  for (int i = 0; i < NR; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dH[i][j] = P.dHN ? P.dHN[state_base + (size_t)(lane + 32 * i) * dv + j] : 0.f;

  const int64_t ck0 = ckpt_first_slot(n, start, p.seq_len, p.cu != nullptr);
  const int nck = (int)((len + kCk - 1) / kCk);
  float *scr = P.scratch + ((((size_t)n * H + h) * (dv / kCols) + tile) * (kCk / kSub)) *
                               (size_t)(L::EL * kBT);

  // tokens [t0, t0 + cnt) of the sequence into shared memory (zeros past cnt)
  auto load_sub = [&](int64_t t0, int cnt, bool bwd) {
    for (int idx = tid; idx < kSub * DK; idx += kBT) {
      const int i = idx / DK, d = idx % DK;
      float kv = 0.f, qv = 0.f;
      if (i < cnt) {
        const size_t off = ((size_t)(start + t0 + i) * H + h) * DK + d;
        kv = to_f32(k[off]);
        if (bwd) qv = to_f32(q[off]);
      }
      sK[idx] = kv;
      sQ[idx] = qv;
      aQ[idx] = 0.f;
      aK[idx] = 0.f;
    }
    for (int idx = tid; idx < kSub * kCols; idx += kBT) {
      const int i = idx / kCols, c = idx % kCols;
      float vv = 0.f, dd = 0.f;
      if (i < cnt) {
        const size_t off = ((size_t)(start + t0 + i) * H + h) * dv + col0 + c;
        vv = to_f32(v[off]);
        if (bwd) dd = to_f32(dO[off]);
      }
      sV[idx] = vv;
      sDO[idx] = dd;
    }
    if (tid < kSub) {
      float al = 1.f, be = 0.f;
      if (tid < cnt) {
        const size_t off = (size_t)(start + t0 + tid) * H + h;
        al = expf(p.g[off]);
        be = to_f32(beta[off]);
      }
      sAl[tid] = al;
      sBe[tid] = be;
      aA[tid] = 0.f;
      aB[tid] = 0.f;
    }
  };

  // one forward token step on this warp's columns; records s_t and u_t
  auto fwd_step = [&](float (&Hr)[NR][4], int i) {
    const float al = sAl[i], be = sBe[i];
    float kr[NR], part[4], s[4];
#pragma unroll
    for (int r = 0; r < NR; ++r) kr[r] = sK[i * DK + lane + 32 * r];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a = 0.f;
#pragma unroll
      for (int r = 0; r < NR; ++r) a = fmaf(Hr[r][j], kr[r], a);
      part[j] = a;
    }
    reduce4(part, s, lane);
    const float4 vq = *reinterpret_cast<const float4 *>(sV + i * kCols + cw);
    const float vv[4] = {vq.x, vq.y, vq.z, vq.w};
    float u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) u[j] = be * (vv[j] - al * s[j]);
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int j = 0; j < 4; ++j) Hr[r][j] = fmaf(al, Hr[r][j], kr[r] * u[j]);
    if (lane < 4) {
      const float sv = lane == 0 ? s[0] : lane == 1 ? s[1] : lane == 2 ? s[2] : s[3];
      const float uv = lane == 0 ? u[0] : lane == 1 ? u[1] : lane == 2 ? u[2] : u[3];
      sS[i * kCols + cw + lane] = sv;
      sU[i * kCols + cw + lane] = uv;
    }
  };
  auto traj_put = [&](int i, const float (&Hr)[NR][4]) {
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int j = 0; j < 4; ++j) traj[(i * L::EL + r * 4 + j) * kBT + tid] = Hr[r][j];
  };

  for (int c = nck - 1; c >= 0; --c) {
    const int64_t cs = (int64_t)c * kCk;
    const int clen = (int)(len - cs < kCk ? len - cs : kCk);
    const int nsub = (clen + kSub - 1) / kSub;

    // (a) from the chunk's checkpoint, the state at each sub-chunk start (when
    // the scan kept only one checkpoint per chunk)
    float Hr[NR][4];
    if (P.sub_ckpt == 1) {
      const float *ck = P.ckpt + ((ck0 + c) * H + h) * (size_t)DK * dv + col0 + cw;
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) Hr[r][j] = ck[(size_t)(lane + 32 * r) * dv + j];
      for (int sb = 0; sb < nsub; ++sb) {
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int j = 0; j < 4; ++j) scr[((size_t)sb * L::EL + r * 4 + j) * kBT + tid] = Hr[r][j];
        if (sb == nsub - 1) break;
        __syncthreads();   // shared buffers free
        load_sub(cs + (int64_t)sb * kSub, kSub, false);
        __syncthreads();
        for (int i = 0; i < kSub; ++i) fwd_step(Hr, i);
      }
    }

    // (b) sub-chunks in reverse: recompute their states, then step backwards
    for (int sb = nsub - 1; sb >= 0; --sb) {
      const int64_t t0 = cs + (int64_t)sb * kSub;
      const int cnt = (int)(clen - sb * kSub < kSub ? clen - sb * kSub : kSub);
      __syncthreads();   // shared buffers free (previous flush done)
      load_sub(t0, cnt, true);
      if (P.sub_ckpt == 8) {   // the scan's checkpoint of this sub-chunk
        const float *ck = P.ckpt + (((ck0 + c) * 8 + sb) * H + h) * (size_t)DK * dv + col0 + cw;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float4 x = *reinterpret_cast<const float4 *>(ck + (size_t)(lane + 32 * r) * dv);
          Hr[r][0] = x.x; Hr[r][1] = x.y; Hr[r][2] = x.z; Hr[r][3] = x.w;
        }
      } else {
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int j = 0; j < 4; ++j) Hr[r][j] = scr[((size_t)sb * L::EL + r * 4 + j) * kBT + tid];
      }
      __syncthreads();
      traj_put(0, Hr);
      for (int i = 0; i < cnt; ++i) {
        fwd_step(Hr, i);
        traj_put(i + 1, Hr);
      }
      __syncwarp();   // s_t, u_t of this warp's columns are in place

      // H_t of the step, carried from the previous (later) step's H_{t-1}
      float Hc[NR][4];
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) Hc[r][j] = traj[(cnt * L::EL + r * 4 + j) * kBT + tid];
      for (int i = cnt - 1; i >= 0; --i) {
        const float al = sAl[i], be = sBe[i];
        float kr[NR], qr[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          kr[r] = sK[i * DK + lane + 32 * r];
          qr[r] = sQ[i * DK + lane + 32 * r];
        }
        const float4 dq4 = *reinterpret_cast<const float4 *>(sDO + i * kCols + cw);
        const float4 v4 = *reinterpret_cast<const float4 *>(sV + i * kCols + cw);
        const float4 s4 = *reinterpret_cast<const float4 *>(sS + i * kCols + cw);
        const float4 u4 = *reinterpret_cast<const float4 *>(sU + i * kCols + cw);
        const float dOj[4] = {dq4.x, dq4.y, dq4.z, dq4.w}, vj[4] = {v4.x, v4.y, v4.z, v4.w};
        const float sj[4] = {s4.x, s4.y, s4.z, s4.w}, uj[4] = {u4.x, u4.y, u4.z, u4.w};
        float Hp[NR][4];   // H_{t-1}
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int j = 0; j < 4; ++j) Hp[r][j] = traj[(i * L::EL + r * 4 + j) * kBT + tid];
        // dH += q do^T;  dq = H_t do
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float dq = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            dH[r][j] = fmaf(qr[r], dOj[j], dH[r][j]);
            dq = fmaf(Hc[r][j], dOj[j], dq);
          }
          atomicAdd(&aQ[i * DK + lane + 32 * r], dq);
        }
        // du = dH^T k;  w = beta du
        float part[4], du[4], w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float a = 0.f;
#pragma unroll
          for (int r = 0; r < NR; ++r) a = fmaf(dH[r][j], kr[r], a);
          part[j] = a;
        }
        reduce4(part, du, lane);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = be * du[j];
        if (lane < 4) {
          const float wv = lane == 0 ? w[0] : lane == 1 ? w[1] : lane == 2 ? w[2] : w[3];
          P.dv[((size_t)(start + t0 + i) * H + h) * dv + col0 + cw + lane] = wv;
        }
        // dbeta = <du, v - alpha s>;  dalpha = <dH, H_{t-1}> - <w, s>
        float db = 0.f, ws = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          db = fmaf(du[j], vj[j] - al * sj[j], db);
          ws = fmaf(w[j], sj[j], ws);
        }
        float da = 0.f;
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int j = 0; j < 4; ++j) da = fmaf(dH[r][j], Hp[r][j], da);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) da += __shfl_xor_sync(0xffffffffu, da, off);
        if (lane == 0) {
          atomicAdd(&aB[i], db);
          atomicAdd(&aA[i], da - ws);
        }
        // dk = dH u - alpha H_{t-1} w;  dH <- alpha (dH - k w^T)
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float dk = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            dk = fmaf(dH[r][j], uj[j], dk);
            dk = fmaf(-al * Hp[r][j], w[j], dk);
            dH[r][j] = al * fmaf(-kr[r], w[j], dH[r][j]);
          }
          atomicAdd(&aK[i * DK + lane + 32 * r], dk);
        }
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int j = 0; j < 4; ++j) Hc[r][j] = Hp[r][j];
      }
      __syncthreads();   // every warp's sums are in
      // the column sums of this CTA into the fp32 outputs
      for (int idx = tid; idx < cnt * DK; idx += kBT) {
        const int i = idx / DK, d = idx % DK;
        const size_t off = ((size_t)(start + t0 + i) * H + h) * DK + d;
        atomicAdd(P.dq + off, aQ[idx]);
        atomicAdd(P.dk + off, aK[idx]);
      }
      if (tid < cnt) {
        const size_t off = (size_t)(start + t0 + tid) * H + h;
        atomicAdd(P.dg + off, aA[tid] * sAl[tid]);
        atomicAdd(P.dbeta + off, aB[tid]);
      }
    }
  }
  if (P.dh0) {
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int j = 0; j < 4; ++j) P.dh0[state_base + (size_t)(lane + 32 * r) * dv + j] = dH[r][j];
  }
}

// Forward scan that keeps the checkpoints the backward kernel restarts from:
// the state entering every 64-token chunk (sub_ckpt = 1) or every 8-token
// sub-chunk (sub_ckpt = 8, slot (chunk slot) * 8 + sub-chunk).  Token by token
// in fp32 -- the recurrence as written, the same step as the backward's
// recompute -- with the CTA and warp layout of the backward kernel: a CTA owns
// 32 value columns of one (sequence, head), each warp 4 of them with the key
// rows over the lanes, and the tokens are staged a chunk at a time in shared
// memory.  Tokens after the last checkpoint are not scanned.
template <int DK, typename Tin>
__global__ void __launch_bounds__(kBT)
gdn_bwd_ckpt_kernel(const FwdParams p, const int sub_ckpt) {
  constexpr int NR = DK / 32;
  __shared__ float sK[kCk * DK];
  __shared__ float sV[kCk * kCols];
  __shared__ float sAl[kCk], sBe[kCk];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv;
  const int col0 = tile * kCols, cw = 4 * warp;
  int64_t start, len;
  if (!sequence_bounds(p, n, h, start, len)) return;
  const Tin *k = static_cast<const Tin *>(p.k);
  const Tin *v = static_cast<const Tin *>(p.v);
  const Tin *beta = static_cast<const Tin *>(p.beta);
  const size_t state_base = ((size_t)n * H + h) * (size_t)DK * dv + col0 + cw;

  float Hr[NR][4];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.s0) x = *reinterpret_cast<const float4 *>(p.s0 + state_base + (size_t)(lane + 32 * r) * dv);
    Hr[r][0] = x.x; Hr[r][1] = x.y; Hr[r][2] = x.z; Hr[r][3] = x.w;
  }
  auto put = [&](int64_t slot) {
    float *ck = p.ckpt + (slot * H + h) * (size_t)DK * dv + col0 + cw;
#pragma unroll
    for (int r = 0; r < NR; ++r)
      *reinterpret_cast<float4 *>(ck + (size_t)(lane + 32 * r) * dv) =
          make_float4(Hr[r][0], Hr[r][1], Hr[r][2], Hr[r][3]);
  };
  const int64_t ck0 = ckpt_first_slot(n, start, p.seq_len, p.cu != nullptr);
  const int nck = (int)((len + kCk - 1) / kCk);
  for (int c = 0; c < nck; ++c) {
    const int64_t t0 = (int64_t)c * kCk;
    const int clen = (int)(len - t0 < kCk ? len - t0 : kCk);
    put((ck0 + c) * sub_ckpt);
    // tokens to scan in this chunk: up to the next checkpoint that exists
    const int cnt = c < nck - 1 ? kCk : (sub_ckpt == 8 ? ((clen - 1) / kSub) * kSub : 0);
    if (cnt == 0) break;
    __syncthreads();   // the previous chunk's tokens are consumed
    for (int idx = tid; idx < cnt * DK; idx += kBT) {
      const int i = idx / DK, d = idx % DK;
      sK[idx] = to_f32(k[((size_t)(start + t0 + i) * H + h) * DK + d]);
    }
    for (int idx = tid; idx < cnt * kCols; idx += kBT) {
      const int i = idx / kCols, cc = idx % kCols;
      sV[idx] = to_f32(v[((size_t)(start + t0 + i) * H + h) * dv + col0 + cc]);
    }
    if (tid < cnt) {
      const size_t off = (size_t)(start + t0 + tid) * H + h;
      sAl[tid] = expf(p.g[off]);
      sBe[tid] = to_f32(beta[off]);
    }
    __syncthreads();
#pragma unroll 1
    for (int i = 0; i < cnt; ++i) {
      if (sub_ckpt == 8 && i > 0 && (i & (kSub - 1)) == 0) put((ck0 + c) * 8 + i / kSub);
      const float al = sAl[i], be = sBe[i];
      float kr[NR], part[4], sv[4];
#pragma unroll
      for (int r = 0; r < NR; ++r) kr[r] = sK[i * DK + lane + 32 * r];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float a = 0.f;
#pragma unroll
        for (int r = 0; r < NR; ++r) a = fmaf(Hr[r][j], kr[r], a);
        part[j] = a;
      }
      reduce4(part, sv, lane);
      const float4 vj = *reinterpret_cast<const float4 *>(sV + i * kCols + cw);
      const float u[4] = {be * (vj.x - al * sv[0]), be * (vj.y - al * sv[1]),
                          be * (vj.z - al * sv[2]), be * (vj.w - al * sv[3])};
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) Hr[r][j] = fmaf(al, Hr[r][j], kr[r] * u[j]);
    }
    // the last sub-chunk start of a short final chunk follows its last scanned token
    if (sub_ckpt == 8 && c == nck - 1) {
      put((ck0 + c) * 8 + cnt / kSub);
      break;
    }
  }
}

template <int DK, typename Tin>
cudaError_t launch_ckpt_dk(const FwdParams &f, int per_chunk, cudaStream_t s) {
  const dim3 grid(f.dv / kCols, f.num_heads, f.num_seqs);
  gdn_bwd_ckpt_kernel<DK, Tin><<<grid, kBT, 0, s>>>(f, per_chunk);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_ckpt_t(const FwdParams &f, int per_chunk, cudaStream_t s) {
  switch (f.dk) {
    case 32: return launch_ckpt_dk<32, Tin>(f, per_chunk, s);
    case 64: return launch_ckpt_dk<64, Tin>(f, per_chunk, s);
    case 128: return launch_ckpt_dk<128, Tin>(f, per_chunk, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int DK, typename Tin>
cudaError_t launch_bwd_dk(const BwdParams &P, cudaStream_t s) {
  auto kern = gdn_bwd_kernel<DK, Tin>;
  const size_t smem = BwdSmem<DK>::kBytes;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const dim3 grid(P.f.dv / kCols, P.f.num_heads, P.f.num_seqs);
  kern<<<grid, kBT, smem, s>>>(P);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_bwd_t(const BwdParams &P, cudaStream_t s) {
  switch (P.f.dk) {
    case 32: return launch_bwd_dk<32, Tin>(P, s);
    case 64: return launch_bwd_dk<64, Tin>(P, s);
    case 128: return launch_bwd_dk<128, Tin>(P, s);
    default: return cudaErrorInvalidValue;
  }
}

// Checkpoints per 64-token chunk: one at every sub-chunk start while that
// array stays within 4 GiB (the backward then skips recomputing the sub-chunk
// starts), else one per chunk.
int ckpt_per_chunk(int64_t num_seqs, int64_t seq_len, int64_t H, int64_t dk, int64_t dv) {
  const int64_t fine = ckpt_slots(num_seqs, seq_len) * (kCk / kSub) * H * dk * dv * 4;
  return fine <= (int64_t(4) << 30) ? kCk / kSub : 1;
}

size_t scratch_floats(int64_t num_seqs, int64_t H, int64_t dk, int64_t dv) {
  return (size_t)num_seqs * H * (dv / kCols) * (kCk / kSub) * (size_t)(dk / 32 * 4 * kBT);
}

bool aligned16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

// A call with no tokens (gdn_api.cu): the state gradient passes through.
gdn_status pass_states(const float *from, float *to, size_t bytes, cudaStream_t s);

// The chunked tensor-core backward for bf16 storage (gdn_bwd_chunk.cu).
bool bwd_chunked_supported(int dk, int dv);
size_t bwd_chunked_ws_bytes(int64_t units, int dk, int dv);
cudaError_t launch_bwd_chunked(const FwdParams &f, const void *dO, const float *dHN, float *dq,
                               float *dk, float *dv, float *dg, float *dbeta, float *dh0,
                               void *ws, int64_t slots, cudaStream_t s);
}  // namespace gdn

extern "C" size_t gdn_bwd_workspace_size(int32_t num_seqs, int32_t seq_len, int32_t num_heads,
                                         int32_t head_dim_k, int32_t head_dim_v) {
  using namespace gdn;
  if (num_seqs <= 0 || seq_len < 0 || num_heads <= 0 || head_dim_k <= 0 || head_dim_v <= 0)
    return 0;
  if (head_dim_v % kCols) return 0;
  const int per = ckpt_per_chunk(num_seqs, seq_len, num_heads, head_dim_k, head_dim_v);
  const size_t ck =
      (size_t)ckpt_slots(num_seqs, seq_len) * per * num_heads * head_dim_k * head_dim_v;
  size_t need = kStatusBytes + 4 * (ck + scratch_floats(num_seqs, num_heads, head_dim_k, head_dim_v));
  // bf16 storage with small heads takes the chunked path, with its own records
  if (bwd_chunked_supported(head_dim_k, head_dim_v)) {
    const size_t chunked = kStatusBytes + bwd_chunked_ws_bytes(
        ckpt_slots(num_seqs, seq_len) * num_heads, head_dim_k, head_dim_v);
    if (chunked > need) need = chunked;
  }
  return need;
}

extern "C" gdn_status gdn_bwd(const void *q, const void *k, const void *v, const float *g,
                              const void *beta, const float *initial_state,
                              const int32_t *cu_seqlens, const void *d_o,
                              const float *d_final_state, float *dq, float *dk, float *dv,
                              float *dg, float *dbeta, float *d_initial_state, int32_t batch,
                              int32_t seq_len, int32_t num_heads, int32_t head_dim_k,
                              int32_t head_dim_v, int32_t num_seqs, gdn_dtype dtype,
                              uint32_t flags, void *workspace, size_t workspace_bytes,
                              void *stream) {
  using namespace gdn;
  if (batch <= 0 || seq_len < 0 || num_heads <= 0 || head_dim_k <= 0 || head_dim_v <= 0 ||
      num_seqs <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (flags != 0u) return GDN_ERR_INVALID_ARG;
  if (cu_seqlens ? batch != 1 : num_seqs != batch) return GDN_ERR_INVALID_ARG;
  if (!(head_dim_k == 32 || head_dim_k == 64 || head_dim_k == 128)) return GDN_ERR_UNSUPPORTED;
  if (head_dim_v < 32 || head_dim_v > 256 || head_dim_v % 32) return GDN_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_heads > 65535) return GDN_ERR_UNSUPPORTED;
  if (seq_len == 0)   // no tokens: the state gradient passes through, nothing else is read
    return pass_states(d_final_state, d_initial_state,
                       (size_t)num_seqs * num_heads * head_dim_k * head_dim_v * 4,
                       (cudaStream_t)stream);
  if (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta)
    return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, initial_state, cu_seqlens, d_o, d_final_state,
                        dq, dk, dv, dg, dbeta, d_initial_state};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  if (!workspace) return GDN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_bwd_workspace_size(num_seqs, seq_len, num_heads, head_dim_k, head_dim_v);
  if (workspace_bytes < need) return GDN_ERR_WORKSPACE;

  // aliasing: the gradients overlap no input and no other gradient
  const size_t e = dtype == GDN_F32 ? 4 : 2;
  const size_t rows = (size_t)batch * seq_len * num_heads;
  const size_t b_qk = rows * head_dim_k * e, b_v = rows * head_dim_v * e;
  const size_t b_g = rows * 4, b_beta = rows * e;
  const size_t b_state = (size_t)num_seqs * num_heads * head_dim_k * head_dim_v * 4;
  const size_t b_cu = cu_seqlens ? (size_t)(num_seqs + 1) * 4 : 0;
  struct Range { const void *p; size_t n; };
  const Range ins[] = {{q, b_qk}, {k, b_qk}, {v, b_v}, {g, b_g}, {beta, b_beta},
                       {initial_state, b_state}, {cu_seqlens, b_cu}, {d_o, b_v},
                       {d_final_state, b_state}, {workspace, workspace_bytes}};
  const Range outs[] = {{dq, rows * head_dim_k * 4}, {dk, rows * head_dim_k * 4},
                        {dv, rows * head_dim_v * 4}, {dg, rows * 4}, {dbeta, rows * 4},
                        {d_initial_state, b_state}};
  for (const Range &o : outs) {
    for (const Range &i : ins)
      if (overlaps(o.p, o.n, i.p, i.n)) return GDN_ERR_INVALID_ARG;
    for (const Range &o2 : outs)
      if (&o2 != &o && overlaps(o.p, o.n, o2.p, o2.n)) return GDN_ERR_INVALID_ARG;
  }

  cudaStream_t s = (cudaStream_t)stream;
  unsigned char *ws = static_cast<unsigned char *>(workspace);

  BwdParams P;
  FwdParams &f = P.f;
  f.q = q; f.k = k; f.v = v; f.beta = beta; f.g = g;
  f.s0 = initial_state; f.cu = cu_seqlens; f.o = nullptr; f.sN = nullptr;
  f.d_skip = nullptr; f.out_gate = nullptr;
  f.ext = Extents{};
  f.status = reinterpret_cast<DeviceStatus *>(ws);
  f.ckpt = nullptr;
  f.seq_len = seq_len;
  f.num_heads = num_heads; f.dk = head_dim_k; f.dv = head_dim_v; f.num_seqs = num_seqs;
  f.flags = 0;

  // bf16 storage, head_dim_k and head_dim_v up to 64: the chunked backward,
  // which writes every gradient once (no zero fills, no atomics)
  if (dtype == GDN_BF16 && bwd_chunked_supported(head_dim_k, head_dim_v)) {
    const cudaError_t err = launch_bwd_chunked(
        f, d_o, d_final_state, dq, dk, dv, dg, dbeta, d_initial_state, ws + kStatusBytes,
        ckpt_slots(num_seqs, seq_len), s);
    return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  }

  float *ckpt = reinterpret_cast<float *>(ws + kStatusBytes);
  const int per = ckpt_per_chunk(num_seqs, seq_len, num_heads, head_dim_k, head_dim_v);
  float *scratch = ckpt + (size_t)ckpt_slots(num_seqs, seq_len) * per * num_heads * head_dim_k *
                              head_dim_v;

  // the gradients gathered with atomics start from zero
  if (cudaMemsetAsync(dq, 0, rows * head_dim_k * 4, s) != cudaSuccess ||
      cudaMemsetAsync(dk, 0, rows * head_dim_k * 4, s) != cudaSuccess ||
      cudaMemsetAsync(dg, 0, rows * 4, s) != cudaSuccess ||
      cudaMemsetAsync(dbeta, 0, rows * 4, s) != cudaSuccess)
    return GDN_ERR_CUDA;

  f.ckpt = ckpt;
  // the forward as a token-serial fp32 scan, keeping only the checkpoints
  cudaError_t err = dtype == GDN_F32 ? launch_ckpt_t<float>(f, per, s)
                                     : launch_ckpt_t<__nv_bfloat16>(f, per, s);
  if (err != cudaSuccess) return GDN_ERR_CUDA;
  f.ckpt = nullptr;
  P.dO = d_o; P.dHN = d_final_state; P.ckpt = ckpt; P.scratch = scratch;
  P.sub_ckpt = per;
  P.dq = dq; P.dk = dk; P.dv = dv; P.dg = dg; P.dbeta = dbeta; P.dh0 = d_initial_state;
  err = dtype == GDN_F32 ? launch_bwd_t<float>(P, s) : launch_bwd_t<__nv_bfloat16>(P, s);
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
