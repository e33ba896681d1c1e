// The HyMo pages' per-row (diagonal) decay combined with the delta rule's
// erase and write strength, for d_state = head_dim = 32.  Per batch row and
// head, token by token ("Model Architecture Walkthrough", section 5.2.1 for
// the decay exp(g_t A), A = -exp(A_log), and the keys b (write) and c (read);
// the erase and beta are those of the gated delta rule of the main path):
//
//   hbar = exp(g_t A) (.) h          (row s scaled by exp(g_t A_s))
//   h    = hbar + beta_t b_t (v_t - hbar^T b_t)^T
//   o_t  = h^T c_t
//
// The step is affine in the state, so a run of tokens maps h_start to
// M h_start + X, and each output to o_t = o0_t + r_t^T h_start, where X and
// o0_t are the run from a zero state and column k of M and r_t[k] the run
// from the unit vector e_k with v = 0 (the read of that run: r_t = M_t^T c_t).
//
// Work split: one CTA of two warps per (batch row, head, 128-token segment).
// A warp holds a 32 x 32 state in registers, an 8 x 4 block per lane.  Warp 0
// runs the segment from a zero state (from the initial state in segment 0),
// keeping o0 in shared memory; warp 1 runs it from the identity with v = 0,
// keeping r.  Then the segment's start state comes from its predecessor
// segment's published end state (a look-back one segment deep), the CTA
// publishes its own end state M h_start + X, and writes o = o0 + r^T h_start.
// CTAs take their segment from a ticket counter in launch order, segment-major,
// so a CTA only waits on a CTA that started before it; every wait is bounded.
//
// Per token a lane reads 8 rows of d, b and c and 4 values of v from shared
// memory and does 64 packed two-lane fp32 operations on pairs of state rows;
// the column sums over the state rows take 16 shuffles.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace ddelta {

using namespace ptx;

constexpr int kS = 32;            // state rows (d_state)
constexpr int kD = 32;            // value columns (head_dim)
constexpr int kTile = 16;         // tokens per staged tile
constexpr int kSeg = 128;         // tokens per segment (one CTA)
constexpr int kThreads = 64;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// Workspace: [0, 256) status word (first 16 bytes) and counters at byte 64;
// then one flag per task and one published end state per task.
struct Counters {
  uint32_t ticket, done, epoch, pad;
};
constexpr size_t kCountersOff = 64;

struct Workspace {
  size_t flags, hend, total;
};
inline Workspace workspace_layout(int64_t tasks) {
  Workspace w;
  w.flags = kStatusBytes;
  w.hend = (w.flags + (size_t)tasks * 4 + 255) & ~(size_t)255;
  w.total = w.hend + (size_t)tasks * kS * kD * 4;
  return w;
}

#ifdef GDN_DDELTA_PROBE
// Phase-timing build only: globaltimer stamps of thread 0, [ticket][phase].
static __device__ unsigned long long g_ddelta_probe[8192 * 6];
#define GDN_DDPROBE(k)                                                        \
  do {                                                                        \
    if (threadIdx.x == 0 && ticket < 8192u)                                   \
      ::gdn::ddelta::g_ddelta_probe[ticket * 6u + (k)] = globaltimer_ns();    \
  } while (0)
#else
#define GDN_DDPROBE(k) \
  do {                 \
  } while (0)
#endif

struct Params {
  const void *v, *b, *c, *beta;
  const float *g, *A_log, *h0;
  const float *D_skip, *out_gate;   // block epilogue (NULL = off)
  void *o;
  float *hN;
  DeviceStatus *status;
  Counters *ctr;
  uint32_t *flags;
  float *hend;
  int32_t batch, seq_len, num_heads, nseg;
  uint32_t opts;                    // GDN_GATE_SIGMOID, GDN_BETA_LOGITS
};

// o0 and r are kept in the storage type T (bf16 storage: the outputs are
// rounded to bf16 anyway, and the smaller buffers let 6 CTAs share an SM)
template <typename T>
struct Smem {
  // staged tiles, double-buffered: rows [d, b, c][token][s], v and beta;
  // after the token loop the tile rows hold M^T and X
  float row[2][3][kTile][kS];
  float vt[2][kTile][kD];
  float bt[2][kTile];
  float hs[kS][kD];                 // h_start
  T obuf[kSeg][kD];                 // o0 (warp 0)
  T rbuf[kSeg][kS];                 // r (warp 1)
  uint32_t misc[4];
};

__device__ __forceinline__ void st4(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }
__device__ __forceinline__ void st4(__nv_bfloat16 *p, float4 x) {
  *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
}
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

__device__ __forceinline__ float ldf(const float *p) { return __ldg(p); }
__device__ __forceinline__ float lds(const float *p) { return *p; }
__device__ __forceinline__ float lds(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

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
__device__ __forceinline__ float sigmoid(float x) { return 1.f / (1.f + ex2(-x * kLog2e)); }

// Four column partial sums, each a packed pair over two rows: add the pair,
// then sum over the four row groups (lane bits 3 and 4).
__device__ __forceinline__ float4 cols_reduce(const uint64_t (&acc)[4]) {
  float4 r;
  float lo, hi;
  upk2(acc[0], lo, hi); r.x = lo + hi;
  upk2(acc[1], lo, hi); r.y = lo + hi;
  upk2(acc[2], lo, hi); r.z = lo + hi;
  upk2(acc[3], lo, hi); r.w = lo + hi;
#pragma unroll
  for (int m = 8; m <= 16; m <<= 1) {
    r.x += __shfl_xor_sync(0xffffffffu, r.x, m);
    r.y += __shfl_xor_sync(0xffffffffu, r.y, m);
    r.z += __shfl_xor_sync(0xffffffffu, r.z, m);
    r.w += __shfl_xor_sync(0xffffffffu, r.w, m);
  }
  return r;
}

// Lane layout: lane = 8 rg + cg holds the state rows 8 rg .. 8 rg + 7 and the
// columns 4 cg .. 4 cg + 3, packed in pairs of rows (h2[q][k]: rows 8 rg + 2q
// and + 1 of column 4 cg + k), so that a token reads 8 rows of d, b, c (as
// pairs, no repacking) and 4 values of v from shared memory per lane, and the
// column sums over the rows take two shuffle levels.
template <typename T>
__global__ void __launch_bounds__(kThreads) gdn_diag_delta_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem<T> &sm = *reinterpret_cast<Smem<T> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = lane >> 3, cg = lane & 7, r0 = 8 * rg, c0 = 4 * cg;
  const int H = p.num_heads, Tn = p.seq_len;
  if (tid == 0) {
    sm.misc[0] = atomicAdd(&p.ctr->ticket, 1u);
    sm.misc[1] = *reinterpret_cast<volatile uint32_t *>(&p.ctr->epoch);
  }
  __syncthreads();
  const uint32_t ticket = sm.misc[0];
  const uint32_t tag = 2u * sm.misc[1] + 1u;   // odd: never the zeroed flag
  const int units = p.batch * H;
  const int seg = (int)(ticket / (uint32_t)units), unit = (int)(ticket % (uint32_t)units);
  const int bb = unit / H, hd = unit % H;
  const int64_t t0 = (int64_t)seg * kSeg;
  const int len = (int)min((int64_t)kSeg, (int64_t)Tn - t0);
  const bool first = seg == 0, last = seg == p.nseg - 1;
  const bool transport = warp == 1;
  const bool runs = !(first && transport);      // segment 0 needs no transport run
  GDN_DDPROBE(0);
  const T *vp = static_cast<const T *>(p.v), *bp = static_cast<const T *>(p.b);
  const T *cp = static_cast<const T *>(p.c), *betap = static_cast<const T *>(p.beta);
  // element (token t of this segment, s) of a [B][T][H][32] tensor
  auto at = [&](int t, int s) -> int64_t {
    return (((int64_t)bb * Tn + t0 + t) * H + hd) * 32 + s;
  };
  auto gate_at = [&](int t) -> int64_t { return ((int64_t)bb * Tn + t0 + t) * H + hd; };
  const size_t srow = ((size_t)bb * H + hd) * kS * kD;

  const float a2 = -expf(p.A_log[hd * kS + lane]) * kLog2e;   // row `lane`: d = 2^(g a2)
  const bool gate_sig = (p.opts & GDN_GATE_SIGMOID) != 0;
  const bool beta_sig = (p.opts & GDN_BETA_LOGITS) != 0;

  // the state block: zero, the initial state, or the identity
  // h2[q][k] packs rows r0 + 2q and r0 + 2q + 1 of column c0 + k, so that the
  // per-row factors d, b, c load from shared memory as ready-made pairs
  uint64_t h2[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float4 x[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int s = r0 + 2 * q + e;
      x[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (transport) {
        x[e] = make_float4(s == c0 ? 1.f : 0.f, s == c0 + 1 ? 1.f : 0.f, s == c0 + 2 ? 1.f : 0.f,
                           s == c0 + 3 ? 1.f : 0.f);
      } else if (first && p.h0) {
        x[e] = *reinterpret_cast<const float4 *>(p.h0 + srow + (size_t)s * kD + c0);
      }
    }
    h2[q][0] = pk2(x[0].x, x[1].x);
    h2[q][1] = pk2(x[0].y, x[1].y);
    h2[q][2] = pk2(x[0].z, x[1].z);
    h2[q][3] = pk2(x[0].w, x[1].w);
  }

  // ---- staging: thread (warp w, lane s) handles tokens 8w .. 8w+7 of a tile ----
  float rb[8], rc[8], rg8[8], rv[8], rbeta = 0.f;
  auto fetch = [&](int tt) {   // tile starting at segment token tt, into registers
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = tt + 8 * warp + i;
      const bool ok = t < len;
      rb[i] = ok ? ldf(bp + at(t, lane)) : 0.f;
      rc[i] = ok ? ldf(cp + at(t, lane)) : 0.f;
      rv[i] = ok ? ldf(vp + at(t, lane)) : 0.f;
      rg8[i] = ok ? p.g[gate_at(t)] : 0.f;
    }
    const int tb = tt + 8 * warp + lane;
    rbeta = (lane < 8 && tb < len) ? ldf(betap + gate_at(tb)) : 0.f;
  };
  auto commit = [&](int buf, int tt) {   // registers -> shared tile `buf`
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int tl = 8 * warp + i;
      const bool ok = tt + tl < len;   // a padded token is an identity step
      const float g = gate_sig ? sigmoid(rg8[i]) : rg8[i];
      sm.row[buf][0][tl][lane] = ok ? ex2(g * a2) : 1.f;
      sm.row[buf][1][tl][lane] = rb[i];
      sm.row[buf][2][tl][lane] = rc[i];
      sm.vt[buf][tl][lane] = rv[i];
    }
    if (lane < 8) {
      const int tl = 8 * warp + lane;
      sm.bt[buf][tl] = (tt + tl < len) ? (beta_sig ? sigmoid(rbeta) : rbeta) : 0.f;
    }
  };

  const int ntiles = (len + kTile - 1) / kTile;
  fetch(0);
  commit(0, 0);
  __syncthreads();
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1, tt = it * kTile;
    if (it + 1 < ntiles) fetch(tt + kTile);
    if (runs) {
      T *out = transport ? &sm.rbuf[0][0] : &sm.obuf[0][0];
#pragma unroll 1
      for (int tl = 0; tl < kTile; ++tl) {
        // rows r0 .. r0 + 7 of d, b, c as four packed pairs each
        const ulonglong2 *rd = reinterpret_cast<const ulonglong2 *>(&sm.row[buf][0][tl][r0]);
        const ulonglong2 *rbk = reinterpret_cast<const ulonglong2 *>(&sm.row[buf][1][tl][r0]);
        const ulonglong2 *rc = reinterpret_cast<const ulonglong2 *>(&sm.row[buf][2][tl][r0]);
        const ulonglong2 d01 = rd[0], d23 = rd[1], k01 = rbk[0], k23 = rbk[1];
        const uint64_t dp[4] = {d01.x, d01.y, d23.x, d23.y};
        const uint64_t kp[4] = {k01.x, k01.y, k23.x, k23.y};
        // hbar = d (.) h, and b^T hbar over this lane's rows (pairs of rows)
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            h2[q][k] = mul2(dp[q], h2[q][k]);
            acc[k] = fma2(kp[q], h2[q][k], acc[k]);
          }
        }
        const float4 pred = cols_reduce(acc);
        const float4 vv = transport ? make_float4(0.f, 0.f, 0.f, 0.f)
                                    : *reinterpret_cast<const float4 *>(&sm.vt[buf][tl][c0]);
        const float be = sm.bt[buf][tl];
        const float u[4] = {be * (vv.x - pred.x), be * (vv.y - pred.y), be * (vv.z - pred.z),
                            be * (vv.w - pred.w)};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t uu = pk2(u[k], u[k]);
#pragma unroll
          for (int q = 0; q < 4; ++q) h2[q][k] = fma2(kp[q], uu, h2[q][k]);
        }
        // o = c^T h over this lane's rows, then over the row groups
        const ulonglong2 c01 = rc[0], c23 = rc[1];
        const uint64_t cp2[4] = {c01.x, c01.y, c23.x, c23.y};
        uint64_t oacc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int k = 0; k < 4; ++k) oacc[k] = fma2(cp2[q], h2[q][k], oacc[k]);
        }
        const float4 o = cols_reduce(oacc);
        if (rg == 0 && tt + tl < len) st4(out + (tt + tl) * 32 + c0, o);
      }
    }
    if (it + 1 < ntiles) commit(buf ^ 1, tt + kTile);
    __syncthreads();
  }
  GDN_DDPROBE(1);

  // ---- the start state and the composition ----
  // M^T[m][s] = M[s][m] (column m of M is the run from e_m) and X[s][j], over
  // the tile rows (dead after the loop)
  float (*Mt)[kS] = reinterpret_cast<float (*)[kS]>(&sm.row[0][0][0][0]);
  float (*Xs)[kD] = Mt + kS;
  if (runs) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float lo[4], hi[4];   // rows r0 + 2q and r0 + 2q + 1, columns c0 .. c0 + 3
#pragma unroll
      for (int k = 0; k < 4; ++k) upk2(h2[q][k], lo[k], hi[k]);
      if (transport) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          Mt[c0 + k][r0 + 2 * q] = lo[k];
          Mt[c0 + k][r0 + 2 * q + 1] = hi[k];
        }
      } else {
        *reinterpret_cast<float4 *>(&Xs[r0 + 2 * q][c0]) = make_float4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<float4 *>(&Xs[r0 + 2 * q + 1][c0]) =
            make_float4(hi[0], hi[1], hi[2], hi[3]);
      }
    }
  }
  if (!first && tid == 0) {
    const uint32_t *flag = p.flags + (ticket - (uint32_t)units);
    const uint64_t t_start = globaltimer_ns();
    bool ok = false;
    for (uint32_t n = 0;; ++n) {
      if (ld_acquire_gpu(flag) == tag) { ok = true; break; }
      if ((n & 15u) == 15u) {
        if (globaltimer_ns() - t_start > kWaitNs) break;
        __nanosleep(64);
      }
    }
    if (!ok) report(p.status, GDN_ERR_TIMEOUT, (uint32_t)bb, (uint32_t)hd, 3u);
    sm.misc[2] = ok ? 1u : 0u;
  }
  GDN_DDPROBE(2);
  __syncthreads();
  // h_start (segment 0: M = I and X is already its end state, so zero here)
  const bool have_start = !first && sm.misc[2] != 0u;
  {
    const float *src = p.hend + (size_t)(ticket - (first ? 0u : (uint32_t)units)) * kS * kD;
    for (int q = tid; q < kS * kD / 4; q += kThreads) {
      const float4 x = have_start ? __ldcg(reinterpret_cast<const float4 *>(src) + q)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4 *>(&sm.hs[0][0])[q] = x;
    }
  }
  __syncthreads();
  // end state X + M h_start: thread tid computes row tid / 2, columns
  // 16 (tid & 1) .. + 15
  {
    const int s = tid >> 1, cb = 16 * (tid & 1);
    float e[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) e[j] = Xs[s][cb + j];
    if (!first) {
#pragma unroll 4
      for (int m = 0; m < kS; ++m) {
        const float msm = Mt[m][s];
        const float4 *hr = reinterpret_cast<const float4 *>(&sm.hs[m][cb]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 x = hr[q];
          e[4 * q] = fmaf(msm, x.x, e[4 * q]);
          e[4 * q + 1] = fmaf(msm, x.y, e[4 * q + 1]);
          e[4 * q + 2] = fmaf(msm, x.z, e[4 * q + 2]);
          e[4 * q + 3] = fmaf(msm, x.w, e[4 * q + 3]);
        }
      }
    }
    float *dst = p.hend + (size_t)ticket * kS * kD + (size_t)s * kD + cb;
    float *fin = last && p.hN ? p.hN + srow + (size_t)s * kD + cb : nullptr;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 x = make_float4(e[4 * q], e[4 * q + 1], e[4 * q + 2], e[4 * q + 3]);
      __stcg(reinterpret_cast<float4 *>(dst) + q, x);
      if (fin) reinterpret_cast<float4 *>(fin)[q] = x;
    }
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) st_release_gpu(p.flags + ticket, tag);
  GDN_DDPROBE(3);

  // ---- outputs: o = o0 + r^T h_start, then the block epilogue ----
  // lane j: column j of h_start in registers, the row r_t broadcast
  {
    float hcol[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) hcol[q] = sm.hs[q][lane];
    const float dsk = p.D_skip ? p.D_skip[hd] : 0.f;
    T *op = static_cast<T *>(p.o);
#pragma unroll 1
    for (int t = warp; t < len; t += 2) {
      float o = lds(&sm.obuf[t][lane]);
      if (!first) {
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 r = ld4(&sm.rbuf[t][q]);
          a[0] = fmaf(r.x, hcol[q], a[0]);
          a[1] = fmaf(r.y, hcol[q + 1], a[1]);
          a[2] = fmaf(r.z, hcol[q + 2], a[2]);
          a[3] = fmaf(r.w, hcol[q + 3], a[3]);
        }
        o += (a[0] + a[1]) + (a[2] + a[3]);
      }
      if (p.D_skip) o = fmaf(dsk, ldf(vp + at(t, lane)), o);
      if (p.out_gate) o *= p.out_gate[gate_at(t)];
      stf(op + at(t, lane), o);
    }
  }

  GDN_DDPROBE(4);
  // ---- launch bookkeeping: the last CTA out resets the ticket and advances the epoch ----
  if (tid == 0) {
    const uint32_t d = atomicAdd(&p.ctr->done, 1u);
    if (d == gridDim.x - 1) {
      p.ctr->ticket = 0u;
      p.ctr->done = 0u;
      __threadfence();
      atomicAdd(&p.ctr->epoch, 1u);
    }
  }
}

template <typename T>
cudaError_t launch_t(const Params &p, int64_t tasks, cudaStream_t stream) {
  const int smem = (int)sizeof(Smem<T>);
  cudaError_t err = cudaFuncSetAttribute(gdn_diag_delta_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  gdn_diag_delta_kernel<T><<<(unsigned)tasks, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

bool aligned16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace ddelta
}  // namespace gdn

extern "C" size_t gdn_diag_delta_workspace_size(int32_t batch, int32_t seq_len,
                                                int32_t num_heads, int32_t d_state,
                                                int32_t head_dim) {
  using namespace gdn::ddelta;
  if (batch <= 0 || seq_len <= 0 || num_heads <= 0 || d_state <= 0 || head_dim <= 0) return 0;
  const int64_t nseg = ((int64_t)seq_len + kSeg - 1) / kSeg;
  return workspace_layout((int64_t)batch * num_heads * nseg).total;
}

extern "C" gdn_status gdn_diag_delta_fwd(const void *v, const void *b, const void *c,
                                         const float *g, const float *A_log, const void *beta,
                                         const float *D_skip, const float *out_gate,
                                         const float *initial_state, void *o,
                                         float *final_state, int32_t batch, int32_t seq_len,
                                         int32_t num_heads, int32_t d_state, int32_t head_dim,
                                         gdn_dtype dtype, uint32_t flags, void *workspace,
                                         size_t workspace_bytes, void *stream) {
  using namespace gdn;
  using namespace gdn::ddelta;
  if (batch <= 0 || seq_len <= 0 || num_heads <= 0 || d_state <= 0 || head_dim <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)(GDN_GATE_SIGMOID | GDN_BETA_LOGITS)) return GDN_ERR_INVALID_ARG;
  if (d_state != kS || head_dim != kD) return GDN_ERR_UNSUPPORTED;
  const int64_t nseg = ((int64_t)seq_len + kSeg - 1) / kSeg;
  const int64_t tasks = (int64_t)batch * num_heads * nseg;
  if (tasks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if (!v || !b || !c || !g || !A_log || !beta || !o) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {v, b, c, g, A_log, beta, D_skip, out_gate, initial_state, o, final_state};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  if (!workspace) return GDN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GDN_ERR_INVALID_ARG;
  const Workspace wl = workspace_layout(tasks);
  if (workspace_bytes < wl.total) return GDN_ERR_WORKSPACE;

  const size_t e = dtype == GDN_F32 ? 4 : 2;
  const size_t rows = (size_t)batch * (size_t)seq_len * (size_t)num_heads;
  const size_t b_v = rows * kD * e, b_bc = rows * kS * e, b_g = rows * 4, b_beta = rows * e;
  const size_t b_A = (size_t)num_heads * kS * 4;
  const size_t b_state = (size_t)batch * num_heads * kS * kD * 4;
  const size_t b_D = (size_t)num_heads * 4;
  struct Range { const void *p; size_t n; };
  const Range inputs[] = {{v, b_v},     {b, b_bc},     {c, b_bc},       {g, b_g},
                          {A_log, b_A}, {beta, b_beta}, {D_skip, b_D},  {out_gate, b_g},
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
  Params p;
  p.v = v; p.b = b; p.c = c; p.beta = beta; p.g = g; p.A_log = A_log; p.h0 = initial_state;
  p.D_skip = D_skip; p.out_gate = out_gate; p.o = o; p.hN = final_state;
  p.status = reinterpret_cast<DeviceStatus *>(ws);
  p.ctr = reinterpret_cast<Counters *>(ws + kCountersOff);
  p.flags = reinterpret_cast<uint32_t *>(ws + wl.flags);
  p.hend = reinterpret_cast<float *>(ws + wl.hend);
  p.batch = batch; p.seq_len = seq_len; p.num_heads = num_heads; p.nseg = (int32_t)nseg;
  p.opts = flags;
  const cudaError_t err =
      dtype == GDN_F32 ? launch_t<float>(p, tasks, (cudaStream_t)stream)
                       : launch_t<__nv_bfloat16>(p, tasks, (cudaStream_t)stream);
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

#ifdef GDN_DDELTA_PROBE
extern "C" int gdn_ddelta_probe_read(unsigned long long *host) {
  return (int)cudaMemcpyFromSymbol(host, gdn::ddelta::g_ddelta_probe,
                                   sizeof(gdn::ddelta::g_ddelta_probe));
}
#endif
