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
// Lane j of a warp owns column j of a 32 x 32 state in registers.  Warp 0
// runs the segment from a zero state (from the initial state in segment 0),
// keeping o0 in shared memory; warp 1 runs it from the identity with v = 0,
// keeping r.  Then the segment's start state comes from its predecessor
// segment's published end state (a look-back one segment deep), the CTA
// publishes its own end state M h_start + X, and writes o = o0 + r^T h_start.
// CTAs take their segment from a ticket counter in launch order, segment-major,
// so a CTA only waits on a CTA that started before it; every wait is bounded.
//
// Per token a warp reads four 32-float rows from shared memory (b (.) d, d, b,
// c, broadcast to every lane) and does 64 packed two-lane fp32 operations.
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

struct Smem {
  // staged tiles, double-buffered: rows [b (.) d, d, b, c][token][s]; after
  // the token loop the first buffer holds M and X for the composition
  float row[2][4][kTile][kS];
  float vt[2][kTile][kD];
  float bt[2][kTile];
  float obuf[kSeg][kD];             // o0 (warp 0)
  float rbuf[kSeg][kS];             // r (warp 1)
  uint32_t misc[4];
};

__device__ __forceinline__ float ldf(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float sum2(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
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

// sum over s of row[s] * h[s] (h packed in pairs), four independent chains
__device__ __forceinline__ float dot32(const float *row, const uint64_t (&h2)[16]) {
  const ulonglong2 *r = reinterpret_cast<const ulonglong2 *>(row);
  uint64_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const ulonglong2 x = r[i], y = r[i + 1];
    a0 = fma2(x.x, h2[2 * i], a0);
    a1 = fma2(x.y, h2[2 * i + 1], a1);
    a2 = fma2(y.x, h2[2 * i + 2], a2);
    a3 = fma2(y.y, h2[2 * i + 3], a3);
  }
  return (sum2(a0) + sum2(a1)) + (sum2(a2) + sum2(a3));
}

template <typename T>
__global__ void __launch_bounds__(kThreads) gdn_diag_delta_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  const bool runs = !(first && transport);
  GDN_DDPROBE(0);      // segment 0 needs no transport run
  const T *vp = static_cast<const T *>(p.v), *bp = static_cast<const T *>(p.b);
  const T *cp = static_cast<const T *>(p.c), *betap = static_cast<const T *>(p.beta);
  // element (token t of this segment, s) of a [B][T][H][32] tensor
  auto at = [&](int t, int s) -> int64_t {
    return (((int64_t)bb * Tn + t0 + t) * H + hd) * 32 + s;
  };
  auto gate_at = [&](int t) -> int64_t { return ((int64_t)bb * Tn + t0 + t) * H + hd; };

  const float a2 = -expf(p.A_log[hd * kS + lane]) * kLog2e;   // row `lane`: d = 2^(g a2)
  const bool gate_sig = (p.opts & GDN_GATE_SIGMOID) != 0;
  const bool beta_sig = (p.opts & GDN_BETA_LOGITS) != 0;

  // the state column `lane`: zero, the initial state, or the identity column
  uint64_t h2[16];
  {
    const size_t srow = ((size_t)bb * H + hd) * kS * kD;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float x0 = 0.f, x1 = 0.f;
      if (transport) {
        x0 = (2 * i == lane) ? 1.f : 0.f;
        x1 = (2 * i + 1 == lane) ? 1.f : 0.f;
      } else if (first && p.h0) {
        x0 = p.h0[srow + (size_t)(2 * i) * kD + lane];
        x1 = p.h0[srow + (size_t)(2 * i + 1) * kD + lane];
      }
      h2[i] = pk2(x0, x1);
    }
  }

  // ---- staging: thread (warp w, lane s) handles tokens 8w .. 8w+7 of a tile ----
  float rb[8], rc[8], rg[8], rv[8], rbeta = 0.f;
  auto fetch = [&](int tt) {   // tile starting at segment token tt, into registers
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = tt + 8 * warp + i;
      const bool ok = t < len;
      rb[i] = ok ? ldf(bp + at(t, lane)) : 0.f;
      rc[i] = ok ? ldf(cp + at(t, lane)) : 0.f;
      rv[i] = ok ? ldf(vp + at(t, lane)) : 0.f;
      rg[i] = ok ? p.g[gate_at(t)] : 0.f;
    }
    const int tb = tt + 8 * warp + lane;
    rbeta = (lane < 8 && tb < len) ? ldf(betap + gate_at(tb)) : 0.f;
  };
  auto commit = [&](int buf, int tt) {   // registers -> shared tile `buf`
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int tl = 8 * warp + i;
      const bool ok = tt + tl < len;   // a padded token is an identity step
      const float g = gate_sig ? sigmoid(rg[i]) : rg[i];
      const float d = ok ? ex2(g * a2) : 1.f;
      sm.row[buf][0][tl][lane] = rb[i] * d;
      sm.row[buf][1][tl][lane] = d;
      sm.row[buf][2][tl][lane] = rb[i];
      sm.row[buf][3][tl][lane] = rc[i];
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
      float *out = transport ? &sm.rbuf[0][0] : &sm.obuf[0][0];
#pragma unroll 1
      for (int tl = 0; tl < kTile; ++tl) {
        const float *r_bd = sm.row[buf][0][tl], *r_d = sm.row[buf][1][tl];
        const float *r_b = sm.row[buf][2][tl], *r_c = sm.row[buf][3][tl];
        const float pred = dot32(r_bd, h2);              // hbar^T b, column `lane`
        const float vj = transport ? 0.f : sm.vt[buf][tl][lane];
        const float u = sm.bt[buf][tl] * (vj - pred);
        const uint64_t uu = pk2(u, u);
        const ulonglong2 *D2 = reinterpret_cast<const ulonglong2 *>(r_d);
        const ulonglong2 *B2 = reinterpret_cast<const ulonglong2 *>(r_b);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const ulonglong2 d = D2[i], bk = B2[i];
          h2[2 * i] = fma2(bk.x, uu, mul2(d.x, h2[2 * i]));
          h2[2 * i + 1] = fma2(bk.y, uu, mul2(d.y, h2[2 * i + 1]));
        }
        const float o = dot32(r_c, h2);
        if (tt + tl < len) out[(tt + tl) * 32 + lane] = o;
      }
    }
    if (it + 1 < ntiles) commit(buf ^ 1, tt + kTile);
    __syncthreads();
  }

  GDN_DDPROBE(1);
  // ---- the start state and the composition ----
  // M[s][k] (column k is transport lane k) over rows 0-1 of the first
  // buffer, X[s][j] over rows 2-3 (32 x 32 floats each)
  float (*Ms)[kS] = reinterpret_cast<float (*)[kS]>(&sm.row[0][0][0][0]);
  float (*Xs)[kD] = reinterpret_cast<float (*)[kD]>(&sm.row[0][2][0][0]);
  {
    float x[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float lo, hi;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(h2[i]));
      x[2 * i] = lo;
      x[2 * i + 1] = hi;
    }
    float(*dst)[32] = transport ? Ms : Xs;
    if (runs) {
#pragma unroll
      for (int s = 0; s < 32; ++s) dst[s][lane] = x[s];
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
  // h_start column `lane` (segment 0: M = I, X = its run, so nothing to add)
  float hs[32];
  const bool have_start = !first && sm.misc[2] != 0u;
  {
    const float *src = p.hend + (size_t)(ticket - (first ? 0u : (uint32_t)units)) * kS * kD;
#pragma unroll
    for (int s = 0; s < 32; ++s) hs[s] = have_start ? __ldcg(src + s * kD + lane) : 0.f;
  }
  // end state rows 16 w .. 16 w + 15: X + M h_start (segment 0: X)
  {
    uint64_t hs2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) hs2[i] = pk2(hs[2 * i], hs[2 * i + 1]);
    float *dst = p.hend + (size_t)ticket * kS * kD;
    float *fin = last && p.hN ? p.hN + ((size_t)bb * H + hd) * kS * kD : nullptr;
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
      const int s = 16 * warp + r;
      const float e = Xs[s][lane] + (first ? 0.f : dot32(Ms[s], hs2));
      __stcg(dst + s * kD + lane, e);
      if (fin) fin[s * kD + lane] = e;
    }
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) st_release_gpu(p.flags + ticket, tag);
  GDN_DDPROBE(3);

  // ---- outputs: o = o0 + r^T h_start, then the block epilogue ----
  {
    uint64_t hs2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) hs2[i] = pk2(hs[2 * i], hs[2 * i + 1]);
    const float dsk = p.D_skip ? p.D_skip[hd] : 0.f;
    T *op = static_cast<T *>(p.o);
#pragma unroll 1
    for (int t = warp; t < len; t += 2) {
      float o = sm.obuf[t][lane];
      if (!first) o += dot32(sm.rbuf[t], hs2);
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
  const int smem = (int)sizeof(Smem);
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
