// One recurrent step of the gated delta rule per (sequence, head): the
// token-by-token form of the operation, for incremental inference with the
// state carried between calls.  With H = S^T (dk x dv, fp32):
//
//   u  = beta (v - alpha H^T k)        (the delta: target minus decayed read)
//   H' = alpha H + k u^T               (= alpha (I - beta k k^T) H + beta k v^T)
//   o  = H'^T q                        (the read after the write)
//
// (gated delta rule, Yang et al. arXiv 2412.06464; decay alpha = exp(g),
// "Model Architecture Walkthrough", section 5.2.1; the per-token step of the
// recurrence, same page, section 5.5, step 5.)
//
// The step moves the whole state through HBM once in each direction and does
// 4 dk dv flops on it, so it is bound by HBM bandwidth.  One CTA of 256 threads
// owns a 32-column slice of one head's state: thread t holds columns
// 4 (t % 8) .. +3 of rows t / 8 + 32 m (m < dk / 32) in registers, loaded and
// stored as 16-byte vectors (each row slice is 128 contiguous bytes).  The two
// column sums (H^T k and H'^T q) reduce over the row groups with warp
// shuffles and one shared-memory pass.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecCols = 32;  // value columns per CTA

struct DecodeParams {
  const void *q, *k, *v, *beta;
  const float *g;
  const float *s_in;
  float *s_out;
  void *o;
  int32_t num_heads, dk, dv;
  uint32_t flags;
};

__device__ __forceinline__ float ld(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }

template <typename T, int DKT>
__global__ void __launch_bounds__(kDecThreads)
gdn_decode_kernel(const DecodeParams p) {
  constexpr int RPT = DKT / 32;  // rows of the state per thread
  __shared__ float sk[DKT], sq[DKT], sv[kDecCols], su[kDecCols];
  __shared__ float part[8][kDecCols];
  __shared__ float snorm[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv;
  const int cg = tid & 7, rg = tid >> 3;   // column group (4 columns), row group
  const int col = tile * kDecCols + 4 * cg;
  const size_t head = (size_t)n * H + h;

  const T *q = static_cast<const T *>(p.q) + head * DKT;
  const T *k = static_cast<const T *>(p.k) + head * DKT;
  const T *v = static_cast<const T *>(p.v) + head * dv + tile * kDecCols;

  // ---- the state slice (issued first: it is the bulk of the traffic) ----
  float4 hv[RPT];
  const size_t sbase = head * (size_t)DKT * dv;
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    const int i = rg + 32 * m;
    hv[m] = p.s_in ? *reinterpret_cast<const float4 *>(p.s_in + sbase + (size_t)i * dv + col)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- q, k (optionally L2-normalised), v, alpha, beta ----
  for (int i = tid; i < DKT; i += kDecThreads) {
    sk[i] = ld(k, i);
    sq[i] = ld(q, i);
  }
  if (tid < kDecCols) sv[tid] = ld(v, tid);
  const float alpha = expf(p.g[head]);
  const float beta = ld(static_cast<const T *>(p.beta), head);
  __syncthreads();
  if (p.flags & GDN_QK_L2NORM) {
    if (warp < 2) {
      const float *x = warp == 0 ? sk : sq;
      float ss = 0.f;
      for (int i = lane; i < DKT; i += 32) ss = fmaf(x[i], x[i], ss);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) snorm[warp] = rsqrtf(ss + 1e-6f);
    }
    __syncthreads();
    for (int i = tid; i < DKT; i += kDecThreads) {
      sk[i] *= snorm[0];
      sq[i] *= snorm[1];
    }
    __syncthreads();
  }

  // ---- H^T k over this thread's rows, then over the 32 row groups ----
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    const float ki = sk[rg + 32 * m];
    a.x = fmaf(ki, hv[m].x, a.x);
    a.y = fmaf(ki, hv[m].y, a.y);
    a.z = fmaf(ki, hv[m].z, a.z);
    a.w = fmaf(ki, hv[m].w, a.w);
  }
  // the four row groups of a warp share a column group: lanes cg, cg+8, cg+16, cg+24
#pragma unroll
  for (int off = 8; off < 32; off <<= 1) {
    a.x += __shfl_xor_sync(0xffffffffu, a.x, off);
    a.y += __shfl_xor_sync(0xffffffffu, a.y, off);
    a.z += __shfl_xor_sync(0xffffffffu, a.z, off);
    a.w += __shfl_xor_sync(0xffffffffu, a.w, off);
  }
  if (lane < 8) *reinterpret_cast<float4 *>(&part[warp][4 * lane]) = a;
  __syncthreads();
  if (tid < kDecCols) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[w][tid];
    su[tid] = beta * (sv[tid] - alpha * s);  // u = beta (v - alpha H^T k)
  }
  __syncthreads();

  // ---- H' = alpha H + k u^T (stored), then H'^T q ----
  const float4 u = *reinterpret_cast<const float4 *>(&su[4 * cg]);
  float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    const int i = rg + 32 * m;
    const float ki = sk[i], qi = sq[i];
    float4 x = hv[m];
    x.x = fmaf(alpha, x.x, ki * u.x);
    x.y = fmaf(alpha, x.y, ki * u.y);
    x.z = fmaf(alpha, x.z, ki * u.z);
    x.w = fmaf(alpha, x.w, ki * u.w);
    *reinterpret_cast<float4 *>(p.s_out + sbase + (size_t)i * dv + col) = x;
    b.x = fmaf(qi, x.x, b.x);
    b.y = fmaf(qi, x.y, b.y);
    b.z = fmaf(qi, x.z, b.z);
    b.w = fmaf(qi, x.w, b.w);
  }
#pragma unroll
  for (int off = 8; off < 32; off <<= 1) {
    b.x += __shfl_xor_sync(0xffffffffu, b.x, off);
    b.y += __shfl_xor_sync(0xffffffffu, b.y, off);
    b.z += __shfl_xor_sync(0xffffffffu, b.z, off);
    b.w += __shfl_xor_sync(0xffffffffu, b.w, off);
  }
  // every thread has read part[] above (before the second __syncthreads)
  if (lane < 8) *reinterpret_cast<float4 *>(&part[warp][4 * lane]) = b;
  __syncthreads();
  if (tid < kDecCols) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[w][tid];
    store_out(static_cast<T *>(p.o) + head * dv + tile * kDecCols + tid, s);
  }
}

template <typename T>
cudaError_t launch_t(const DecodeParams &p, int num_seqs, cudaStream_t stream) {
  const dim3 grid(p.dv / kDecCols, p.num_heads, num_seqs);
  switch (p.dk) {
    case 32: gdn_decode_kernel<T, 32><<<grid, kDecThreads, 0, stream>>>(p); break;
    case 64: gdn_decode_kernel<T, 64><<<grid, kDecThreads, 0, stream>>>(p); break;
    case 128: gdn_decode_kernel<T, 128><<<grid, kDecThreads, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

bool aligned16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_decode(const void *q, const void *k, const void *v, const float *g,
                                 const void *beta, const float *state_in, float *state_out,
                                 void *o, int32_t num_seqs, int32_t num_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, gdn_dtype dtype,
                                 uint32_t flags, void *stream) {
  using namespace gdn;
  if (num_seqs <= 0 || num_heads <= 0 || head_dim_k <= 0 || head_dim_v <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)GDN_QK_L2NORM) return GDN_ERR_INVALID_ARG;
  if (!(head_dim_k == 32 || head_dim_k == 64 || head_dim_k == 128)) return GDN_ERR_UNSUPPORTED;
  if (head_dim_v < 32 || head_dim_v > 256 || head_dim_v % 32) return GDN_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_heads > 65535) return GDN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !g || !beta || !state_out || !o) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, state_in, state_out, o};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;

  // aliasing: outputs overlap no input, except state_out == state_in exactly
  const size_t e = dtype == GDN_F32 ? 4 : 2;
  const size_t rows = (size_t)num_seqs * num_heads;
  const size_t b_qk = rows * head_dim_k * e, b_v = rows * head_dim_v * e;
  const size_t b_g = rows * 4, b_beta = rows * e;
  const size_t b_state = rows * head_dim_k * head_dim_v * 4;
  struct Range { const void *p; size_t n; };
  const Range inputs[] = {{q, b_qk}, {k, b_qk}, {v, b_v}, {g, b_g}, {beta, b_beta}};
  for (const Range &r : inputs) {
    if (overlaps(o, b_v, r.p, r.n)) return GDN_ERR_INVALID_ARG;
    if (overlaps(state_out, b_state, r.p, r.n)) return GDN_ERR_INVALID_ARG;
  }
  if (overlaps(o, b_v, state_out, b_state) || overlaps(o, b_v, state_in, b_state))
    return GDN_ERR_INVALID_ARG;
  if (state_in && state_in != state_out && overlaps(state_in, b_state, state_out, b_state))
    return GDN_ERR_INVALID_ARG;

  DecodeParams p;
  p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g;
  p.s_in = state_in; p.s_out = state_out; p.o = o;
  p.num_heads = num_heads; p.dk = head_dim_k; p.dv = head_dim_v; p.flags = flags;
  const cudaError_t err =
      dtype == GDN_F32 ? launch_t<float>(p, num_seqs, (cudaStream_t)stream)
                       : launch_t<__nv_bfloat16>(p, num_seqs, (cudaStream_t)stream);
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
