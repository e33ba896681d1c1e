// Prologue of the HyMo GDN block: causal depthwise conv1d followed by SiLU
// ("Model Architecture Walkthrough", section 5.4.1: a depthwise Conv1d with
// d_conv = 4 taps, padding d_conv - 1 and the tail trimmed, i.e. causal;
// section 5.5, step 2: SiLU after the conv).  Per batch row n, channel ch and
// token t, with x[t] for t < 0 taken from the optional prefix (else zero):
//
//   y[n, t, ch] = silu( sum_{k < K} w[ch, k] * x[n, t - (K - 1) + k, ch] ),   silu(z) = z / (1 + e^-z)
//
// The pass is bound by HBM bandwidth: every input element is read once from
// HBM (the K-1 token halo of a run is the previous run's data, an L1/L2 hit)
// and every output element written once.  A thread owns a vector of 4
// channels (8 bytes of bf16 or 16 of fp32) over a run of 8 tokens: it issues all
// 8 + K-1 loads of its window at once, so that enough bytes are in flight to
// cover the HBM latency, then produces the 8 outputs.  Consecutive lanes own
// consecutive vectors, so each warp-wide load or store is 256 or 512
// contiguous bytes of one token row.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRun = 8;          // tokens per thread
constexpr int kConvThreads = 256;
constexpr int kVecWarps = 8;     // token runs per CTA (one per warp)
// resident CTAs per SM: bf16 fits 64 registers, fp32 needs 80
template <typename T> constexpr int kConvBlocks() { return sizeof(T) == 2 ? 4 : 3; }

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 4;   // 4 channels: one 8-byte vector
  using Raw = uint2;
  __device__ static void unpack(const Raw r, float (&x)[N]) {
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xffff0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xffff0000u);
  }
  __device__ static void store(void *p, const float (&x)[N]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    *reinterpret_cast<uint2 *>(p) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
  }
};
template <> struct Vec<float> {
  static constexpr int N = 4;   // 4 channels: one 16-byte vector
  using Raw = uint4;
  __device__ static void unpack(const Raw r, float (&x)[N]) {
    x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
  }
  __device__ static void store(void *p, const float (&x)[N]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};

struct ConvParams {
  const void *x, *x_prev;
  const float *w;
  void *y, *x_tail;
  int32_t batch, seq_len, channels, taps;
};

// silu(z) = z / (1 + e^-z) = z * rcp(1 + 2^(-z log2 e)) on the hardware's
// approximate 2^x and reciprocal (flush-to-zero forms: no denormal fix-ups).
// Large negative z gives 2^(+big) = inf, rcp(inf) = 0 and silu -> -0.
__device__ __forceinline__ float silu(float z) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return z * r;
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, kConvBlocks<T>())
gdn_conv_silu_kernel(const ConvParams p) {
  using V = Vec<T>;
  constexpr int N = V::N;
  const int lane = threadIdx.x & 31, wrp = threadIdx.x >> 5;
  const int cbase = blockIdx.x * 32 * N;              // first channel of this CTA
  const int c0 = cbase + lane * N;                    // first channel of this thread
  const int t0 = (blockIdx.y * kVecWarps + wrp) * kRun;
  const int n = blockIdx.z;
  const int C = p.channels, L = p.seq_len;
  const size_t e = sizeof(T);
  const unsigned char *x = static_cast<const unsigned char *>(p.x);
  auto row = [&](int t) { return ((size_t)n * L + t) * C + c0; };

  // the CTA's weights, staged tap-major ([K][32 N]) with one coalesced pass
  __shared__ float4 s_w4[K * 32 * N / 4];
  float *s_w = reinterpret_cast<float *>(s_w4);
  for (int i = threadIdx.x; i < 32 * N * K; i += kConvThreads) {
    const int ch = i / K, k = i % K;
    s_w[k * 32 * N + ch] = cbase + ch < C ? __ldg(p.w + (size_t)(cbase + ch) * K + k) : 0.f;
  }
  __syncthreads();
  if (c0 >= C || t0 >= L) return;
  float w[K][N];
#pragma unroll
  for (int k = 0; k < K; ++k)
#pragma unroll
    for (int j4 = 0; j4 < N / 4; ++j4) {
      const float4 q = s_w4[(k * 32 * N + lane * N) / 4 + j4];
      w[k][4 * j4] = q.x; w[k][4 * j4 + 1] = q.y; w[k][4 * j4 + 2] = q.z; w[k][4 * j4 + 3] = q.w;
    }

  // raw[r] holds x[t0 - (K - 1) + r]: the halo, then this run's tokens, all
  // loads issued before the first use.  Runs away from the sequence ends (the
  // common case) load without per-token tests, from one base pointer.
  constexpr int R = kRun + K - 1;
  typename V::Raw raw[R];
  const size_t rstride = (size_t)C * e;                 // bytes between tokens
  if (t0 >= K - 1 && t0 + kRun <= L) {
    const unsigned char *xb = x + row(t0 - (K - 1)) * e;
#pragma unroll
    for (int r = 0; r < R; ++r) raw[r] = *reinterpret_cast<const typename V::Raw *>(xb + r * rstride);
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int t = t0 - (K - 1) + r;
      if (t >= 0 && t < L) {
        raw[r] = *reinterpret_cast<const typename V::Raw *>(x + row(t) * e);
      } else if (t < 0 && p.x_prev) {   // prefix: the K-1 inputs before token 0
        raw[r] = *reinterpret_cast<const typename V::Raw *>(
            static_cast<const unsigned char *>(p.x_prev) +
            (((size_t)n * (K - 1) + (K - 1) + t) * C + c0) * e);
      } else {
        raw[r] = typename V::Raw{};
      }
    }
  }
  const int t_end = t0 + kRun < L ? t0 + kRun : L;
  // every input unpacked once; output q reads inputs q .. q + K - 1
  float xf[R][N];
#pragma unroll
  for (int r = 0; r < R; ++r) V::unpack(raw[r], xf[r]);
  unsigned char *yb = static_cast<unsigned char *>(p.y) + row(t0) * e;
  const bool full = t_end == t0 + kRun;
#pragma unroll
  for (int q = 0; q < kRun; ++q) {
    float out[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
      float a = 0.f;
#pragma unroll
      for (int k = 0; k < K; ++k) a = fmaf(w[k][j], xf[q + k][j], a);
      out[j] = silu(a);
    }
    if (full || t0 + q < t_end) V::store(yb + q * rstride, out);
  }
  // the last K-1 inputs (prefix of the next call): written by the run that
  // holds them, which is the run ending at the last token
  if (p.x_tail && t_end == L) {
    // inputs t_end - (K - 1) + k, k < K - 1, sit at raw[t_end - t0 + k]
    const int base = t_end - t0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int k = r - base;
      if (k >= 0 && k < K - 1)
        *reinterpret_cast<typename V::Raw *>(static_cast<unsigned char *>(p.x_tail) +
                                             (((size_t)n * (K - 1) + k) * C + c0) * e) = raw[r];
    }
  }
}

template <typename T, int K>
cudaError_t launch_k(const ConvParams &p, cudaStream_t s) {
  constexpr int N = Vec<T>::N;
  const dim3 grid((p.channels / N + 31) / 32, (p.seq_len + kRun * kVecWarps - 1) / (kRun * kVecWarps),
                  p.batch);
  gdn_conv_silu_kernel<T, K><<<grid, kConvThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const ConvParams &p, cudaStream_t s) {
  switch (p.taps) {
    case 1: return launch_k<T, 1>(p, s);
    case 2: return launch_k<T, 2>(p, s);
    case 3: return launch_k<T, 3>(p, s);
    case 4: return launch_k<T, 4>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

bool aligned16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t u = reinterpret_cast<uintptr_t>(a), v = reinterpret_cast<uintptr_t>(b);
  return u < v + nb && v < u + na;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_conv_silu(const void *x, const float *w, const void *x_prev, void *y,
                                    void *x_tail, int32_t batch, int32_t seq_len,
                                    int32_t channels, int32_t taps, gdn_dtype dtype,
                                    void *stream) {
  using namespace gdn;
  if (batch <= 0 || seq_len <= 0 || channels <= 0 || taps <= 0) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (taps > 4) return GDN_ERR_UNSUPPORTED;
  if (channels % 4) return GDN_ERR_UNSUPPORTED;
  if (batch > 65535) return GDN_ERR_UNSUPPORTED;
  if (!x || !w || !y) return GDN_ERR_INVALID_ARG;
  if (x_tail && taps == 1) return GDN_ERR_INVALID_ARG;   // no prefix to keep
  const void *ptrs[] = {x, w, x_prev, y, x_tail};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  const size_t e = dtype == GDN_F32 ? 4 : 2;
  const size_t b_x = (size_t)batch * seq_len * channels * e;
  const size_t b_w = (size_t)channels * taps * 4;
  const size_t b_p = (size_t)batch * (taps - 1) * channels * e;
  // Outputs overlap no input: other runs read x and x_prev as their halos
  // while the run that ends at seq_len writes x_tail.
  const struct { const void *p; size_t n; } in[] = {{x, b_x}, {w, b_w}, {x_prev, b_p}};
  for (const auto &r : in) {
    if (overlaps(y, b_x, r.p, r.n)) return GDN_ERR_INVALID_ARG;
    if (overlaps(x_tail, b_p, r.p, r.n)) return GDN_ERR_INVALID_ARG;
  }
  if (overlaps(x_tail, b_p, y, b_x)) return GDN_ERR_INVALID_ARG;

  ConvParams p;
  p.x = x; p.x_prev = x_prev; p.w = w; p.y = y; p.x_tail = x_tail;
  p.batch = batch; p.seq_len = seq_len; p.channels = channels; p.taps = taps;
  const cudaError_t err = dtype == GDN_F32 ? launch_t<float>(p, (cudaStream_t)stream)
                                           : launch_t<__nv_bfloat16>(p, (cudaStream_t)stream);
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
