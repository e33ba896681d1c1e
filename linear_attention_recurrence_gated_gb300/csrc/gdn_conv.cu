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
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

using namespace ptx;
constexpr uint64_t kConvWaitNs = 2000000000ull;  // bounded TMA waits: 2 s

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

// ---- two fp32 lanes in one 64-bit register (Blackwell's packed fp32 FMA/MUL/ADD:
// each lane is an ordinary IEEE fp32 operation) ----
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
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// silu on a pair: z * rcp(1 + 2^(-z log2 e)), the scale, the 1 + and the
// final product packed; 2^x and the reciprocal per lane (as in silu above)
__device__ __forceinline__ void silu2(uint64_t z, float &o0, float &o1) {
  float t0, t1, e0, e1, r0, r1;
  upk2(mul2(z, pk2(-1.4426950408889634f, -1.4426950408889634f)), t0, t1);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
  float s0, s1;
  upk2(add2(pk2(e0, e1), pk2(1.f, 1.f)), s0, s1);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(s0));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(s1));
  upk2(mul2(z, pk2(r0, r1)), o0, o1);
}

// ---- TMA-staged variant (token rows of C * sizeof(T) bytes a multiple of 16) ----
// A persistent CTA owns one block of 32 channel vectors for the whole call and
// walks (batch row, 64-token) tiles of it.  One thread loads each tile, with
// its K-1 token halo, as one 3-D TMA box into a shared-memory stage; the box
// of the next tile is in flight while the current one computes.  Rows before
// token 0 and past the end, and channels past C, arrive as zeros (the box may
// start at a negative token coordinate); the prefix rows of a call's first
// tile are then overwritten from x_prev.
constexpr int kTileTok = kRun * kVecWarps;   // 64 tokens per tile

template <typename T, int K>
struct TmaTile {
  static constexpr int VB = sizeof(typename Vec<T>::Raw);   // bytes per lane vector
  static constexpr int ROWS = kTileTok + K - 1;              // tile + halo
  static constexpr int ROWB = 32 * VB;                       // bytes per staged token row
  static constexpr int STAGE = (ROWS * ROWB + 1023) / 1024 * 1024;
  static constexpr int NS = 2;                               // stages (3 measured no faster)
  static constexpr int BYTES = NS * STAGE + 1024;            // + alignment slack
};

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, kConvBlocks<T>())
gdn_conv_silu_tma_kernel(const ConvParams p, const __grid_constant__ CUtensorMap tmap_x) {
  using V = Vec<T>;
  using TL = TmaTile<T, K>;
  constexpr int N = V::N, VB = TL::VB, ROWS = TL::ROWS, ROWB = TL::ROWB;
  extern __shared__ __align__(1024) unsigned char sraw[];
  unsigned char *sx = sraw + ((1024u - (smem_u32(sraw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full_bar[TL::NS];
  __shared__ int s_fail;
  const int tid = threadIdx.x, lane = tid & 31, wrp = tid >> 5;
  const int cbase = blockIdx.x * 32 * N;              // first channel of this CTA
  const int c0 = cbase + lane * N;                    // first channel of this lane
  const bool lane_ok = c0 < p.channels;
  const int C = p.channels, L = p.seq_len;
  const size_t e = sizeof(T);
  const int ntb = (L + kTileTok - 1) / kTileTok;
  const int ntile = ntb * p.batch;
  const uint32_t bar0 = smem_u32(&full_bar[0]);

  // the CTA's weights, staged tap-major ([K][32 N]) with one coalesced pass
  __shared__ float4 s_w4[K * 32 * N / 4];
  float *s_w = reinterpret_cast<float *>(s_w4);
  for (int i = tid; i < 32 * N * K; i += kConvThreads) {
    const int ch = i / K, k = i % K;
    s_w[k * 32 * N + ch] = cbase + ch < C ? __ldg(p.w + (size_t)(cbase + ch) * K + k) : 0.f;
  }
  if (tid == 0) {
    for (int b = 0; b < TL::NS; ++b) mbar_init(bar0 + 8 * b, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  float w[K][N];
#pragma unroll
  for (int k = 0; k < K; ++k)
#pragma unroll
    for (int j4 = 0; j4 < N / 4; ++j4) {
      const float4 q = s_w4[(k * 32 * N + lane * N) / 4 + j4];
      w[k][4 * j4] = q.x; w[k][4 * j4 + 1] = q.y; w[k][4 * j4 + 2] = q.z; w[k][4 * j4 + 3] = q.w;
    }
  static_assert(N == 4, "two channel pairs per lane vector");
  uint64_t wp[K][2];   // weights of channel pairs (0,1) and (2,3)
#pragma unroll
  for (int k = 0; k < K; ++k) {
    wp[k][0] = pk2(w[k][0], w[k][1]);
    wp[k][1] = pk2(w[k][2], w[k][3]);
  }
  auto issue = [&](int tile, int b) {   // one thread
    const int n = tile / ntb, t0 = (tile % ntb) * kTileTok;
    mbar_arrive_expect_tx(bar0 + 8 * b, (uint32_t)(ROWS * ROWB));
    tma_load_3d(smem_u32(sx) + b * TL::STAGE, &tmap_x, cbase, t0 - (K - 1), n, bar0 + 8 * b);
  };

  constexpr int NS = TL::NS;
  const int gy = (int)gridDim.y;
  int tile = blockIdx.y;
  if (tid == 0)
    for (int j = 0; j < NS - 1; ++j)
      if (tile + j * gy < ntile) issue(tile + j * gy, j);
  for (int it = 0; tile < ntile; ++it, tile += gy) {
    const int b = it % NS;
    // the box NS-1 tiles ahead goes to the stage every thread finished reading
    // before the barrier that closed the previous iteration
    const bool ahead = tile + (NS - 1) * gy < ntile;
    if (tid == 0 && ahead) issue(tile + (NS - 1) * gy, (it + NS - 1) % NS);
    if (!mbar_wait_bounded(bar0 + 8 * b, (it / NS) & 1, kConvWaitNs)) s_fail = 1;
    const int n = tile / ntb, tt0 = (tile % ntb) * kTileTok;
    unsigned char *st = sx + b * TL::STAGE;
    // a sequence's first tile: the K-1 rows before token 0 from the prefix
    if (tt0 == 0 && p.x_prev && lane_ok && wrp < K - 1)
      *reinterpret_cast<typename V::Raw *>(st + wrp * ROWB + lane * VB) =
          *reinterpret_cast<const typename V::Raw *>(
              static_cast<const unsigned char *>(p.x_prev) +
              (((size_t)n * (K - 1) + wrp) * C + c0) * e);
    __syncthreads();
    if (s_fail) {   // a box never arrived: leave after the ones still in flight
      if (tid == 0)
        for (int j = 1; j < NS; ++j)
          if (tile + j * gy < ntile)
            mbar_wait_bounded(bar0 + 8 * ((it + j) % NS), ((it + j) / NS) & 1, kConvWaitNs);
      break;
    }
    const int t0 = tt0 + wrp * kRun;
    if (lane_ok && t0 < L) {
      const unsigned char *rb = st + wrp * kRun * ROWB + lane * VB;
      constexpr int R = kRun + K - 1;
      uint64_t xp[R][2];   // channel pairs of x[t0 - (K - 1) + r]
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float f[N];
        V::unpack(*reinterpret_cast<const typename V::Raw *>(rb + r * ROWB), f);
        xp[r][0] = pk2(f[0], f[1]);
        xp[r][1] = pk2(f[2], f[3]);
      }
      const int t_end = t0 + kRun < L ? t0 + kRun : L;
      const size_t rstride = (size_t)C * e;
      unsigned char *yb = static_cast<unsigned char *>(p.y) + (((size_t)n * L + t0) * C + c0) * e;
#pragma unroll
      for (int q = 0; q < kRun; ++q) {
        float out[N];
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          uint64_t a = mul2(wp[0][pr], xp[q][pr]);
#pragma unroll
          for (int k = 1; k < K; ++k) a = fma2(wp[k][pr], xp[q + k][pr], a);
          silu2(a, out[2 * pr], out[2 * pr + 1]);
        }
        if (t0 + q < t_end) V::store(yb + q * rstride, out);
      }
      // the last K-1 inputs (prefix of the next call), by the warp whose run
      // ends at the last token: input t_end - (K-1) + k is row t_end - t0 + k
      if (p.x_tail && t_end == L) {
#pragma unroll
        for (int k = 0; k < K - 1; ++k)
          *reinterpret_cast<typename V::Raw *>(static_cast<unsigned char *>(p.x_tail) +
                                               (((size_t)n * (K - 1) + k) * C + c0) * e) =
              *reinterpret_cast<const typename V::Raw *>(rb + (t_end - t0 + k) * ROWB);
      }
    }
    // every thread is done with this stage (and its prefix rows, written by
    // the generic proxy) before a box is issued into it again
    fence_proxy_async_smem();
    __syncthreads();
  }
}

// x as a [batch][tokens][channels] tensor map; box = 32 lane vectors x (64 + K - 1) tokens x 1 row.
template <typename T, int K>
bool make_conv_tmap(CUtensorMap *m, const ConvParams &p) {
  tc::EncodeTiledFn enc = tc::encode_fn();
  const size_t e = sizeof(T);
  if (!enc || ((size_t)p.channels * e) % 16 != 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)p.channels, (cuuint64_t)p.seq_len, (cuuint64_t)p.batch};
  const cuuint64_t strides[2] = {(cuuint64_t)p.channels * e, (cuuint64_t)p.channels * e * p.seq_len};
  const cuuint32_t box[3] = {(cuuint32_t)(32 * Vec<T>::N), (cuuint32_t)TmaTile<T, K>::ROWS, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
             const_cast<void *>(p.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int K>
cudaError_t launch_k(const ConvParams &p, cudaStream_t s) {
  constexpr int N = Vec<T>::N;
  const int cblocks = (p.channels / N + 31) / 32;
  CUtensorMap tm;
  if (make_conv_tmap<T, K>(&tm, p)) {
    // TMA-staged persistent kernel: one wave of kConvBlocks CTAs per SM
    static int sms = 0;
    if (sms == 0) {
      int dev = 0, v = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return cudaErrorInvalidDevice;
      sms = v;
    }
    using TL = TmaTile<T, K>;
    cudaError_t err = cudaFuncSetAttribute(gdn_conv_silu_tma_kernel<T, K>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, TL::BYTES);
    if (err != cudaSuccess) return err;
    const int64_t ntile = (int64_t)((p.seq_len + kTileTok - 1) / kTileTok) * p.batch;
    int64_t per = ((int64_t)sms * kConvBlocks<T>() + cblocks - 1) / cblocks;
    if (per > ntile) per = ntile;
    if (per > 65535) per = 65535;
    gdn_conv_silu_tma_kernel<T, K><<<dim3(cblocks, (unsigned)per, 1), kConvThreads, TL::BYTES, s>>>(p, tm);
    return cudaGetLastError();
  }
  // token rows not 16-byte multiples: one 8-token run per warp, loads from registers
  const dim3 grid(cblocks, (p.seq_len + kRun * kVecWarps - 1) / (kRun * kVecWarps), p.batch);
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
