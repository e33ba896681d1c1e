// Pieces shared by the tensor-core kernels: swizzled tile addressing, bounded
// mbarrier waits, TMA tensor-map encoding and the optional phase-timing stamps.
#pragma once

#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace tc {

using namespace ptx;

#ifdef GDN_PHASE_PROBE
// Phase timing build only: clock stamps of CTA (0,0,0), [warp][chunk][phase].
static __device__ unsigned long long g_phase_probe[32 * 64 * 16];
#define GDN_PHASE(ph)                                                                      \
  do {                                                                                     \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && lane == 0 && c >= 0 &&    \
        c < 64 && warp < 32)                                                               \
      ::gdn::tc::g_phase_probe[(warp * 64 + c) * 16 + (ph)] = clock64();                   \
  } while (0)
// Any value into slot [w][cc][ph] (thread-agnostic; used by single-thread roles).
#define GDN_PROBE_AT(w, cc, ph, val)                                                       \
  do {                                                                                     \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (cc) >= 0 && (cc) < 64 && \
        (w) >= 0 && (w) < 32)                                                              \
      ::gdn::tc::g_phase_probe[((w) * 64 + (cc)) * 16 + (ph)] = (val);                     \
  } while (0)
#else
#define GDN_PHASE(ph) \
  do {                \
  } while (0)
#define GDN_PROBE_AT(w, cc, ph, val) \
  do {                               \
  } while (0)
#endif

constexpr int kDvt = 64;  // value columns per CTA
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// Byte address of element (row, col) of a bf16 tile stored as [64][64]
// sub-tiles of 128-byte rows with the 128-byte swizzle (16-byte granule index
// XOR row mod 8, the layout TMA writes with SWIZZLE_128B); SUB_STRIDE is the
// distance between the sub-tiles of consecutive 64-column groups.
template <int SUB_STRIDE>
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int col) {
  return base + (col >> 6) * SUB_STRIDE + row * 128 +
         ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1);
}
__device__ __forceinline__ uint32_t qk_addr(uint32_t base, int row, int col) {
  return swz<16384>(base, row, col);
}
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int col) {
  return swz<8192>(base, row, col);
}

struct Shared {
  volatile int *abort_flag;
};

#ifdef GDN_PHASE_PROBE
// Phase timing build only: try_wait calls per warp of CTA (0,0,0).
static __device__ unsigned long long g_wait_iters[32];
#define GDN_COUNT_WAIT(it)                                                                 \
  do {                                                                                     \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (threadIdx.x & 31) == 0)  \
      atomicAdd(&::gdn::tc::g_wait_iters[threadIdx.x >> 5], (unsigned long long)(it));     \
  } while (0)
#else
#define GDN_COUNT_WAIT(it) \
  do {                     \
  } while (0)
#endif

// Slow path of role_wait, one shared copy: keep polling (try_wait suspends the
// thread until the phase completes or a hardware time limit passes), give up
// after kWaitTimeoutNs or once another role has raised the abort flag.
static __device__ __noinline__ bool role_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                   DeviceStatus *status, int n, int h, uint32_t where) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) {
      GDN_COUNT_WAIT(it);
      return true;
    }
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        report(status, GDN_ERR_TIMEOUT, (uint32_t)n, (uint32_t)h, where);
        return false;
      }
    }
  }
}

// Wait for phase `parity` of the mbarrier at `bar`; false once the wait gave
// up (GDN_ERR_TIMEOUT recorded) or the CTA is aborting.
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, const Shared &S,
                                          const FwdParams &p, int n, int h, uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  return role_wait_slow(bar, parity, S.abort_flag, p.status, n, h, where);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Token rows of a tensor map: all of them, or under GDN_DEBUG_CHECKS no more
// than the buffer's extent holds, so that no TMA box reaches past it (at least
// one row, for a valid map: a block whose rows pass the extent returns before
// its first copy).
inline int64_t tmap_rows(const FwdParams &p, int64_t tokens, int64_t extent, int cols) {
  if (!(p.flags & GDN_DEBUG_CHECKS)) return tokens;
  const int64_t r = extent / ((int64_t)p.num_heads * cols);
  return r < 1 ? 1 : r < tokens ? r : tokens;
}

// [tokens][heads][cols] bf16 viewed as a 3-D tensor; box = 64 cols x 1 head x
// box_rows tokens (the chunk: 64, or 32 / 128 for the chunk-size variants).
inline bool make_tmap(CUtensorMap *m, const void *ptr, int cols, int heads, int64_t tokens,
                      int box_rows = 64) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * heads * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace gdn
