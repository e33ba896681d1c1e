// The two small kernels of a split sequence (GDN_SEQ_SPLIT, head_dim_k 128)
// that follow the segments' chain launch: the composition of the segments'
// affine state maps, H_(s+1) = M_s H_s + X_s, one step per launch in segment
// order, and the correction of the later segments' outputs, o += r H_s.
// ("Optimization Quartet", Triton GDN kernel section 3.2, names the
// inter-chunk carry as the serial part of the chunked form; the maps and
// their composition are what lets the segments run at the same time.)
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kSplitDK = 128;

// One step of the composition, H_(s+1) = M_s H_s + X_s (fp32; M_s is dk x dk;
// the last step gives the caller's final state), for a block of 32 rows and
// 32 value columns of one (sequence, head): the CTA stages its 32 rows of M_s
// and the 32 columns of H_s in shared memory (every load in flight at once),
// then lane = column and each warp takes 4 rows.  grid: (dv / 32 * dk / 32,
// H, N).
__global__ void __launch_bounds__(256) seg_compose_kernel(const FwdParams p, int s) {
  __shared__ __align__(16) float ms[32][kSplitDK + 4];
  __shared__ __align__(16) float hs[kSplitDK][32];
  const int nc = p.dv / 32;
  const int c0 = (blockIdx.x % nc) * 32, r0 = (blockIdx.x / nc) * 32;
  const int h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv, S = p.seg_count, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const size_t unit = ((size_t)n * S + s) * H + h;
  const float *M = p.seg_m + unit * kSplitDK * kSplitDK;
  const float *Hs = p.seg_state + unit * kSplitDK * dv;
  const float *X = p.seg_x + unit * kSplitDK * dv;
  // segment s + 1, or after the last segment the caller's final state
  float *Hn = s + 1 < S ? p.seg_state + (unit + H) * kSplitDK * dv
                        : p.sN ? p.sN + ((size_t)n * H + h) * kSplitDK * dv : nullptr;
  if (Hn == nullptr) return;  // uniform over the CTA
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int q = tid + 256 * e;                  // 1024 float4 of each tile
    const int mr = q / (kSplitDK / 4), mc = q % (kSplitDK / 4);
    *reinterpret_cast<float4 *>(&ms[mr][4 * mc]) =
        *reinterpret_cast<const float4 *>(M + (size_t)(r0 + mr) * kSplitDK + 4 * mc);
    const int hr = q / 8, hc = q % 8;
    *reinterpret_cast<float4 *>(&hs[hr][4 * hc]) =
        *reinterpret_cast<const float4 *>(Hs + (size_t)hr * dv + c0 + 4 * hc);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * warp + i;
    float a0 = X[(size_t)(r0 + r) * dv + c0 + lane], a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
    for (int q = 0; q < kSplitDK / 4; ++q) {
      const float4 m = *reinterpret_cast<const float4 *>(&ms[r][4 * q]);
      a0 = fmaf(m.x, hs[4 * q][lane], a0);
      a1 = fmaf(m.y, hs[4 * q + 1][lane], a1);
      a2 = fmaf(m.z, hs[4 * q + 2][lane], a2);
      a3 = fmaf(m.w, hs[4 * q + 3][lane], a3);
    }
    Hn[(size_t)(r0 + r) * dv + c0 + lane] = (a0 + a1) + (a2 + a3);
  }
}

// The correction of a split sequence's later segments: o[t] += r[t] H_s for
// every token t of segment s >= 1 (r [tokens][H][dk] and H_s in bf16 on
// mma.sync, fp32 sums, o read and written in bf16).  A CTA takes up to
// kCorrBlocks blocks of 64 tokens inside one segment and 64 NT value columns
// of one (sequence, head), so that each row of r is read once per NT column
// tiles: H_s is converted once; the next block's rows of r are fetched
// (cp.async) and its o values loaded into registers while the current block
// is computed.  Warp w computes rows 16 (w % 4) .. + 15 of a block, value
// columns 64 (w / 4) .. + 63.  grid: (dv / (64 NT), (S - 1) * block groups
// per segment, N H).
constexpr int kCorrBlocks = 8;
constexpr int kCorrLR = kSplitDK + 8;   // padded bf16 rows (16-byte multiples)
template <int NT>
struct CorrSmem {
  static constexpr int LH = 64 * NT + 8;
  static constexpr int BYTES = (kSplitDK * LH + 2 * 64 * kCorrLR) * 2;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
}

template <int NT>
__global__ void __launch_bounds__(128 * NT) seg_correct_kernel(const FwdParams p, int groups) {
  constexpr int kCorrLH = CorrSmem<NT>::LH, NTH = 128 * NT, NCOL = 64 * NT;
  extern __shared__ __align__(16) uint8_t corr_smem[];
  __nv_bfloat16 *sh = reinterpret_cast<__nv_bfloat16 *>(corr_smem);   // [dk][LH]
  __nv_bfloat16 *sr = sh + kSplitDK * kCorrLH;                          // [2][64][LR]
  const int H = p.num_heads, dv = p.dv, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = blockIdx.x * NCOL, n = blockIdx.z / H, h = blockIdx.z % H;
  const int s = 1 + (int)blockIdx.y / groups, grp = (int)blockIdx.y % groups;
  // segment s >= 1 starts after segment 0, which takes the chunks that the
  // later segments (seg_len tokens each, ending at the last chunk's end) leave
  const int64_t first = (p.seq_len + 63) / 64 * 64 - (int64_t)(p.seg_count - 1) * p.seg_len;
  const int64_t seg0 = first + (int64_t)(s - 1) * p.seg_len;          // segment start
  const int64_t seg_end = seg0 + p.seg_len < p.seq_len ? seg0 + p.seg_len : p.seq_len;
  const int64_t t_first = seg0 + (int64_t)grp * kCorrBlocks * 64;
  if (t_first >= seg_end) return;   // uniform over the CTA
  const int nb = (int)((seg_end - t_first + 63) / 64) < kCorrBlocks
                     ? (int)((seg_end - t_first + 63) / 64)
                     : kCorrBlocks;
  const __nv_bfloat16 *r = static_cast<const __nv_bfloat16 *>(p.seg_r);
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
  const size_t tok0 = (size_t)n * p.seq_len;   // token index of the sequence's start
  const int m0 = 16 * (warp & 3), n0 = 64 * (warp >> 2);
  auto rows_of = [&](int b) {   // valid rows of block b
    const int64_t t = t_first + (int64_t)b * 64;
    return (int)(seg_end - t < 64 ? seg_end - t : 64);
  };
  auto fetch = [&](int b) {   // rows of r of block b into buffer b & 1
    const int64_t t = t_first + (int64_t)b * 64;
    const int valid = rows_of(b);
    __nv_bfloat16 *dr = sr + (b & 1) * 64 * kCorrLR;
    for (int idx = tid; idx < 64 * kSplitDK / 8; idx += NTH) {
      const int rr = idx / (kSplitDK / 8), cc = (idx % (kSplitDK / 8)) * 8;
      const bool ok = rr < valid;
      cp_async16(smem_u32(dr + rr * kCorrLR + cc),
                 r + (((tok0 + t + (ok ? rr : 0)) * H + h) * kSplitDK + cc), ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // this thread's o values of block b (the accumulator positions), two bf16 a word
  auto load_o = [&](int b, uint32_t (&w)[8][2]) {
    const int64_t t = t_first + (int64_t)b * 64;
    const int valid = rows_of(b);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int rr = m0 + (lane >> 2) + 8 * half, cc = n0 + 8 * q + 2 * (lane & 3);
        w[q][half] = rr < valid
                         ? *reinterpret_cast<const uint32_t *>(o + ((tok0 + t + rr) * H + h) * dv +
                                                               c0 + cc)
                         : 0u;
      }
    }
  };
  fetch(0);
  uint32_t ow[8][2], onext[8][2];
  load_o(0, ow);
  {  // H_s, columns c0 .. c0 + 64 NT - 1, in bf16
    const float *Hs = p.seg_state + (((size_t)n * p.seg_count + s) * H + h) * kSplitDK * dv + c0;
    for (int idx = tid; idx < kSplitDK * NCOL / 4; idx += NTH) {
      const int k = idx / (NCOL / 4), cc = (idx % (NCOL / 4)) * 4;
      const float4 x = *reinterpret_cast<const float4 *>(Hs + (size_t)k * dv + cc);
      *reinterpret_cast<uint2 *>(&sh[k * kCorrLH + cc]) =
          make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    }
  }
  for (int b = 0; b < nb; ++b) {
    if (b + 1 < nb) {
      fetch(b + 1);
      load_o(b + 1, onext);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();   // block b's rows of r (and, the first time, H_s) are in place
    const __nv_bfloat16 *br = sr + (b & 1) * 64 * kCorrLR;
    float acc[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < kSplitDK; k0 += 16) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(smem_u32(br + (m0 + (lane & 7) + ((lane >> 3) & 1) * 8) * kCorrLR + k0 +
                       (lane >> 4) * 8),
              a0, a1, a2, a3);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = lane >> 3;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(sh + (k0 + (i & 1) * 8 + (lane & 7)) * kCorrLH + n0 + 16 * q +
                           (i >> 1) * 8),
                  b0, b1, b2, b3);
        mma_bf16(acc[2 * q], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[2 * q + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    const int64_t t = t_first + (int64_t)b * 64;
    const int valid = rows_of(b);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int rr = m0 + (lane >> 2) + 8 * half, cc = n0 + 8 * q + 2 * (lane & 3);
        if (rr < valid) {
          const uint32_t w = ow[q][half];
          *reinterpret_cast<uint32_t *>(o + ((tok0 + t + rr) * H + h) * dv + c0 + cc) =
              pack_bf16(bf16_lo(w) + acc[q][2 * half], bf16_hi(w) + acc[q][2 * half + 1]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      ow[q][0] = onext[q][0];
      ow[q][1] = onext[q][1];
    }
    __syncthreads();   // buffer b & 1 is refilled by the fetch of block b + 2
  }
}

}  // namespace

cudaError_t launch_seg_compose(const FwdParams &p, int s, cudaStream_t stream) {
  seg_compose_kernel<<<dim3(p.dv / 32 * (kSplitDK / 32), p.num_heads, p.num_seqs), 256, 0,
                       stream>>>(p, s);
  return cudaGetLastError();
}

cudaError_t launch_seg_correct(const FwdParams &p, cudaStream_t stream) {
  const int S = p.seg_count;
  const int groups = (p.seg_len / 64 + kCorrBlocks - 1) / kCorrBlocks;
  const dim3 cgrid((p.dv % 128 == 0 ? p.dv / 128 : p.dv / 64), (S - 1) * groups,
                   p.num_seqs * p.num_heads);
  cudaError_t err;
  if (p.dv % 128 == 0) {   // 128 value columns a CTA: each row of r read once per two tiles
    if ((err = cudaFuncSetAttribute(seg_correct_kernel<2>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    CorrSmem<2>::BYTES)) != cudaSuccess)
      return err;
    seg_correct_kernel<2><<<cgrid, 256, CorrSmem<2>::BYTES, stream>>>(p, groups);
  } else {
    if ((err = cudaFuncSetAttribute(seg_correct_kernel<1>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    CorrSmem<1>::BYTES)) != cudaSuccess)
      return err;
    seg_correct_kernel<1><<<cgrid, 128, CorrSmem<1>::BYTES, stream>>>(p, groups);
  }
  return cudaGetLastError();
}

}  // namespace gdn
