// The two small kernels of a split sequence (GDN_SEQ_SPLIT, head_dim_k 128)
// that follow the segments' chain launch: the composition of the segments'
// affine state maps, H_(s+1) = M_s H_s + X_s, every step in segment order in
// one launch, and the correction of the later segments' outputs, o += r H_s.
// ("Optimization Quartet", Triton GDN kernel section 3.2, names the
// inter-chunk carry as the serial part of the chunked form; the maps and
// their composition are what lets the segments run at the same time.)
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kSplitDK = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
}

// The composition, H_(s+1) = M_s H_s + X_s for s = s_first .. S-1 in order
// (fp32; M_s is dk x dk; the last step gives the caller's final state), in one
// launch.  M_s mixes rows only, so value columns evolve independently: a CTA
// takes kCompCols value columns of one (sequence, head) through every step
// with nothing exchanged between CTAs.  Thread (row tid / 2, half tid % 2)
// forms 8 columns of its row; H_s sits in shared memory, M_s too (rows
// padded to kCompLM floats), and M_(s+1) is fetched into the other buffer
// (cp.async) and X_(s+1) into registers while step s is computed.  grid:
// (dv / kCompCols, H, N), 256 threads.
constexpr int kCompCols = 16;
constexpr int kCompLM = kSplitDK + 4;
constexpr int kCompBytes = (2 * kSplitDK * kCompLM + kSplitDK * kCompCols) * 4;

__global__ void __launch_bounds__(256) seg_compose_kernel(const FwdParams p, int s_first) {
  extern __shared__ __align__(16) float comp_smem[];
  float *ms = comp_smem;                          // [2][dk][kCompLM]
  float *hs = comp_smem + 2 * kSplitDK * kCompLM;  // [dk][kCompCols]
  const int c0 = blockIdx.x * kCompCols, h = blockIdx.y, n = blockIdx.z;
  const int H = p.num_heads, dv = p.dv, S = p.seg_count, tid = threadIdx.x;
  const int r = tid >> 1, cl = 8 * (tid & 1);     // this thread's row and first column
  auto unit = [&](int s) { return ((size_t)n * S + s) * H + h; };
  auto fetch_m = [&](int s) {   // M_s into buffer s & 1: 4096 pieces of 16 bytes
    const float *M = p.seg_m + unit(s) * kSplitDK * kSplitDK;
    float *dst = ms + (s & 1) * kSplitDK * kCompLM;
#pragma unroll 4
    for (int i = tid; i < kSplitDK * kSplitDK / 4; i += 256) {
      const int mr = i / (kSplitDK / 4), mc = 4 * (i % (kSplitDK / 4));
      cp_async16(smem_u32(dst + mr * kCompLM + mc), M + (size_t)mr * kSplitDK + mc, true);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto load_x = [&](int s, float4 &x0, float4 &x1) {   // this thread's 8 values of X_s
    const float *X = p.seg_x + unit(s) * kSplitDK * dv + (size_t)r * dv + c0 + cl;
    x0 = *reinterpret_cast<const float4 *>(X);
    x1 = *reinterpret_cast<const float4 *>(X + 4);
  };
  fetch_m(s_first);
  {  // H_(s_first), the state entering that segment: 512 float4, two a thread
    const float *Hs = p.seg_state + unit(s_first) * kSplitDK * dv + c0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = tid + 256 * e, hr = i / 4, hc = 4 * (i % 4);
      *reinterpret_cast<float4 *>(&hs[hr * kCompCols + hc]) =
          *reinterpret_cast<const float4 *>(Hs + (size_t)hr * dv + hc);
    }
  }
  float4 x0, x1;
  load_x(s_first, x0, x1);
  for (int s = s_first; s < S; ++s) {
    float4 xn0 = x0, xn1 = x1;
    if (s + 1 < S) {
      fetch_m(s + 1);
      load_x(s + 1, xn0, xn1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();   // M_s and H_s in place
    float acc[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const float *mrow = ms + (s & 1) * kSplitDK * kCompLM + r * kCompLM;
#pragma unroll 4
    for (int k = 0; k < kSplitDK; k += 4) {
      const float4 m4 = *reinterpret_cast<const float4 *>(mrow + k);
      const float mk[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 a = *reinterpret_cast<const float4 *>(&hs[(k + j) * kCompCols + cl]);
        const float4 b = *reinterpret_cast<const float4 *>(&hs[(k + j) * kCompCols + cl + 4]);
        acc[0] = fmaf(mk[j], a.x, acc[0]);
        acc[1] = fmaf(mk[j], a.y, acc[1]);
        acc[2] = fmaf(mk[j], a.z, acc[2]);
        acc[3] = fmaf(mk[j], a.w, acc[3]);
        acc[4] = fmaf(mk[j], b.x, acc[4]);
        acc[5] = fmaf(mk[j], b.y, acc[5]);
        acc[6] = fmaf(mk[j], b.z, acc[6]);
        acc[7] = fmaf(mk[j], b.w, acc[7]);
      }
    }
    __syncthreads();   // H_s and buffer s & 1 read by every thread
    const float4 y0 = make_float4(acc[0], acc[1], acc[2], acc[3]);
    const float4 y1 = make_float4(acc[4], acc[5], acc[6], acc[7]);
    *reinterpret_cast<float4 *>(&hs[r * kCompCols + cl]) = y0;
    *reinterpret_cast<float4 *>(&hs[r * kCompCols + cl + 4]) = y1;
    // segment s + 1's entry state (the correction reads it), or after the last
    // segment the caller's final state
    float *Hn = s + 1 < S ? p.seg_state + unit(s + 1) * kSplitDK * dv
                          : p.sN ? p.sN + ((size_t)n * H + h) * kSplitDK * dv : nullptr;
    if (Hn) {
      *reinterpret_cast<float4 *>(Hn + (size_t)r * dv + c0 + cl) = y0;
      *reinterpret_cast<float4 *>(Hn + (size_t)r * dv + c0 + cl + 4) = y1;
    }
    x0 = xn0;
    x1 = xn1;
  }
}

// The correction of a split sequence's later segments: o[t] += r[t] H_s for
// every token t of segment s >= 1 (r [tokens][H][dk] and H_s in bf16 on
// mma.sync, fp32 sums, o read and written in bf16).  A CTA takes up to
// kCorrBlocks blocks of 64 tokens inside one segment and 64 NT value columns
// of one (sequence, head), so that each row of r is read once per NT column
// tiles; H_s is converted once.  Block b + 2's rows of r are fetched
// (cp.async, three buffers) and its o values loaded into registers (three
// sets) while block b is computed, so every load has two blocks' time to
// land; the block loop is unrolled so that the register sets stay distinct.
// Warp w computes rows 16 (w % 4) .. + 15 of a block, value columns
// 64 (w / 4) .. + 63.  grid: (dv / (64 NT), (S - 1) * block groups per
// segment, N H).
constexpr int kCorrBlocks = 8;
constexpr int kCorrBufs = 3;
constexpr int kCorrLR = kSplitDK + 8;   // padded bf16 rows (16-byte multiples)
template <int NT>
struct CorrSmem {
  static constexpr int LH = 64 * NT + 8;
  static constexpr int BYTES = (kSplitDK * LH + kCorrBufs * 64 * kCorrLR) * 2;
};

template <int NT>
__global__ void __launch_bounds__(128 * NT, 2) seg_correct_kernel(const FwdParams p, int groups) {
  constexpr int kCorrLH = CorrSmem<NT>::LH, NTH = 128 * NT, NCOL = 64 * NT;
  extern __shared__ __align__(16) uint8_t corr_smem[];
  __nv_bfloat16 *sh = reinterpret_cast<__nv_bfloat16 *>(corr_smem);   // [dk][LH]
  __nv_bfloat16 *sr = sh + kSplitDK * kCorrLH;                          // [3][64][LR]
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
  auto fetch = [&](int b) {   // rows of r of block b into buffer b % 3
    const int64_t t = t_first + (int64_t)b * 64;
    const int valid = rows_of(b);
    __nv_bfloat16 *dr = sr + (b % kCorrBufs) * 64 * kCorrLR;
#pragma unroll
    for (int e = 0; e < 64 * kSplitDK / 8 / NTH; ++e) {
      const int idx = tid + e * NTH;
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
  uint32_t ow[kCorrBufs][8][2];
  fetch(0);
  load_o(0, ow[0]);
  if (nb > 1) {
    fetch(1);
    load_o(1, ow[1]);
  }
  {  // H_s, columns c0 .. c0 + 64 NT - 1, in bf16 (eight loads in flight a thread)
    const float *Hs = p.seg_state + (((size_t)n * p.seg_count + s) * H + h) * kSplitDK * dv + c0;
#pragma unroll 8
    for (int e = 0; e < kSplitDK * NCOL / 4 / NTH; ++e) {
      const int idx = tid + e * NTH;
      const int k = idx / (NCOL / 4), cc = (idx % (NCOL / 4)) * 4;
      const float4 x = *reinterpret_cast<const float4 *>(Hs + (size_t)k * dv + cc);
      *reinterpret_cast<uint2 *>(&sh[k * kCorrLH + cc]) =
          make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    }
  }
#pragma unroll
  for (int b = 0; b < kCorrBlocks; ++b) {
    if (b < nb) {   // uniform over the CTA
      if (b + 2 < nb) {
        fetch(b + 2);
        load_o(b + 2, ow[(b + 2) % kCorrBufs]);
        asm volatile("cp.async.wait_group 2;" ::: "memory");
      } else if (b + 1 < nb) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      __syncthreads();   // block b's rows of r (and, the first time, H_s) are in place
      const __nv_bfloat16 *br = sr + (b % kCorrBufs) * 64 * kCorrLR;
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
            const uint32_t w = ow[b % kCorrBufs][q][half];
            *reinterpret_cast<uint32_t *>(o + ((tok0 + t + rr) * H + h) * dv + c0 + cc) =
                pack_bf16(bf16_lo(w) + acc[q][2 * half], bf16_hi(w) + acc[q][2 * half + 1]);
          }
        }
      }
      __syncthreads();   // buffer b % 3 is refilled by the fetch of block b + 3
    }
  }
}

}  // namespace

cudaError_t launch_seg_compose(const FwdParams &p, int s, cudaStream_t stream) {
  cudaError_t err =
      cudaFuncSetAttribute(seg_compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kCompBytes);
  if (err != cudaSuccess) return err;
  seg_compose_kernel<<<dim3(p.dv / kCompCols, p.num_heads, p.num_seqs), 256, kCompBytes,
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
