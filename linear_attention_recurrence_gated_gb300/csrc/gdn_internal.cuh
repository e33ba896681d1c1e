// Internal declarations shared by the CUDA translation units of libgdn.
// Not part of the public ABI (that is include/gdn.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;  // tokens per chunk of the tensor-core kernels (the default)
constexpr int kMaxSegments = 8;  // GDN_SEQ_SPLIT: segments per sequence at most

// Device status record at the start of the workspace.  The first error wins
// (atomicCAS from 0); `seq` and `head` locate it, `aux` carries a detail.
struct DeviceStatus {
  uint32_t code;
  uint32_t seq;
  uint32_t head;
  uint32_t aux;
};
constexpr size_t kStatusBytes = 256;

// Elements each buffer of a forward call holds: derived from the shapes, or
// declared by the caller of gdn_fwd_debug.  Read only under GDN_DEBUG_CHECKS.
struct Extents {
  int64_t q, k, v, g, beta, o, s0, sN, gate;
};

// Sites recorded in DeviceStatus::aux by a failed GDN_DEBUG_CHECKS range check.
enum DebugSite : uint32_t {
  kSiteQ = 1, kSiteK, kSiteV, kSiteG, kSiteBeta, kSiteO, kSiteS0, kSiteSN, kSiteGate,
  kSiteTmaX,  // a TMA box's innermost coordinate is not on a 16-byte boundary
};

// Everything one gdn_fwd launch needs, passed by value as a kernel argument.
struct FwdParams {
  const void *q, *k, *v, *beta;
  const float *g;
  const float *s0;
  const int32_t *cu;
  void *o;
  float *sN;
  const float *d_skip;    // [H] skip weights of the block epilogue, or NULL (0)
  const float *out_gate;  // [tokens][H] output gate of the block epilogue, or NULL (1)
  DeviceStatus *status;
  float *ckpt;          // backward only: state at every 64-token chunk start (else NULL)
  int64_t seq_len;      // tokens per batch row (dense) or packed total (varlen)
  int32_t num_heads, dk, dv, num_seqs;
  uint32_t flags;
  Extents ext;
  // Sequence split (dense inputs, head_dim_k 128; GDN_SEQ_SPLIT): each
  // sequence is cut into seg_count segments, all run by one launch (grid z =
  // segment * num_seqs + sequence).  Segments 1 .. seg_count-1 hold seg_len
  // tokens each (whole chunks, the last ending at the sequence's end);
  // segment 0 takes the chunks they leave at the front.  Segment 0 starts from
  // the caller's state and ends in seg_state of segment 1.  Later segments
  // start from zero on the value columns (their outputs o0 and end state X)
  // and from the identity on dk extra columns (their per-token reads r, to
  // seg_r, and end state M): the segment maps H -> M H + X and o -> o0 + r H.
  // seg_len = 0: no split.
  int32_t seg_len = 0, seg_count = 0;
  float *seg_state = nullptr;  // [N][seg_count][H][dk][dv]: entry states (s >= 1)
  float *seg_x = nullptr;      // [N][seg_count][H][dk][dv]
  float *seg_m = nullptr;      // [N][seg_count][H][dk][dk]
  void *seg_r = nullptr;       // [N * seq_len][H][dk] bf16
};

__device__ __forceinline__ void report(DeviceStatus *st, uint32_t code, uint32_t seq,
                                       uint32_t head, uint32_t aux) {
  if (atomicCAS(&st->code, 0u, code) == 0u) {
    st->seq = seq;
    st->head = head;
    st->aux = aux;
  }
}

// Bounds of sequence n: [start, start + len), len = 0 for an empty sequence.
// Returns false (after recording GDN_ERR_BAD_SEQLENS) when cu_seqlens breaks
// 0 = cu[0] <= ... <= cu[N] = T.
__device__ __forceinline__ bool sequence_bounds(const FwdParams &p, int n, int h,
                                                int64_t &start, int64_t &len) {
  if (p.cu == nullptr) {
    start = (int64_t)n * p.seq_len;
    len = p.seq_len;
    return true;
  }
  const int64_t s = p.cu[n], e = p.cu[n + 1];
  const bool ok = s >= 0 && e >= s && e <= p.seq_len && (n != 0 || s == 0) &&
                  (n != p.num_seqs - 1 || e == p.seq_len);
  if (!ok) {
    report(p.status, GDN_ERR_BAD_SEQLENS, (uint32_t)n, (uint32_t)h, 0u);
    return false;
  }
  start = s;
  len = e - s;
  return true;
}

// GDN_DEBUG_CHECKS: before its first global access, the block that owns value
// columns [col0, col0 + ncols) of (sequence n, head h) checks the whole index
// range it will touch in every buffer, with the kernels' own index formulas
// (all monotone in the token, the row and the column), against the extents;
// `tma_x` asks for the TMA rule that a box's innermost coordinate times the
// element size be a multiple of 16 bytes (the q/k boxes start at column 0,
// the v/o boxes at col0).  The first violation is recorded as
// GDN_ERR_DEVICE_CHECK with (n, h, site) and the block must then end without
// any access; returns false in that case.  Uniform over the block.
__device__ __forceinline__ bool debug_ranges_ok(const FwdParams &p, int n, int h, int64_t start,
                                                int64_t len, int col0, int ncols, int elem_bytes,
                                                bool tma_x) {
  const int64_t H = p.num_heads, dk = p.dk, dv = p.dv;
  const Extents &x = p.ext;
  uint32_t site = 0;
  if (tma_x && ((int64_t)col0 * elem_bytes) % 16 != 0) site = kSiteTmaX;
  if (len > 0 && site == 0) {
    const int64_t t_hi = start + len - 1;            // last token of the sequence
    const int64_t qk_hi = (t_hi * H + h) * dk + dk - 1;  // last q/k element read
    const int64_t vo_hi = (t_hi * H + h) * dv + col0 + ncols - 1;
    const int64_t row_hi = t_hi * H + h;              // last g / beta / gate element
    if (start < 0) site = kSiteQ;
    else if (qk_hi >= x.q) site = kSiteQ;
    else if (qk_hi >= x.k) site = kSiteK;
    else if (vo_hi >= x.v) site = kSiteV;
    else if (row_hi >= x.g) site = kSiteG;
    else if (row_hi >= x.beta) site = kSiteBeta;
    else if (vo_hi >= x.o) site = kSiteO;
    else if (p.out_gate && row_hi >= x.gate) site = kSiteGate;
  }
  if (site == 0) {
    const int64_t st_hi = ((n * H + h) * dk + dk - 1) * dv + col0 + ncols - 1;
    if (p.s0 && st_hi >= x.s0) site = kSiteS0;
    else if (p.sN && st_hi >= x.sN) site = kSiteSN;
  }
  if (site == 0) return true;
  if (threadIdx.x == 0) report(p.status, GDN_ERR_DEVICE_CHECK, (uint32_t)n, (uint32_t)h, site);
  return false;
}

// An empty sequence leaves its state as it came: the CTA that owns value
// columns [col0, col0 + ncols) of (sequence n, head h) copies that slice of the
// initial state (zeros without one) to the final state.
__device__ __forceinline__ void pass_state_through(const FwdParams &p, int n, int h, int col0,
                                                   int ncols) {
  if (p.sN == nullptr) return;
  const size_t base = ((size_t)n * p.num_heads + h) * (size_t)p.dk * p.dv;
  for (int idx = threadIdx.x; idx < p.dk * ncols; idx += blockDim.x) {
    const size_t off = base + (size_t)(idx / ncols) * p.dv + col0 + idx % ncols;
    p.sN[off] = p.s0 ? p.s0[off] : 0.f;
  }
}

// The block epilogue (o + D_h v) * gate of one output element (a NULL skip
// reads as 0, a NULL gate as 1).
__device__ __forceinline__ float block_epilogue(float o, float v, float d_h, float gate) {
  return (o + d_h * v) * gate;
}
// beta as stored, or sigmoid of it when the caller passes logits
__device__ __forceinline__ float beta_value(float b, uint32_t flags) {
  return (flags & GDN_BETA_LOGITS) ? 1.f / (1.f + expf(-b)) : b;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// First checkpoint slot of sequence n in a [slots][H][dk][dv] array of
// 64-token chunk-start states: dense rows n * ceil(T / 64); packed sequences
// floor(start / 64) + n, which never overlaps the previous sequence's slots.
__host__ __device__ inline int64_t ckpt_first_slot(int64_t n, int64_t start, int64_t seq_len,
                                                   bool varlen) {
  return varlen ? start / 64 + n : n * ((seq_len + 63) / 64);
}
__host__ __device__ inline int64_t ckpt_slots(int64_t num_seqs, int64_t seq_len) {
  const int64_t dense = num_seqs * ((seq_len + 63) / 64), packed = seq_len / 64 + num_seqs + 1;
  return dense > packed ? dense : packed;
}

// A forward call that passed the host-side checks, ready to launch.
struct FwdCall {
  FwdParams p;
  bool states_only;     // seq_len == 0: the states pass through, no kernel runs
  size_t state_bytes;   // bytes of one [N, H, dk, dv] fp32 state array
  int chunk;
  gdn_dtype dtype;
};
// Every host-side check of gdn_fwd (shapes, alignment, workspace size,
// aliasing); returns GDN_OK and fills `call`, or the error and enqueues nothing.
gdn_status fwd_validate(const void *q, const void *k, const void *v, const float *g,
                        const void *beta, const float *initial_state,
                        const int32_t *cu_seqlens, void *o, float *final_state,
                        const float *D_skip, const float *out_gate, int32_t batch,
                        int32_t seq_len, int32_t num_heads, int32_t head_dim_k,
                        int32_t head_dim_v, int32_t num_seqs, int32_t chunk_size,
                        gdn_dtype dtype, uint32_t flags, void *workspace,
                        size_t workspace_bytes, FwdCall *call);
gdn_status fwd_launch(const FwdCall &call, cudaStream_t stream);

// Launchers (one per kernel family).  Return a cudaError_t from the launch.
cudaError_t launch_fwd_simt(const FwdParams &p, gdn_dtype dtype, int chunk, cudaStream_t stream);
bool simt_chunk_supported(int chunk, int dk);   // chunk in {32, 64, 128}, not 128 with dk 128
cudaError_t launch_fwd_tc(const FwdParams &p, cudaStream_t stream);    // bf16 storage only
cudaError_t launch_fwd_tc64(const FwdParams &p, cudaStream_t stream);  // bf16, head_dim_k 64
// GDN_SEQ_SPLIT: the most segments the tensor-core launch cuts each sequence
// of this call into (1: the call cannot be split); the host plan picks the count
int seq_split_segments(const FwdParams &p);
// The split's composition steps s .. seg_count-1 in one launch (H_(s+1) =
// M_s H_s + X_s in order; the last step gives the caller's final state) and
// the correction o += r H_s of the later segments (gdn_seq_split.cu).
cudaError_t launch_seg_compose(const FwdParams &p, int s, cudaStream_t stream);
cudaError_t launch_seg_correct(const FwdParams &p, cudaStream_t stream);
bool tc_supported(int dk, int dv);
// chunk_size 32 and 128 on the tensor cores: bf16, head_dim_k 64
bool tcc_supported(int chunk, int dk, int dv);
cudaError_t launch_fwd_tcc(const FwdParams &p, int chunk, cudaStream_t stream);

}  // namespace gdn
