// Host side of the C ABI declared in include/gdn.h: argument validation,
// kernel selection and launch, and the status-word check.  Nothing here
// computes any part of the recurrence; every step runs in the CUDA kernels.
#include <stdint.h>
#include <string.h>

#include "gdn_internal.cuh"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Half-open byte ranges [a, a+na) and [b, b+nb) overlap.
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool supported_dk(int dk) { return dk == 32 || dk == 64 || dk == 128; }
bool supported_dv(int dv) { return dv >= 32 && dv <= 256 && dv % 32 == 0; }

bool use_tc(int dk, int dv, gdn_dtype dtype, uint32_t flags) {
  return dtype == GDN_BF16 && !(flags & GDN_FORCE_SIMT) && gdn::tc_supported(dk, dv);
}
// the tensor-core chunk-size variants (chunk_size 32 and 128)
bool use_tcc(int chunk, int dk, int dv, gdn_dtype dtype, uint32_t flags) {
  return dtype == GDN_BF16 && !(flags & GDN_FORCE_SIMT) && gdn::tcc_supported(chunk, dk, dv);
}

}  // namespace

namespace gdn {
// A call with no tokens: copy each initial state to the final state (zeros
// without one); nothing else is read or written.
gdn_status pass_states(const float *from, float *to, size_t bytes, cudaStream_t s) {
  if (to == nullptr) return GDN_OK;
  if (!aligned16(to) || (from && !aligned16(from))) return GDN_ERR_INVALID_ARG;
  if (from && from != to && overlaps(from, bytes, to, bytes)) return GDN_ERR_INVALID_ARG;
  const cudaError_t e = from == nullptr ? cudaMemsetAsync(to, 0, bytes, s)
                        : from == to    ? cudaSuccess
                                        : cudaMemcpyAsync(to, from, bytes, cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
}  // namespace gdn

namespace gdn {
// Every host-side check of gdn_fwd, in one place, so that each entry point
// that runs the forward pass validates its arguments before it enqueues any
// work.  Fills `call` on success.
int plan_segments(FwdParams &p, int chunk, gdn_dtype dtype);

gdn_status fwd_validate(const void *q, const void *k, const void *v, const float *g,
                        const void *beta, const float *initial_state,
                        const int32_t *cu_seqlens, void *o, float *final_state,
                        const float *D_skip, const float *out_gate, int32_t batch,
                        int32_t seq_len, int32_t num_heads, int32_t head_dim_k,
                        int32_t head_dim_v, int32_t num_seqs, int32_t chunk_size,
                        gdn_dtype dtype, uint32_t flags, void *workspace,
                        size_t workspace_bytes, FwdCall *call) {
  // ---- shapes ----
  if (batch <= 0 || seq_len < 0 || num_heads <= 0 || head_dim_k <= 0 || head_dim_v <= 0 ||
      num_seqs <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)(GDN_QK_L2NORM | GDN_FORCE_SIMT | GDN_BETA_LOGITS | GDN_DEBUG_CHECKS |
                          GDN_SEQ_SPLIT))
    return GDN_ERR_INVALID_ARG;
  if (cu_seqlens ? batch != 1 : num_seqs != batch) return GDN_ERR_INVALID_ARG;
  if (!supported_dk(head_dim_k) || !supported_dv(head_dim_v)) return GDN_ERR_UNSUPPORTED;
  if (!simt_chunk_supported(chunk_size, head_dim_k)) return GDN_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_heads > 65535) return GDN_ERR_UNSUPPORTED;
  const size_t b_state = (size_t)num_seqs * num_heads * head_dim_k * head_dim_v * 4;
  call->states_only = seq_len == 0;
  call->state_bytes = b_state;
  call->chunk = chunk_size;
  call->dtype = dtype;
  if (seq_len == 0) {  // no tokens: every state passes through, nothing else is read
    if (final_state == nullptr) { call->p.s0 = initial_state; call->p.sN = nullptr; return GDN_OK; }
    if (!aligned16(final_state) || (initial_state && !aligned16(initial_state)))
      return GDN_ERR_INVALID_ARG;
    if (initial_state && initial_state != final_state &&
        overlaps(initial_state, b_state, final_state, b_state))
      return GDN_ERR_INVALID_ARG;
    call->p.s0 = initial_state;
    call->p.sN = final_state;
    return GDN_OK;
  }

  // ---- pointers ----
  if (!q || !k || !v || !g || !beta || !o) return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, initial_state, cu_seqlens, o, final_state, D_skip,
                        out_gate};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  if (!workspace) return GDN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GDN_ERR_INVALID_ARG;
  if (workspace_bytes <
      gdn_fwd_workspace_size(num_seqs, num_heads, head_dim_k, head_dim_v, flags))
    return GDN_ERR_WORKSPACE;

  // ---- aliasing: outputs must not overlap inputs (initial_state == final_state allowed) ----
  const size_t e = dtype == GDN_F32 ? 4 : 2;
  const size_t rows = (size_t)batch * (size_t)seq_len * (size_t)num_heads;
  const size_t b_qk = rows * head_dim_k * e, b_v = rows * head_dim_v * e;
  const size_t b_g = rows * 4, b_beta = rows * e;
  const size_t b_cu = cu_seqlens ? (size_t)(num_seqs + 1) * 4 : 0;
  struct Range { const void *p; size_t n; };
  const Range inputs[] = {{q, b_qk}, {k, b_qk}, {v, b_v}, {g, b_g}, {beta, b_beta},
                          {cu_seqlens, b_cu}, {workspace, workspace_bytes},
                          {D_skip, D_skip ? (size_t)num_heads * 4 : 0},
                          {out_gate, out_gate ? b_g : 0}};
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

  FwdParams &p = call->p;
  p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g;
  p.s0 = initial_state; p.cu = cu_seqlens; p.o = o; p.sN = final_state;
  p.d_skip = D_skip; p.out_gate = out_gate;
  p.status = static_cast<DeviceStatus *>(workspace);
  p.ckpt = nullptr;
  p.seq_len = seq_len;
  p.num_heads = num_heads; p.dk = head_dim_k; p.dv = head_dim_v; p.num_seqs = num_seqs;
  p.flags = flags;
  // extents from the shapes (gdn_fwd_debug may declare smaller ones)
  const int64_t r = (int64_t)rows;
  p.ext.q = p.ext.k = r * head_dim_k;
  p.ext.v = p.ext.o = r * head_dim_v;
  p.ext.g = p.ext.beta = p.ext.gate = r;
  p.ext.s0 = p.ext.sN = (int64_t)num_seqs * num_heads * head_dim_k * head_dim_v;
  // a call that will be split keeps its per-token maps in the workspace
  FwdParams plan = p;
  if (plan_segments(plan, chunk_size, dtype) > 1 &&
      workspace_bytes <
          gdn_fwd_split_workspace_size(num_seqs, seq_len, num_heads, head_dim_k, head_dim_v))
    return GDN_ERR_WORKSPACE;
  return GDN_OK;
}

// The split plan's cost model: the time, in chunk steps, of one launch that
// dispatches `a` CTAs of `first` chunks (segment 0's value tiles) and then
// `b` CTAs of `len` chunks (the later segments' value and transport tiles)
// on `sm` SMs, one CTA per SM, each CTA to the first SM that frees.  The
// sm - a SMs that segment 0 leaves free take later CTAs from the start, the
// other a from `first` on.  a < sm.
int64_t split_makespan(int64_t a, int64_t b, int64_t first, int64_t len, int64_t sm) {
  const int64_t idle = sm - a;   // SMs that segment 0 leaves free
  int64_t done = 0, rounds_idle = 0, rounds_a = 0, last = 0;
  while (done < b) {
    const int64_t tf = idle > 0 ? rounds_idle * len : INT64_MAX, ta = first + rounds_a * len;
    if (tf <= ta) {
      done += idle;
      last = tf;
      ++rounds_idle;
    } else {
      done += a;
      last = ta;
      ++rounds_a;
    }
  }
  return last + len > first ? last + len : first;
}

constexpr int kMaxFirstLens = 16;   // segment 0: at most this many later lengths

// The split plan of GDN_SEQ_SPLIT: fills p.seg_len / p.seg_count (0 when
// the call is not split) and returns the segment count (1: not split).  The
// block epilogue is not combined with a split (the correction would have to
// pass through it), nor GDN_DEBUG_CHECKS (the composition and correction
// kernels check no declared extents): such calls run unsplit.
//
// Segments 1 .. S-1 hold seg_len tokens each (whole chunks, the last ending
// at the sequence's end); segment 0 takes the chunks they leave at the
// front.  Its CTAs are few (value tiles only) and are dispatched first, so it
// can be k times longer while the SMs it leaves free run the later segments.
// The plan takes the S in 2 .. kMaxSegments and k in 1 .. kMaxFirstLens
// (seg_len = chunks / (k + S - 1), at least 4 chunks) with the shortest
// split_makespan, the fewest segments among equals, and splits only when
// that beats the unsplit launch by a quarter (the composition steps and the
// correction cost a little).  A call whose first segments alone fill the SMs
// is not split.
int plan_segments(FwdParams &p, int chunk, gdn_dtype dtype) {
  p.seg_len = p.seg_count = 0;
  if (!(p.flags & GDN_SEQ_SPLIT) || (p.flags & GDN_DEBUG_CHECKS) || chunk != kChunk ||
      !use_tc(p.dk, p.dv, dtype, p.flags) || p.d_skip || p.out_gate)
    return 1;
  const int most = seq_split_segments(p);   // what the tensor-core launch takes
  if (most < 2) return 1;
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (sms[dev] == 0 &&
      cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  const int64_t sm = sms[dev];
  const int64_t units = (int64_t)p.num_seqs * p.num_heads;
  const int64_t a = units * (p.dv / 64);            // segment 0: value tiles
  const int64_t u = units * ((p.dv + p.dk) / 64);   // a later segment: value + transport
  const int64_t chunks = (p.seq_len + kChunk - 1) / kChunk;
  if (a >= sm) return 1;
  double best_span = 0.75 * (double)chunks;   // the unsplit launch: one wave of all chunks
  int best_s = 1;
  int64_t best_len = 0;
  for (int s = 2; s <= most && s <= kMaxSegments; ++s) {
    for (int k = 1; k <= kMaxFirstLens; ++k) {
      const int64_t len = chunks / (k + s - 1);
      if (len < 4) break;
      const int64_t first = chunks - (int64_t)(s - 1) * len;
      const int64_t span = split_makespan(a, (int64_t)(s - 1) * u, first, len, sm);
      if ((double)span < best_span) {
        best_span = (double)span;
        best_s = s;
        best_len = len;
      }
    }
  }
  if (best_s < 2) return 1;
  p.seg_len = (int32_t)(best_len * kChunk);
  p.seg_count = best_s;
  return p.seg_count;
}

// Byte offset of the per-token maps r in a split call's workspace.
size_t split_r_offset(int64_t num_seqs, int64_t num_heads, int64_t dk, int64_t dv) {
  const size_t seg = (size_t)4 * num_seqs * kMaxSegments * num_heads * dk * (2 * dv + dk);
  return (kStatusBytes + seg + 255) & ~(size_t)255;
}

// Enqueue the kernels of a call that fwd_validate accepted.
gdn_status fwd_launch(const FwdCall &call, cudaStream_t stream) {
  if (call.states_only)
    return call.p.sN ? pass_states(call.p.s0, call.p.sN, call.state_bytes, stream) : GDN_OK;
  // bf16 storage runs on the tensor-core kernels: the 64-token ones, or the
  // chunk-size variants for 32 and 128; everything else on the fp32
  // CUDA-core kernel
  FwdParams p = call.p;
  if (plan_segments(p, call.chunk, call.dtype) > 1) {
    // the segments' states, X and M follow the status record in the
    // workspace, then the per-token maps r (fwd_validate checked the size)
    unsigned char *ws = reinterpret_cast<unsigned char *>(p.status);
    float *base = reinterpret_cast<float *>(ws + kStatusBytes);
    const size_t vals = (size_t)p.num_seqs * kMaxSegments * p.num_heads * p.dk * p.dv;
    p.seg_state = base;
    p.seg_x = base + vals;
    p.seg_m = base + 2 * vals;
    p.seg_r = ws + split_r_offset(p.num_seqs, p.num_heads, p.dk, p.dv);
  }
  const cudaError_t err =
      call.chunk == kChunk && use_tc(p.dk, p.dv, call.dtype, p.flags)
          ? launch_fwd_tc(p, stream)
      : use_tcc(call.chunk, p.dk, p.dv, call.dtype, p.flags)
          ? launch_fwd_tcc(p, call.chunk, stream)
          : launch_fwd_simt(p, call.dtype, call.chunk, stream);
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
}  // namespace gdn

extern "C" {

size_t gdn_fwd_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_dim_k,
                              int32_t head_dim_v, uint32_t flags) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim_k <= 0 || head_dim_v <= 0) return 0;
  size_t bytes = gdn::kStatusBytes;
  if ((flags & GDN_SEQ_SPLIT) && head_dim_k == 128)  // per segment: a state, X and M
    bytes += (size_t)4 * num_seqs * gdn::kMaxSegments * num_heads * head_dim_k *
             (2 * (size_t)head_dim_v + head_dim_k);
  return bytes;
}

size_t gdn_fwd_split_workspace_size(int32_t num_seqs, int32_t seq_len, int32_t num_heads,
                                    int32_t head_dim_k, int32_t head_dim_v) {
  if (num_seqs <= 0 || seq_len < 0 || num_heads <= 0 || head_dim_k <= 0 || head_dim_v <= 0)
    return 0;
  if (head_dim_k != 128)
    return gdn_fwd_workspace_size(num_seqs, num_heads, head_dim_k, head_dim_v, GDN_SEQ_SPLIT);
  return gdn::split_r_offset(num_seqs, num_heads, head_dim_k, head_dim_v) +
         (size_t)2 * num_seqs * seq_len * num_heads * head_dim_k;
}

int32_t gdn_fwd_split_segments(int32_t num_seqs, int32_t seq_len, int32_t num_heads,
                               int32_t head_dim_k, int32_t head_dim_v, int32_t chunk_size,
                               gdn_dtype dtype, uint32_t flags, int32_t varlen) {
  if (num_seqs < 1 || num_seqs > 65535 || seq_len < 0 || num_heads < 1 ||
      !supported_dk(head_dim_k) || !supported_dv(head_dim_v) ||
      (dtype != GDN_F32 && dtype != GDN_BF16) ||
      !gdn::simt_chunk_supported(chunk_size, head_dim_k))
    return 0;
  gdn::FwdParams p{};
  p.num_seqs = num_seqs;
  p.seq_len = seq_len;
  p.num_heads = num_heads;
  p.dk = head_dim_k;
  p.dv = head_dim_v;
  p.flags = flags;
  static const int32_t kNonNull = 0;
  p.cu = varlen ? &kNonNull : nullptr;  // only its presence is read
  return gdn::plan_segments(p, chunk_size, dtype);
}

gdn_status gdn_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace || workspace_bytes < gdn::kStatusBytes) return GDN_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

const char *gdn_fwd_kernel_name_chunk(int32_t head_dim_k, int32_t head_dim_v,
                                      int32_t chunk_size, gdn_dtype dtype, uint32_t flags) {
  if (!supported_dk(head_dim_k) || !supported_dv(head_dim_v)) return nullptr;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return nullptr;
  if (!gdn::simt_chunk_supported(chunk_size, head_dim_k)) return nullptr;
  if (chunk_size == gdn::kChunk && use_tc(head_dim_k, head_dim_v, dtype, flags))
    return head_dim_k == 64 ? "tc64_bf16" : "tc128_bf16";
  if (use_tcc(chunk_size, head_dim_k, head_dim_v, dtype, flags))
    return chunk_size == 32 ? "tcc32_bf16" : "tcc128_bf16";
  return dtype == GDN_F32 ? "simt_fp32" : "simt_bf16";
}

const char *gdn_fwd_kernel_name(int32_t head_dim_k, int32_t head_dim_v, gdn_dtype dtype,
                                uint32_t flags) {
  return gdn_fwd_kernel_name_chunk(head_dim_k, head_dim_v, gdn::kChunk, dtype, flags);
}

gdn_status gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                   const void *beta, const float *initial_state, const int32_t *cu_seqlens,
                   void *o, float *final_state, const float *D_skip, const float *out_gate,
                   int32_t batch, int32_t seq_len,
                   int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                   int32_t num_seqs, int32_t chunk_size, gdn_dtype dtype, uint32_t flags,
                   void *workspace, size_t workspace_bytes, void *stream) {
  gdn::FwdCall call;
  const gdn_status st = gdn::fwd_validate(q, k, v, g, beta, initial_state, cu_seqlens, o,
                                          final_state, D_skip, out_gate, batch, seq_len, num_heads, head_dim_k,
                                          head_dim_v, num_seqs, chunk_size, dtype, flags,
                                          workspace, workspace_bytes, &call);
  if (st != GDN_OK) return st;
  return gdn::fwd_launch(call, (cudaStream_t)stream);
}

gdn_status gdn_fwd_debug(const void *q, const void *k, const void *v, const float *g,
                         const void *beta, const float *initial_state, const int32_t *cu_seqlens,
                         void *o, float *final_state, const float *D_skip, const float *out_gate,
                         int32_t batch, int32_t seq_len, int32_t num_heads, int32_t head_dim_k,
                         int32_t head_dim_v, int32_t num_seqs, int32_t chunk_size, gdn_dtype dtype,
                         uint32_t flags, void *workspace, size_t workspace_bytes,
                         const gdn_extents *declared, void *stream) {
  gdn::FwdCall call;
  const gdn_status st = gdn::fwd_validate(
      q, k, v, g, beta, initial_state, cu_seqlens, o, final_state, D_skip, out_gate, batch,
      seq_len, num_heads, head_dim_k, head_dim_v, num_seqs, chunk_size, dtype,
      flags | GDN_DEBUG_CHECKS, workspace, workspace_bytes, &call);
  if (st != GDN_OK) return st;
  if (declared && call.states_only) {  // no kernel runs: the copy's extents are checked here
    const int64_t need = (int64_t)(call.state_bytes / 4);
    if ((call.p.sN && call.p.s0 && declared->initial_state < need) ||
        (call.p.sN && declared->final_state < need))
      return GDN_ERR_INVALID_ARG;
  }
  if (declared) {
    const int64_t d[] = {declared->q, declared->k, declared->v, declared->g, declared->beta,
                         declared->o, declared->initial_state, declared->final_state,
                         declared->out_gate};
    for (int64_t x : d)
      if (x < 0) return GDN_ERR_INVALID_ARG;
    gdn::Extents &e = call.p.ext;
    e.q = declared->q; e.k = declared->k; e.v = declared->v; e.g = declared->g;
    e.beta = declared->beta; e.o = declared->o; e.s0 = declared->initial_state;
    e.sN = declared->final_state; e.gate = declared->out_gate;
  }
  return gdn::fwd_launch(call, (cudaStream_t)stream);
}

gdn_status gdn_check_record(void *workspace, void *stream, int32_t *seq, int32_t *head,
                            int32_t *site) {
  if (seq) *seq = -1;
  if (head) *head = -1;
  if (site) *site = 0;
  if (!workspace) return GDN_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  gdn::DeviceStatus st;
  memset(&st, 0, sizeof st);
  if (cudaMemcpyAsync(&st, workspace, sizeof st, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  if (st.code == 0) return GDN_OK;
  if (cudaMemsetAsync(workspace, 0, sizeof st, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  if (seq) *seq = (int32_t)st.seq;
  if (head) *head = (int32_t)st.head;
  if (site) *site = (int32_t)st.aux;
  return st.code <= GDN_ERR_DEVICE_CHECK ? (gdn_status)st.code : GDN_ERR_DEVICE_CHECK;
}

gdn_status gdn_check(void *workspace, void *stream) {
  return gdn_check_record(workspace, stream, nullptr, nullptr, nullptr);
}

const char *gdn_status_string(int32_t status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: bad pointer, size or aliasing";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: sizes not implemented";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA runtime call or launch failed";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait gave up";
    case GDN_ERR_BAD_SEQLENS: return "GDN_ERR_BAD_SEQLENS: cu_seqlens does not rise from 0 to T without decreasing";
    case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK: a device-side check failed";
    default: return "GDN_ERR_UNKNOWN";
  }
}

}  // extern "C"
