/*
 * gdn.h -- C ABI of the GB300 (sm_103a) forward pass of the gated delta rule.
 *
 * The operation (per sequence n and head h, tokens t = 1..L_n):
 *
 *     S_t = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t,            alpha_t = exp(g_t)
 *
 * is the gated delta rule of Yang et al., "Gated Delta Networks" (arXiv
 * 2412.06464), which "v1.0 Architecture & Design Spec", section 2.3 (Gated
 * Delta Net block) and section 12a.1 (Fused Triton GDN kernel) name as the
 * algorithm of HyMo's GDN kernel.  q_t is the read key and k_t the write key
 * (c and b on the HyMo pages: "Model Architecture Walkthrough", section 5.2.1
 * and 5.2.3); the decay is alpha_t = exp(g_t) with g_t <= 0 the natural-log
 * gate (same page, section 5.2.1 and 5.3.1).  The state S_t (dv x dk) is
 * stored TRANSPOSED, as H_t = S_t^T (dk rows x dv columns, fp32).  There is no
 * 1/sqrt(dk) scale on q: o_t = S_t q_t exactly as written above.
 *
 * Method of the library: the tokens of each sequence are cut into chunks of
 * 64 ("v1.0 Architecture & Design Spec", section 2.3: chunk_size 64 default;
 * "Optimization Quartet", Triton GDN kernel section 3.2: intra-chunk parallel
 * work, inter-chunk serial carry of the state).  Chunks restart at every
 * sequence start.  Arithmetic is fp32 inside, with the state held in fp32 on
 * chip; the output is stored in the caller's dtype ("Optimization Quartet",
 * Triton GDN kernel section 3.3, "FP32 inside, cast back outside").
 *
 * Conventions common to every entry point
 * ---------------------------------------
 *  - Pointers named device pointers must point to memory of the current CUDA
 *    device (cudaMalloc, cudaMallocAsync or a PyTorch CUDA tensor).  Every
 *    device pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All work is enqueued asynchronously on it; only gdn_check,
 *    and gdn_fwd_static_scratch when asked to check, synchronise.
 *  - The caller owns every buffer.  The library allocates no device memory
 *    and keeps no per-call state; it caches device attributes, and holds one
 *    256-byte static device array used only by gdn_fwd_static_scratch.
 *  - There is no CPU fallback: when the library cannot run a call it returns
 *    an error code and enqueues nothing.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Host-side validation errors (INVALID_ARG, UNSUPPORTED,
 * WORKSPACE) are returned before anything is enqueued.  Device-detected errors
 * (TIMEOUT, BAD_SEQLENS, DEVICE_CHECK) are recorded in the workspace status
 * word by the kernels and reported later by gdn_check. */
typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or aliasing  */
  GDN_ERR_UNSUPPORTED = 2,  /* well-formed but not implemented (head dims...) */
  GDN_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than required        */
  GDN_ERR_CUDA = 4,         /* a CUDA runtime call or a launch failed         */
  GDN_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up             */
  GDN_ERR_BAD_SEQLENS = 6,  /* cu_seqlens not 0 = cu[0] < cu[1] < ... = T     */
  GDN_ERR_DEVICE_CHECK = 7  /* a device-side consistency check failed         */
} gdn_status;

/* Storage type of q, k, v, beta and o.  g, the states and all arithmetic are
 * fp32 regardless. */
typedef enum gdn_dtype { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Flags for gdn_fwd. */
enum {
  /* Normalise q_t and k_t in-kernel: x / sqrt(sum(x^2) + 1e-6), fp32 (the
   * gated delta rule's q/k normalisation, part of the block's prologue).  The
   * tensor-core kernels compute each row's factor 1/|x| in fp32 from the
   * loaded bf16 tiles and fold it into the fp32 scaling of the products
   * (row and column factors of Q K^T and K K^T, the rows of W, Ud and O), so
   * the stored bf16 q and k reach the tensor cores unrounded a second time;
   * the fp32 kernel normalises in fp32. */
  GDN_QK_L2NORM = 1u << 0,
  /* Use the fp32 CUDA-core kernel even for bf16 storage (the tensor-core
   * kernel is the default for bf16).  fp32 storage always uses it. */
  GDN_FORCE_SIMT = 1u << 1,
  /* gdn_diag_fwd and gdn_diag_delta_fwd: g holds the gate's logits dt and the kernel uses
   * g = sigmoid(dt) ("Model Architecture Walkthrough", section 5.2.1). */
  GDN_GATE_SIGMOID = 1u << 2,
  /* gdn_fwd and gdn_diag_delta_fwd: beta holds logits and the kernel uses beta_t =
   * sigmoid(beta input) in fp32 (the write strength is a sigmoid of a
   * projection in the gated delta rule block; the pages' block computes its
   * gates the same way, "Model Architecture Walkthrough", section 5.4.3). */
  GDN_BETA_LOGITS = 1u << 3,
  /* gdn_fwd and gdn_fwd_static_scratch: before its first global access, every
   * block of the forward kernels checks the whole index range it will touch
   * in each buffer (q, k, v, g, beta, o, the states, out_gate: computed with
   * the kernels' own index formulas, which are monotone in token, row and
   * column) against the buffers' extents, and that each TMA box's innermost
   * coordinate lies on a 16-byte boundary.  Extents come from the shapes, or
   * are declared by the caller through gdn_fwd_debug, and the tensor maps are
   * cut to them so that no TMA box reaches past.  A violation records
   * GDN_ERR_DEVICE_CHECK with (sequence, head, site) in the status word
   * (gdn_check_record reads them) and the block ends without any access: its
   * outputs are left as they were.  The plain kernels carry one uniform
   * branch for it.  The pages' kernel asserts its inputs and raises instead of
   * falling back ("Optimization Quartet", Triton GDN kernel sections 3.3 and
   * 3.5); this is the device-side counterpart. */
  GDN_DEBUG_CHECKS = 1u << 4,
  /* gdn_fwd: let the head_dim_k 128 tensor-core kernel cut each sequence of a
   * dense call (cu_seqlens NULL, no block epilogue, no GDN_DEBUG_CHECKS) into up to 8 segments of
   * whole chunks when the (sequence, head, 64 value columns) units alone
   * leave SMs idle (gdn_fwd_split_segments gives the plan).  The later
   * segments are of equal length; the first takes the rest of the sequence
   * and is often the longest, its few CTAs starting first while the SMs they
   * leave free run the later ones.  The chunk
   * transition is affine in the state, H' = M H + X, and each output is
   * affine in the state entering the segment, o = o0 + r H, so: one launch
   * runs segment 0 from the caller's state and every later segment from a
   * zero state (o0, X) and, on dk extra columns, from the identity (r, M);
   * small kernels compose the segments' entry states in order and add r H to
   * the later segments' outputs.  The result equals the unsplit one up to
   * rounding.  The workspace must be sized with gdn_fwd_split_workspace_size.
   * Other calls ignore the flag. */
  GDN_SEQ_SPLIT = 1u << 5
};

/* Bytes of device workspace gdn_fwd needs for these sizes (>= 256; the first
 * 256 bytes hold the device status word).  Not enough for a call that
 * GDN_SEQ_SPLIT cuts into segments: size those with
 * gdn_fwd_split_workspace_size.  Never fails; returns 0 only for nonsensical
 * sizes (any argument <= 0). */
size_t gdn_fwd_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_dim_k,
                              int32_t head_dim_v, uint32_t flags);

/* Bytes of device workspace a dense gdn_fwd call with GDN_SEQ_SPLIT needs
 * (batch = num_seqs sequences of seq_len tokens): the status word, each
 * segment's entry state, X and M (fp32, up to 8 segments), and with
 * head_dim_k 128 the per-token maps r of the segments (bf16, [tokens][heads]
 * [head_dim_k]).  A split call with less returns GDN_ERR_WORKSPACE; calls the
 * plan leaves unsplit need only gdn_fwd_workspace_size.  Returns 0 for
 * nonsensical sizes. */
size_t gdn_fwd_split_workspace_size(int32_t num_seqs, int32_t seq_len, int32_t num_heads,
                                    int32_t head_dim_k, int32_t head_dim_v);

/* Enqueue a zero fill of the first `workspace_bytes` bytes of `workspace` on
 * `stream`.  A workspace must be zeroed once before its first use by gdn_fwd
 * (gdn_check clears the status word it reports, so one fill is enough).
 * No passage of the pages defines a workspace: it carries the device status
 * word through which this library surfaces errors found on the GPU (the
 * pages' kernel raises instead of falling back: "Optimization Quartet",
 * Triton GDN kernel section 3.5).  Returns GDN_ERR_WORKSPACE for a NULL or
 * too small (< 256 bytes) workspace, GDN_ERR_CUDA if the fill cannot be
 * enqueued; the workspace stays owned by the caller. */
gdn_status gdn_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_fwd -- forward pass of the gated delta rule (the operation above).
 *
 * Shapes (all dense, row-major, "token-major, head-minor"):
 *   q, k          [batch, seq_len, num_heads, head_dim_k]    dtype     device
 *   v             [batch, seq_len, num_heads, head_dim_v]    dtype     device
 *   g             [batch, seq_len, num_heads]                float32   device
 *   beta          [batch, seq_len, num_heads]                dtype     device
 *   initial_state [num_seqs, num_heads, head_dim_k, head_dim_v] float32 device, or NULL (= zeros)
 *   cu_seqlens    [num_seqs + 1] int32 device, or NULL
 *   o             [batch, seq_len, num_heads, head_dim_v]    dtype     device (written)
 *   final_state   [num_seqs, num_heads, head_dim_k, head_dim_v] float32 device (written), or NULL
 *   D_skip        [num_heads]                                float32   device, or NULL
 *   out_gate      [batch, seq_len, num_heads]                float32   device, or NULL
 *
 * Block epilogue (optional, fused into the output store): the GDN block's
 * skip connection and output gate ("Model Architecture Walkthrough", section
 * 5.5, step 6, and section 5.6), with v the value input of the recurrence:
 *
 *     o_t <- (o_t + D_skip[h] v_t) * out_gate[t, h]
 *
 * A NULL D_skip reads as 0 and a NULL out_gate as 1; with both NULL o is the
 * recurrence output itself.  out_gate is the per-(token, head) scalar the
 * pages form by averaging sigmoid(g_proj x) over the head dimension (section
 * 5.4.3); that projection stays with the caller.
 *
 * Sequences: with cu_seqlens == NULL the batch rows are the sequences and
 * num_seqs must equal batch.  With cu_seqlens != NULL, batch must be 1 and
 * sequence n covers tokens cu_seqlens[n] .. cu_seqlens[n+1]-1 of the packed
 * seq_len tokens; the offsets must satisfy cu_seqlens[0] = 0, non-decreasing,
 * cu_seqlens[num_seqs] = seq_len.  An empty sequence (equal offsets) reads
 * nothing and its final state is its initial state (zeros without one).
 * These offsets live in device memory, so they are checked by the kernel:
 * a sequence whose bounds break the rule writes nothing and records
 * GDN_ERR_BAD_SEQLENS for gdn_check.  No state crosses a sequence boundary.
 * seq_len = 0 (no tokens at all) is legal: nothing is read, cu_seqlens
 * included, and every final state is its initial state.
 *
 * Values: g_t is the natural log of the decay alpha_t (expected <= 0; not
 * clamped).  beta_t is used as given (expected in [0, 1]; not clamped), or
 * with GDN_BETA_LOGITS as sigmoid(beta input).  The state element (i, j) of
 * H = S^T multiplies key dimension i and value dimension j.
 *
 * flags: any of GDN_QK_L2NORM, GDN_BETA_LOGITS, GDN_FORCE_SIMT, GDN_DEBUG_CHECKS,
 * GDN_SEQ_SPLIT.
 *
 * Supported sizes: head_dim_k in {32, 64, 128}; head_dim_v a multiple of 32
 * in [32, 256]; num_heads >= 1; num_seqs in [1, 65535]; chunk_size in {32,
 * 64, 128} except 128 with head_dim_k 128.  The result does not depend on
 * chunk_size beyond rounding; 64 is the pages' default.  With bf16 storage
 * and head_dim_k 64, 32 and 128 run on tensor-core variants of their own
 * (gdn_fwd_kernel_name_chunk names the kernel); other chunk sizes of other
 * shapes run on the fp32 CUDA-core kernel (the pages sweep chunk_size over
 * {32, 64, 128}: "v1.0 Architecture & Design Spec", section 2.3).
 * Anything else returns GDN_ERR_UNSUPPORTED (or INVALID_ARG if malformed).
 *
 * Aliasing: o and final_state must not overlap any input.  final_state may be
 * the same buffer as initial_state (each state is read before it is written),
 * which chains calls: a sequence split in two calls, with the first call's
 * final_state passed as the second call's initial_state, gives the result of
 * one call up to rounding.
 *
 * workspace: device, at least gdn_fwd_workspace_size(...) bytes, zeroed once
 * before first use (gdn_workspace_init).  Calls that share a workspace must
 * not run concurrently on different streams.
 *
 * Returns GDN_OK once the work is enqueued (errors detected on the device are
 * reported by gdn_check), or an error code with nothing enqueued.
 */
gdn_status gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                   const void *beta, const float *initial_state,
                   const int32_t *cu_seqlens, void *o, float *final_state,
                   const float *D_skip, const float *out_gate,
                   int32_t batch, int32_t seq_len, int32_t num_heads,
                   int32_t head_dim_k, int32_t head_dim_v, int32_t num_seqs,
                   int32_t chunk_size, gdn_dtype dtype, uint32_t flags,
                   void *workspace, size_t workspace_bytes, void *stream);

/* The number of segments S GDN_SEQ_SPLIT cuts each sequence of a gdn_fwd
 * call with these arguments (and no block epilogue: a call with D_skip or
 * out_gate is never split, nor one with GDN_DEBUG_CHECKS) into, on the
 * current device (the plan depends on
 * its SM count): S >= 2 when the call is split, and then gdn_fwd launches 3
 * kernels (every segment in one launch, the S - 1 composition steps in one,
 * the output correction); 1 when it is not split (one kernel).  varlen != 0
 * stands for a call with cu_seqlens (never split).  Returns 0 for sizes
 * gdn_fwd rejects.  Host only; launches nothing. */
int32_t gdn_fwd_split_segments(int32_t num_seqs, int32_t seq_len, int32_t num_heads,
                               int32_t head_dim_k, int32_t head_dim_v, int32_t chunk_size,
                               gdn_dtype dtype, uint32_t flags, int32_t varlen);

/* Elements (not bytes) each buffer of a forward call holds, for
 * gdn_fwd_debug.  A field of a NULL buffer is ignored. */
typedef struct gdn_extents {
  int64_t q, k, v, g, beta, o;
  int64_t initial_state, final_state, out_gate;
} gdn_extents;

/*
 * gdn_fwd_debug -- gdn_fwd with GDN_DEBUG_CHECKS, against extents the caller
 * declares (for views into larger allocations, or to test the checks).
 * Arguments, validation and results are gdn_fwd's; `declared` is a host
 * pointer read during the call (NULL = extents from the shapes).  Every field
 * must be >= 0 (else GDN_ERR_INVALID_ARG).  A declared extent smaller than the
 * range some block of the call would touch makes that block record
 * GDN_ERR_DEVICE_CHECK and end without touching anything; the other blocks run
 * as usual.  With seq_len = 0 the state copy is checked on the host and an
 * undersized state extent returns GDN_ERR_INVALID_ARG.  No passage of the
 * pages defines this call (see GDN_DEBUG_CHECKS).
 */
gdn_status gdn_fwd_debug(const void *q, const void *k, const void *v, const float *g,
                         const void *beta, const float *initial_state,
                         const int32_t *cu_seqlens, void *o, float *final_state,
                         const float *D_skip, const float *out_gate, int32_t batch,
                         int32_t seq_len, int32_t num_heads, int32_t head_dim_k,
                         int32_t head_dim_v, int32_t num_seqs, int32_t chunk_size,
                         gdn_dtype dtype, uint32_t flags, void *workspace,
                         size_t workspace_bytes, const gdn_extents *declared, void *stream);

/*
 * gdn_fwd_static_scratch -- gdn_fwd for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point; it exists for
 * callers that must not call cudaMalloc: a plugin or extension running inside
 * a host framework that owns every device allocation through its own pool, a
 * latency-critical loop where an allocation could synchronise the device, or
 * a process held to a fixed device-memory budget.  Such a caller still passes
 * its inputs and outputs, but no workspace.
 *
 * Instead of a caller workspace, the 256-byte device status record lives in a
 * file-scope __device__ array inside the library.  Every GPU that loads the
 * library holds those 256 bytes until the process exits.  The array is shared
 * by every call on that device and keeps the last call's contents, so each
 * call first enqueues a zero fill of it on `stream`.  Calls that overlap on
 * the GPU (different streams, no ordering between them) race on the array and
 * may report each other's device errors; serialise them.
 *
 * Each call made outside stream capture, with the device current, looks up the
 * array's device address (cudaGetSymbolAddress, which allocates nothing) and
 * remembers it per device; a call made while `stream` is capturing uses the
 * remembered address.  So make the first call on a device before any stream
 * capture begins, and after a cudaDeviceReset make one uncaptured call before
 * capturing again.
 *
 * Arguments are those of gdn_fwd without workspace/workspace_bytes, plus
 * `check`: when nonzero the call synchronises `stream` after the launch and
 * returns any error the kernel recorded (GDN_ERR_BAD_SEQLENS, ...); when zero
 * it returns once the work is enqueued and device-detected errors are not
 * reported.  Every host-side check of gdn_fwd runs first; a call that fails
 * one, or whose scratch need (gdn_fwd_workspace_size) exceeds the 256-byte
 * array (GDN_ERR_WORKSPACE), returns its error and enqueues nothing.  The
 * call performs no device allocation or free.
 */
gdn_status gdn_fwd_static_scratch(const void *q, const void *k, const void *v, const float *g,
                                  const void *beta, const float *initial_state,
                                  const int32_t *cu_seqlens, void *o, float *final_state,
                                  const float *D_skip, const float *out_gate, int32_t batch, int32_t seq_len, int32_t num_heads,
                                  int32_t head_dim_k, int32_t head_dim_v, int32_t num_seqs,
                                  int32_t chunk_size, gdn_dtype dtype, uint32_t flags,
                                  int32_t check, void *stream);

/*
 * gdn_decode -- one recurrent step of the operation above per (sequence,
 * head): the token-by-token form used for incremental inference, with the
 * state carried between calls ("Model Architecture Walkthrough", section
 * 5.5, step 5, is the per-token recurrence; section 5.2.1 the decay).  Per
 * (n, h), with H = S^T the fp32 state:
 *
 *     u = beta (v - alpha H^T k),   H' = alpha H + k u^T,   o = H'^T q
 *
 * which is gdn_fwd on one token with initial_state H and final_state H', up
 * to rounding.
 *
 *   q, k       [num_seqs, num_heads, head_dim_k]                 dtype    device
 *   v          [num_seqs, num_heads, head_dim_v]                 dtype    device
 *   g          [num_seqs, num_heads]                             float32  device
 *   beta       [num_seqs, num_heads]                             dtype    device
 *   state_in   [num_seqs, num_heads, head_dim_k, head_dim_v]     float32  device, or NULL (= zeros)
 *   state_out  [num_seqs, num_heads, head_dim_k, head_dim_v]     float32  device (written)
 *   o          [num_seqs, num_heads, head_dim_v]                 dtype    device (written)
 *
 * flags: GDN_QK_L2NORM only.  Sizes as gdn_fwd (head_dim_k in {32, 64, 128},
 * head_dim_v a multiple of 32 in [32, 256], num_seqs and num_heads <= 65535).
 * state_out may be the same buffer as state_in (updated in place); otherwise
 * outputs must not overlap any input.  No workspace: the step has no
 * device-detected error.  Returns GDN_OK once enqueued, or an error code with
 * nothing enqueued.  The pages have no decode entry point; their model
 * carries the state token by token in the same recurrence.
 */
gdn_status gdn_decode(const void *q, const void *k, const void *v, const float *g,
                      const void *beta, const float *state_in, float *state_out, void *o,
                      int32_t num_seqs, int32_t num_heads, int32_t head_dim_k,
                      int32_t head_dim_v, gdn_dtype dtype, uint32_t flags, void *stream);

/*
 * gdn_diag_fwd -- the HyMo pages' own recurrence: per-state-row (diagonal)
 * decay, separate write and read keys, no erase term ("Model Architecture
 * Walkthrough", section 5.2.1; "Optimization Quartet", Triton GDN kernel
 * section 3.2, whose wrapper takes the same five tensors v, b, c, g, A_log).
 * Per batch row n and head h, tokens t = 1..seq_len:
 *
 *     h_t = exp(g_t A) (.) h_{t-1} + b_t v_t^T,    o_t = h_t^T c_t,
 *     A   = -exp(A_log[h])   (one negative rate per state row s)
 *
 * where h_t is d_state x head_dim (fp32) and exp(g_t A) (.) scales row s of
 * the state by exp(g_t A_s).  Arithmetic is fp32 inside; o is stored in the
 * caller's dtype.
 *
 *   v              [batch, seq_len, num_heads, head_dim]       dtype    device
 *   b, c           [batch, seq_len, num_heads, d_state]        dtype    device
 *   g              [batch, seq_len, num_heads]                 float32  device
 *   A_log          [num_heads, d_state]                        float32  device
 *   D_skip         [num_heads]                                 float32  device, or NULL
 *   out_gate       [batch, seq_len, num_heads]                 float32  device, or NULL
 *   initial_state  [batch, num_heads, d_state, head_dim]       float32  device, or NULL (= zeros)
 *   o              [batch, seq_len, num_heads, head_dim]       dtype    device (written)
 *   final_state    [batch, num_heads, d_state, head_dim]       float32  device (written), or NULL
 *
 * Values: g_t is the positive gate (a sigmoid output on the pages) and is
 * used as given, or with flags = GDN_GATE_SIGMOID it holds the logits and
 * g_t = sigmoid(g input); any real g_t and A_log are accepted, the decay
 * factors are products of exp(g_t A_s) and never overflow for g_t >= 0.
 *
 * Block epilogue (same page, section 5.5, step 6), fused into the output
 * store when D_skip or out_gate is given:
 *
 *     o_t <- (o_t + D_skip[h] v_t) * out_gate[n, t, h]
 *
 * with a missing D_skip read as 0 and a missing out_gate as 1.
 *
 * Supported sizes: d_state == 32 and head_dim == 32 (the pages' production
 * shape); batch, num_heads, seq_len >= 1 with batch * num_heads *
 * ceil(seq_len / 128) < 2^31.  flags: 0 or GDN_GATE_SIGMOID.  Anything else returns
 * GDN_ERR_UNSUPPORTED (or INVALID_ARG if malformed).
 *
 * Aliasing as gdn_fwd: o and final_state overlap no input; final_state may be
 * initial_state.
 *
 * workspace: device, at least gdn_diag_workspace_size(...) bytes, zeroed once
 * before its first use (gdn_workspace_init); it carries a launch counter from
 * call to call, so a call that failed to complete (a CUDA error) requires a
 * new gdn_workspace_init.  Calls sharing a workspace must be ordered (same
 * stream).  Device-detected errors (GDN_ERR_TIMEOUT) are reported by
 * gdn_check.  Returns GDN_OK once enqueued, or an error code with nothing
 * enqueued.
 */
size_t gdn_diag_workspace_size(int32_t batch, int32_t seq_len, int32_t num_heads,
                               int32_t d_state, int32_t head_dim);
gdn_status gdn_diag_fwd(const void *v, const void *b, const void *c, const float *g,
                        const float *A_log, const float *D_skip, const float *out_gate,
                        const float *initial_state, void *o,
                        float *final_state, int32_t batch, int32_t seq_len, int32_t num_heads,
                        int32_t d_state, int32_t head_dim, gdn_dtype dtype, uint32_t flags,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_diag_delta_fwd -- the pages' per-row (diagonal) decay combined with the
 * delta rule: the decay of gdn_diag_fwd ("Model Architecture Walkthrough",
 * section 5.2.1: exp(g_t A) scales row s of the state by exp(g_t A_s), A =
 * -exp(A_log[h])) followed by the gated delta rule's erase and write with
 * strength beta_t, the write key b_t also being the erase key.  Per batch row
 * n and head h, tokens t = 1..seq_len:
 *
 *     hbar = exp(g_t A) (.) h_{t-1}
 *     h_t  = hbar + beta_t b_t (v_t - hbar^T b_t)^T,     o_t = h_t^T c_t
 *
 * h_t is d_state x head_dim (fp32).  With beta_t = 1 and a unit b_t the state
 * returns v_t for the key b_t right after the write; with all rates of a
 * head equal it is gdn_fwd's recurrence with q = c, k = b and the natural-log
 * gate g_t A.  Arithmetic is fp32 inside; o is stored in the caller's dtype.
 *
 *   v              [batch, seq_len, num_heads, head_dim]       dtype    device
 *   b, c           [batch, seq_len, num_heads, d_state]        dtype    device
 *   g              [batch, seq_len, num_heads]                 float32  device
 *   A_log          [num_heads, d_state]                        float32  device
 *   beta           [batch, seq_len, num_heads]                 dtype    device
 *   D_skip         [num_heads]                                 float32  device, or NULL
 *   out_gate       [batch, seq_len, num_heads]                 float32  device, or NULL
 *   initial_state  [batch, num_heads, d_state, head_dim]       float32  device, or NULL (= zeros)
 *   o              [batch, seq_len, num_heads, head_dim]       dtype    device (written)
 *   final_state    [batch, num_heads, d_state, head_dim]       float32  device (written), or NULL
 *
 * flags: GDN_GATE_SIGMOID (g holds logits, g_t = sigmoid(g input)) and
 * GDN_BETA_LOGITS (beta_t = sigmoid(beta input)); the block epilogue
 * o_t <- (o_t + D_skip[h] v_t) * out_gate[n, t, h] as in gdn_diag_fwd.  Keys
 * are used as given (the erase is a projection only for beta_t |b_t|^2 <= 2).
 *
 * Supported sizes: d_state == 32 and head_dim == 32; batch, num_heads,
 * seq_len >= 1 with batch * num_heads * ceil(seq_len / 128) < 2^31.  Anything
 * else returns GDN_ERR_UNSUPPORTED (or INVALID_ARG if malformed).  Aliasing as
 * gdn_diag_fwd.
 *
 * workspace: device, at least gdn_diag_delta_workspace_size(...) bytes, zeroed
 * once before its first use (gdn_workspace_init); it carries a launch counter
 * from call to call (a call that failed to complete requires a new
 * gdn_workspace_init), and calls sharing it must be ordered (same stream).
 * The 128-token segments of a sequence run in parallel and are joined through
 * their affine state maps in the workspace.  Device-detected errors
 * (GDN_ERR_TIMEOUT) are reported by gdn_check.  Returns GDN_OK once enqueued,
 * or an error code with nothing enqueued.
 */
size_t gdn_diag_delta_workspace_size(int32_t batch, int32_t seq_len, int32_t num_heads,
                                     int32_t d_state, int32_t head_dim);
gdn_status gdn_diag_delta_fwd(const void *v, const void *b, const void *c, const float *g,
                              const float *A_log, const void *beta, const float *D_skip,
                              const float *out_gate, const float *initial_state, void *o,
                              float *final_state, int32_t batch, int32_t seq_len,
                              int32_t num_heads, int32_t d_state, int32_t head_dim,
                              gdn_dtype dtype, uint32_t flags, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * gdn_conv_silu -- prologue of the HyMo GDN block: causal depthwise conv1d,
 * then SiLU ("Model Architecture Walkthrough", section 5.4.1: a depthwise
 * Conv1d over d_inner channels with d_conv taps and padding d_conv - 1, the
 * tail trimmed so that it is causal; section 5.5, step 2: SiLU after it).
 * Per batch row n, token t and channel ch:
 *
 *     y[n, t, ch] = silu( sum_{k < taps} w[ch, k] * x[n, t - (taps - 1) + k, ch] )
 *     silu(z) = z / (1 + exp(-z))
 *
 * where x at t < 0 is x_prev[n, taps - 1 + t, ch] when x_prev is given, else 0.
 * (w[ch, k] is PyTorch's Conv1d weight[ch, 0, k].)  fp32 arithmetic; y in the
 * caller's dtype.
 *
 *   x        [batch, seq_len, channels]        dtype    device
 *   w        [channels, taps]                  float32  device
 *   x_prev   [batch, taps - 1, channels]       dtype    device, or NULL (= zeros)
 *   y        [batch, seq_len, channels]        dtype    device (written)
 *   x_tail   [batch, taps - 1, channels]       dtype    device (written), or NULL:
 *            the last taps - 1 inputs (of x_prev followed by x), the x_prev of
 *            the next call when a sequence is fed in pieces
 *
 * Supported: 1 <= taps <= 4 (the pages use 4); channels a multiple of 4;
 * batch <= 65535.  Outputs must not overlap any input
 * (to chain calls, alternate two prefix buffers).  No workspace; no
 * device-detected error.  Returns GDN_OK once enqueued, or an error code with
 * nothing enqueued.
 */
gdn_status gdn_conv_silu(const void *x, const float *w, const void *x_prev, void *y,
                         void *x_tail, int32_t batch, int32_t seq_len, int32_t channels,
                         int32_t taps, gdn_dtype dtype, void *stream);

/*
 * gdn_bwd -- backward pass of gdn_fwd's operation: the vector-Jacobian
 * products of o (and of the final state) with respect to every input.  It
 * recomputes what it needs from the inputs, as the pages' kernel does
 * ("Optimization Quartet", Triton GDN kernel section 3.4; the backward runs
 * the recurrence backwards in time: "Model Architecture Walkthrough", section
 * 6.5).  With s_t = H_{t-1}^T k_t, u_t = beta_t (v_t - alpha_t s_t), and dH
 * the running gradient of the state (d_final_state at the end), for t = T..1:
 *
 *   dH += q_t do_t^T,  dq_t = H_t do_t,  du = dH^T k_t,  dv_t = beta_t du,
 *   dbeta_t = <du, v_t - alpha_t s_t>,  dg_t = alpha_t (<dH, H_{t-1}> - beta_t <du, s_t>),
 *   dk_t = dH u_t - alpha_t beta_t H_{t-1} du,  dH <- alpha_t (dH - beta_t k_t du^T)
 *
 * and d_initial_state is the final dH.
 *
 *   q, k, v, g, beta, initial_state, cu_seqlens   as gdn_fwd (inputs)
 *   d_o            [batch, seq_len, num_heads, head_dim_v]     dtype    device
 *   d_final_state  [num_seqs, num_heads, head_dim_k, head_dim_v] float32 device, or NULL (= zeros)
 *   dq, dk         [batch, seq_len, num_heads, head_dim_k]     float32  device (written)
 *   dv             [batch, seq_len, num_heads, head_dim_v]     float32  device (written)
 *   dg, dbeta      [batch, seq_len, num_heads]                 float32  device (written)
 *   d_initial_state [num_seqs, num_heads, head_dim_k, head_dim_v] float32 device (written), or NULL
 *
 * All gradients are fp32 whatever the storage dtype.  Two paths compute them:
 * - bf16 storage with head_dim_k, head_dim_v in {32, 64}: the same algebra in
 *   the chunked (WY) form of gdn_fwd, with bf16 tensor-core products and fp32
 *   accumulation (the precision class of gdn_fwd's tensor-core path); every
 *   gradient is written once, so results are bitwise reproducible;
 * - otherwise: the recurrence above token by token in fp32, from state
 *   checkpoints; dq, dk, dg and dbeta are summed with atomics over
 *   value-column slices, so they agree from run to run to fp32 rounding only.
 * Sizes as gdn_fwd (chunk 64); flags must be 0.  No gradient buffer may
 * overlap an input or another gradient.  workspace: at least
 * gdn_bwd_workspace_size(...) bytes, enough for either path (per-chunk
 * records of the chunked form, or state checkpoints and per-CTA scratch); the
 * first 256 bytes are the status word (zero it once with gdn_workspace_init).
 * Device-detected errors (bad cu_seqlens) are reported by gdn_check.  Returns
 * GDN_OK once enqueued, or an error code with nothing enqueued.  seq_len is
 * the packed token count when cu_seqlens is given.  Empty sequences and
 * seq_len = 0 are legal as for gdn_fwd: d_initial_state of an empty sequence
 * is its d_final_state (zeros without one).
 */
size_t gdn_bwd_workspace_size(int32_t num_seqs, int32_t seq_len, int32_t num_heads,
                              int32_t head_dim_k, int32_t head_dim_v);
gdn_status gdn_bwd(const void *q, const void *k, const void *v, const float *g,
                   const void *beta, const float *initial_state, const int32_t *cu_seqlens,
                   const void *d_o, const float *d_final_state, float *dq, float *dk,
                   float *dv, float *dg, float *dbeta, float *d_initial_state, int32_t batch,
                   int32_t seq_len, int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                   int32_t num_seqs, gdn_dtype dtype, uint32_t flags, void *workspace,
                   size_t workspace_bytes, void *stream);

/* Synchronise `stream`, read the status word in `workspace`, clear it, and
 * return it (GDN_OK if no kernel recorded an error since the last check).
 * Also returns GDN_ERR_CUDA if the stream synchronisation itself failed, and
 * GDN_ERR_WORKSPACE for a NULL workspace.  This is how errors that only the
 * kernels can see (bad device-side cu_seqlens, a bounded wait that gave up,
 * a GDN_DEBUG_CHECKS violation) reach the caller as a clear error code
 * rather than a silent wrong result.  No passage of the pages defines this
 * call; it follows their rule that failures surface as errors, with no silent
 * fallback ("Optimization Quartet", Triton GDN kernel section 3.5). */
gdn_status gdn_check(void *workspace, void *stream);

/* gdn_check that also returns where the recorded error arose: the sequence
 * and head of the block that recorded it and a site code (for
 * GDN_ERR_DEVICE_CHECK: 1 q, 2 k, 3 v, 4 g, 5 beta, 6 o, 7 initial_state,
 * 8 final_state, 9 out_gate, 10 a TMA box coordinate off its 16-byte
 * boundary; 0 otherwise).  Any output pointer may be NULL; with GDN_OK they
 * read -1, -1, 0.  Same synchronisation, clearing and return values as
 * gdn_check (and the same footing in the pages). */
gdn_status gdn_check_record(void *workspace, void *stream, int32_t *seq, int32_t *head,
                            int32_t *site);

/* Static, human-readable name of a status code (never NULL; the string is
 * owned by the library).  Unknown codes give "GDN_ERR_UNKNOWN".  No passage
 * of the pages defines it: it gives the clear error message that the pages'
 * no-silent-fallback rule asks for ("Optimization Quartet", Triton GDN kernel
 * section 3.5). */
const char *gdn_status_string(int32_t status);

/* Name of the kernel gdn_fwd would launch for these arguments with
 * chunk_size 64 ("simt_fp32", "simt_bf16", "tc64_bf16", "tc128_bf16") or NULL
 * when the arguments are unsupported.  Host only. */
const char *gdn_fwd_kernel_name(int32_t head_dim_k, int32_t head_dim_v,
                                gdn_dtype dtype, uint32_t flags);

/* The same for any chunk_size: "tcc32_bf16" / "tcc128_bf16" for the
 * tensor-core chunk-size variants (bf16 storage, head_dim_k 64, chunk_size 32
 * or 128), else the names above; NULL when the arguments are unsupported.
 * Host only. */
const char *gdn_fwd_kernel_name_chunk(int32_t head_dim_k, int32_t head_dim_v,
                                      int32_t chunk_size, gdn_dtype dtype, uint32_t flags);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
