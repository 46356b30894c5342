/*
 * ttt_mlp.h -- C ABI of the B300 (sm_103a) In-Place TTT fast-weight MLP layer.
 *
 * What the layer computes (sources: "In-Place Test-Time Training",
 * paperlayer.ai summary of arXiv 2604.06169v1, section 3 "In-Place Adaptation",
 * "Chunk-Wise Updates", "LM-Aligned Objective" and appendix B "Context Parallel
 * Algorithm"; iplexlaw.co.kr walkthrough of the same paper, sections 2-4 and 6):
 *
 *   The tokens of a call are cut into non-overlapping chunks of C tokens
 *   (a document start restarts the chunking; the last chunk may be short).
 *   For every chunk c, in order:
 *     Z_c     = SiLU(X_c W_gate^T) (.) (X_c W_up^T)          gated intermediate
 *     O_c     = Z_c W_c^T                                      apply (pre-update W)
 *     U_c[t]  = sum_{j<k} conv[j] (.) X0_c[t+1+j]              zero past the chunk end
 *     V_c     = U_c W_target                                   next-token target
 *     W_{c+1} = W_c + eta V_c^T Z_c                            update
 *   The fast weight W (= the MLP's down projection) starts at the frozen
 *   W_down = W_0 and is reset to W_0 at every document start.
 *   Options (ttt_mlp_config): the target window (target_mode, the ablation
 *   axes and reconstruction target of section 4 / section 2 of the summary
 *   page) and per-chunk update clipping (clip_tau: each chunk's delta
 *   eta V_c^T Z_c is scaled by min(1, clip_tau / ||eta V_c^T Z_c||_F); the
 *   summary page's appendix C.2 and section 6 of the walkthrough bound the
 *   update delta's Frobenius norm).
 *
 * Conventions shared by every call:
 *   - Layouts are row-major.  W_gate, W_up: f x d; W_down (W_0): d x f;
 *     conv: k x d; W_target: d x d given as in x out (V = U W_target);
 *     X, X0, O: n x d (row = token); the fast weight W: d x f, always fp32.
 *   - Activations and weights are fp32 (TTT_F32) or bf16 (TTT_BF16) as set by
 *     ttt_mlp_config.act_dtype; O has the same dtype.
 *   - Device memory is never allocated by the library.  The caller owns the
 *     weights, the workspace and the per-call buffers; weights and workspace
 *     are borrowed by the handle and must outlive it.  The handle owns only
 *     host memory.  Pointers are device pointers unless named *_host.
 *   - Every call is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns without synchronising, except where stated.
 *   - No exception or abort crosses the ABI.  Arguments are checked on the
 *     host before anything is enqueued; a call that fails its checks changes
 *     no state and returns TTT_EINVAL or TTT_EUNSUPPORTED.  CUDA errors map
 *     to TTT_ECUDA.  ttt_mlp_last_error() gives the text of the last failure.
 *   - Kernels never hang: every in-kernel wait is bounded.  A wait that runs
 *     out records a code in the workspace's error word; ttt_mlp_check()
 *     reports it as TTT_ETIMEOUT.
 *   - Setting the environment variable TTT_FAULT to one of
 *     create|forward|reset|get|set|check makes that call fail with
 *     TTT_EFAULT_INJECTED before it does anything (host-side fault injection).
 *     TTT_FAULT=kernel_wait instead makes the next forward call's
 *     target-projection kernel withhold one of its own operand loads, so
 *     that kernel's bounded waits run out (about 4 s): the call itself
 *     succeeds, ttt_mlp_check then reports TTT_ETIMEOUT, and the slot's fast
 *     weight is undefined until it is reset.  TTT_FAULT=group_wait does the
 *     same in the call's first fused apply+update (group) launch, whose
 *     other tiles then time out on the completion counters the withheld
 *     tile never raises.  (Both test the failure path without faulting the
 *     GPU.)
 */
#ifndef TTT_MLP_H
#define TTT_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TTT_OK = 0,
  TTT_EINVAL = 1,           /* a bad argument (null pointer, size, alignment, order) */
  TTT_EUNSUPPORTED = 2,     /* valid but outside what this build supports */
  TTT_ECUDA = 3,            /* a CUDA runtime/driver call failed */
  TTT_ETIMEOUT = 4,         /* a bounded in-kernel wait ran out (see ttt_mlp_check) */
  TTT_EFAULT_INJECTED = 5   /* TTT_FAULT named this call */
} ttt_status;

typedef enum { TTT_F32 = 0, TTT_BF16 = 1 } ttt_dtype;

/* Target window of U[t] = sum_{j<k} conv[j] (.) X0[t + off(j)]; every term
 * whose token lies outside t's chunk is zero. */
typedef enum {
  TTT_TARGET_NEXT = 0,     /* off(j) = 1 + j: next token onwards (default) */
  TTT_TARGET_CURRENT = 1,  /* off(j) = j: current token onwards (k = 1: reconstruction target) */
  TTT_TARGET_CAUSAL = 2    /* off(j) = 1 - j: causal window ending at the next token */
} ttt_target_mode;

typedef struct {
  int32_t d;            /* model width; >= 8 and a multiple of 8 */
  int32_t f;            /* MLP intermediate width; >= 8 and a multiple of 8 */
  int32_t chunk;        /* C, tokens per chunk; 1..1024 */
  int32_t conv_k;       /* depthwise Conv1D taps k; 1..8 */
  int32_t n_docs;       /* document slots; each has its own fast weight; >= 1 */
  float eta;            /* fast-weight learning rate */
  int32_t act_dtype;    /* ttt_dtype of X, X0, O and all weights */
  int64_t max_tokens;   /* largest n_tokens of one forward call; >= 1 */
  int32_t target_mode;  /* ttt_target_mode */
  float clip_tau;       /* per-chunk update clipping threshold; 0 = off, else > 0 */
} ttt_mlp_config;

typedef struct ttt_mlp ttt_mlp; /* opaque handle */

/* Bytes of device workspace a handle with this configuration needs (0 if the
 * configuration is invalid).  The workspace holds the n_docs fast weights
 * (fp32 values; on the tcgen05 path each is kept as two 16-bit planes, the
 * upper half of its bits rounded half up in magnitude -- the bf16 operand of
 * the apply -- twice, and the exact signed remainder), the per-call
 * intermediates (Z, U, V, the intra-group Gram blocks), host-staging buffers
 * and a small control area.  Host only; no CUDA call. */
size_t ttt_mlp_workspace_bytes(const ttt_mlp_config* cfg);

/* Create a handle.  The five weight pointers are device buffers of act_dtype
 * in the layouts above; they must be 16-byte aligned and stay valid and
 * unchanged for the handle's lifetime (W_0 is read again at every reset).
 * `workspace` is a device buffer of at least ttt_mlp_workspace_bytes(cfg)
 * bytes, 256-byte aligned.  Enqueues: every slot's W <- W_0 and a transposed
 * copy of W_target.  On success *out receives the handle. */
ttt_status ttt_mlp_create(const ttt_mlp_config* cfg, const void* w_gate, const void* w_up,
                          const void* w_down0, const void* conv_w, const void* w_target,
                          void* workspace, size_t workspace_bytes, void* stream,
                          ttt_mlp** out);

/* The workspace in two parts, for several handles (for example the layers of
 * a stack) that share one scratch buffer.  The state part holds what belongs
 * to one handle across calls: a control block (the in-kernel error word and
 * tile counters), the n_docs fast weights and the transposed W_target.  The scratch part holds what one forward call needs
 * and leaves behind: Z, U, V, the intra-group Gram blocks and the
 * host-staging buffers.  ttt_mlp_workspace_bytes(cfg) is the state part
 * rounded up to 256 bytes plus the scratch part.  Both return 0 for an
 * invalid configuration.  Host only; no CUDA call. */
size_t ttt_mlp_state_bytes(const ttt_mlp_config* cfg);
size_t ttt_mlp_scratch_bytes(const ttt_mlp_config* cfg);

/* ttt_mlp_create with the two parts given separately: `state` of at least
 * ttt_mlp_state_bytes(cfg) bytes and `scratch` of at least
 * ttt_mlp_scratch_bytes(cfg) bytes, both device buffers, 256-byte aligned,
 * not overlapping.  The state is the handle's alone; the scratch may be shared
 * by handles whose configurations need no more than its size, provided their
 * calls never overlap on the GPU (one stream, or ordered by the caller): a
 * forward call overwrites the scratch, and ttt_mlp_intermediates() shows the
 * last call of any handle that shares it.  Otherwise as ttt_mlp_create
 * (which is this call with the workspace cut into its two parts). */
ttt_status ttt_mlp_create_split(const ttt_mlp_config* cfg, const void* w_gate, const void* w_up,
                                const void* w_down0, const void* conv_w, const void* w_target,
                                void* state, size_t state_bytes, void* scratch,
                                size_t scratch_bytes, void* stream, ttt_mlp** out);

/* Run the layer over n_tokens tokens of document slot `doc`, continuing that
 * slot's fast weight.  x, x0: n_tokens x d device buffers (x0 may equal x);
 * o: n_tokens x d output (must not overlap x or x0).  doc_starts: host array
 * of n_doc_starts strictly increasing offsets in [0, n_tokens) at which a new
 * document begins (W <- W_0 there); may be NULL when n_doc_starts == 0.  The
 * call always starts a fresh chunk at token 0; its trailing partial chunk is
 * processed as a short chunk, and the slot's W afterwards is the state after
 * the last chunk.  0 <= n_tokens <= max_tokens. */
ttt_status ttt_mlp_forward_chunks(ttt_mlp* h, int32_t doc, const void* x, const void* x0,
                                  int64_t n_tokens, const int64_t* doc_starts,
                                  int32_t n_doc_starts, void* o, void* stream);

/* The block's static MLP, o = SwiGLU(x) W_0^T = (SiLU(x W_gate^T) (.)
 * (x W_up^T)) W_down^T, with the frozen W_down and no fast weight: the
 * ordinary MLP block of the layers that do not carry In-Place TTT (the
 * summary page's appendix C.3 puts TTT in every sixth MLP block; the others
 * are unchanged), and what the layer computes with eta = 0.  x, o:
 * n_tokens x d device buffers (o must not overlap x); 0 <= n_tokens <=
 * max_tokens.  Uses the scratch part; reads and writes no fast weight. */
ttt_status ttt_mlp_forward_static(ttt_mlp* h, const void* x, int64_t n_tokens, void* o,
                                  void* stream);

/* The same call with host buffers: x_host / x0_host are copied to device
 * staging inside the workspace, the layer runs, and O is copied back into
 * o_host.  The call is cut at group starts into segments of about 8192 tokens
 * (TTT_HOST_SEGMENT overrides; on a shared scratch the first segment is half
 * as long, since its input copy cannot overlap the previous call there), the
 * last segment being the call's last group alone (its output copy is the one
 * no layer overlaps); the segments give the same bits as one call.  Segment
 * k+1's input copy and segment k-1's output copy run on two copy streams of
 * the handle while segment k runs on `stream`.  The output copies start after
 * everything already enqueued on `stream`, and `stream` waits for the last
 * one.  The input copies of a handle made by ttt_mlp_create (which owns its
 * scratch) go to one of two staging buffers that alternate between calls, so
 * they may start while the handle's previous call still runs: they wait only
 * for the layers of the call before that, which read the same buffer.  A
 * handle made by ttt_mlp_create_split (whose scratch may be shared) starts
 * them after everything already enqueued on `stream`.  Either way x_host is
 * read asynchronously and the results are as if everything ran on `stream`.
 * Pinned (page-locked) host buffers make the copies asynchronous and let
 * them overlap; the call returns once everything is enqueued, so the caller
 * must synchronise `stream` before reading o_host or reusing x_host.  If the
 * call fails after its first segment was enqueued, copies of earlier segments
 * may still be in flight on the copy streams: synchronise the device before
 * freeing or reusing the host buffers. */
ttt_status ttt_mlp_forward_chunks_host(ttt_mlp* h, int32_t doc, const void* x_host,
                                       const void* x0_host, int64_t n_tokens,
                                       const int64_t* doc_starts, int32_t n_doc_starts,
                                       void* o_host, void* stream);

/* Reset slot `doc` (or every slot when doc == -1) to W <- W_0 (document
 * boundary, appendix B of the summary page). */
ttt_status ttt_mlp_reset(ttt_mlp* h, int32_t doc, void* stream);

/* Copy slot `doc`'s fp32 fast weight (d x f) to / from a device buffer.  Every
 * fp32 bit pattern goes through unchanged. */
ttt_status ttt_mlp_get_fast_weight(ttt_mlp* h, int32_t doc, float* dst, void* stream);
ttt_status ttt_mlp_set_fast_weight(ttt_mlp* h, int32_t doc, const float* src, void* stream);

/* Synchronise `stream` and read the workspace's error word: TTT_OK, or
 * TTT_ETIMEOUT if an in-kernel wait ran out since the last check (the word is
 * cleared), or TTT_ECUDA on an asynchronous CUDA error. */
ttt_status ttt_mlp_check(ttt_mlp* h, void* stream);

/* Free the handle (host memory only; device memory stays the caller's). */
ttt_status ttt_mlp_destroy(ttt_mlp* h);

/* Text of the last failure on this handle ("" if none); with h == NULL, of
 * the last failure of a call that had no handle.  Valid until the next call. */
const char* ttt_mlp_last_error(const ttt_mlp* h);

/* Device pointers, inside the workspace, of the last forward call's Z
 * (n x f) and eta-scaled target V (n x d, i.e. eta * U W_target, times each
 * chunk's clip scale when clipping is on), and their
 * element type (*dtype: TTT_BF16 on the tcgen05 path, TTT_F32 on the SIMT
 * path).  For inspection and tests; valid until the next forward call. */
ttt_status ttt_mlp_intermediates(const ttt_mlp* h, const void** z, const void** v,
                                 int32_t* dtype);

/* Phase timing for benchmarks.  While enabled, every forward call records
 * CUDA events on its stream at the boundaries of its phases (no extra
 * synchronisation).  ttt_mlp_profile_read synchronises those events and
 * returns, summed over the calls since profiling was (re-)enabled,
 * ms[0] Conv1D target source, ms[1] SwiGLU producer, ms[2] target projection,
 * ms[3] intra-group Gram blocks, ms[4] fused apply+update group kernels
 * (ms must hold 5 floats), and counts[0] forward calls, counts[1] group
 * kernel launches, counts[2] all kernel launches of the library (counts must
 * hold 3 int64).  Enabling clears what was recorded. */
ttt_status ttt_mlp_profile_enable(ttt_mlp* h, int32_t enable);
ttt_status ttt_mlp_profile_read(ttt_mlp* h, float* ms, int64_t* counts);

/* Which kernel family runs a forward call of this handle: "tcgen05" (bf16
 * tensor-core path) or "simt" (fp32 FFMA path).  Host only. */
const char* ttt_mlp_path(const ttt_mlp* h);

/* ---- allocation-free target computation ----
 *
 * The paper has no counterpart to this call; it exists for callers that may
 * not allocate device memory at all (for example code that runs inside
 * another runtime's memory pool or an allocator-free embedded host, where
 * cudaMalloc is forbidden or unavailable) and so cannot provide the
 * workspace the handle-based calls need.
 *
 * It computes the same target as a forward call with the default window
 * (TTT_TARGET_NEXT) and no clipping, V = eta * Conv1D(X0) W_target
 * (chunk-local, causal-shifted depthwise Conv1D; chunking restarts at each
 * document start), into the caller's v, with the bf16 tensor-core kernels.
 * Its scratch (the Conv1D output, the transposed W_target, a tile counter and
 * an error word) lives in one file-scope device array of
 * TTT_NOALLOC_SCRATCH_BYTES bytes that every GPU which loads the library
 * holds until the process exits; the call allocates nothing.
 *
 * x0: n_tokens x d bf16; conv_w: conv_k x d bf16; w_target: d x d bf16
 * (in x out); v: n_tokens x d bf16 output; all device, 16-byte aligned.
 * d must be a multiple of 64 and >= 256; 1 <= chunk <= 1024; 1 <= conv_k <= 8;
 * doc_starts as in ttt_mlp_forward_chunks.  A call whose scratch need,
 * 2*d*d + 2*n_tokens*d bytes plus 512, exceeds TTT_NOALLOC_SCRATCH_BYTES
 * returns TTT_EUNSUPPORTED before anything is enqueued.
 *
 * The first call on a device sets up that device (it looks up the scratch
 * array's device address and configures the kernel); make that first call
 * before any CUDA stream capture.  Every call on a device shares the one
 * array and the call clears what must start at zero, so calls whose kernels
 * overlap on the GPU (different streams, or different host threads) race and
 * must be serialised by the caller.  status: optional device int32 that
 * receives 0, or the code of an in-kernel wait that ran out (the output is
 * then incomplete).  With status == NULL such a timeout is recorded only in
 * the shared array, which the next call clears, so it cannot be detected:
 * callers that need to know whether v is complete must pass status. */
#define TTT_NOALLOC_SCRATCH_BYTES (32u << 20)
ttt_status ttt_target_noalloc(const void* x0, const void* conv_w, const void* w_target,
                              int64_t n_tokens, int32_t d, int32_t conv_k, int32_t chunk,
                              const int64_t* doc_starts, int32_t n_doc_starts, float eta,
                              void* v, int32_t* status, void* stream);

/* ---- residual-stack glue (pre-norm blocks h <- h + MLP_TTT(RMSNorm(h))) ---- */

/* x[t] = RMSNorm(h[t]) = h[t] / sqrt(mean(h[t]^2) + eps), unit gain, cast to
 * out_dtype.  h: n x d fp32; x: n x d.  Returns TTT_EINVAL on bad sizes. */
ttt_status ttt_rmsnorm(const float* h, void* x, int64_t n, int32_t d, float eps,
                       int32_t out_dtype, void* stream);

/* h += o elementwise; h: n x d fp32, o: n x d of o_dtype. */
ttt_status ttt_residual_add(float* h, const void* o, int64_t n, int32_t d, int32_t o_dtype,
                            void* stream);

/* The two in one pass over h: h += o, then x = RMSNorm(h) (the next block's
 * input).  The same results as ttt_residual_add followed by ttt_rmsnorm.
 * h: n x d fp32; o: n x d of o_dtype; x: n x d of x_dtype. */
ttt_status ttt_residual_rmsnorm(float* h, const void* o, void* x, int64_t n, int32_t d, float eps,
                                int32_t o_dtype, int32_t x_dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TTT_MLP_H */
