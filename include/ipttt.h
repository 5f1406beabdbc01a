/*
 * libipttt -- the fast-weight hot path of In-Place Test-Time Training, for
 * NVIDIA B300 (sm_103a).
 *
 * The method (In-Place TTT write-ups: itsolotime §2.1-2.3 and Fig. 1;
 * su666666 "first/second/third axe") reuses the final projection W_o of a
 * gated MLP as a fast weight.  Per layer and per sequence of L tokens:
 *
 *   Z = SiLU(X W_g) * (X W_u)                  gated activation, W_g W_u frozen
 *   V = Proj(Conv(E))                          target from token embeddings E
 *   for each chunk k of B tokens (K = L/B):
 *       O_k     = Z_k W_k                      apply the current fast weight
 *       W_{k+1} = W_k - (eta/B) Z_k^T (Z_k W_k - V_k)     MSE rule, or
 *       W_{k+1} = W_k + (eta/B) Z_k^T V_k                 additive rule
 *
 * Conv is depthwise, width 4, tap j multiplies E[t+j], no bias, and reads
 * zeros past the end of the token's own chunk (no update reads past its
 * chunk).  Row-vector convention: x is 1 x d, W_g and W_u are d x d_ff, W_o is
 * d_ff x d.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array pointer is a DEVICE pointer owned by the caller, row-major and
 *   contiguous, aligned to 16 bytes.  Token-major activations hold sequence s
 *   in rows s*L .. s*L+L-1.  Nothing passed in is freed or kept.
 * - "act" arrays (X, E, W_g, W_u, P, Z, V, O) have the element type given by
 *   dims->dtype: IPTTT_BF16 (bfloat16) or IPTTT_FP32 (float).  The fast weight
 *   (W_o0, W_final) and the conv weights are always float32.
 * - IPTTT_BF16 computes on the tensor cores (bf16 operands, fp32 accumulation,
 *   fp32 master fast weight).  IPTTT_FP32 computes every product in fp32 on
 *   the CUDA cores; it is the exact-arithmetic mode.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream) and never synchronise it.  A call returns IPTTT_OK once its
 *   kernels are queued; a device-side failure (a capped wait that ran out) is
 *   recorded on the device and reported by ipttt_sync_status().
 * - Scratch memory (activations Z and V inside the layer calls, partial sums,
 *   the split planes of the fast weight, group states of the additive scan,
 *   the [Z | S] and [W_0 ; V] blocks of the block-causal form, the tables of
 *   packed documents) comes from a per-device pool owned by the library: grown
 *   with cudaMalloc on first need (a call that needs to grow it synchronises
 *   the device), reused by later calls, freed by ipttt_release().  Calls that
 *   share the pool must be ordered (one stream, or the caller's own events).
 *   So must calls that run the gated up-projection (ipttt_gate_up and the
 *   layer calls): its tiles are handed out by one counter per device.
 *   ipttt_workspace_size reports the need of ipttt_layer_forward and
 *   ipttt_chunk_forward; the packed-document and multi-layer calls need the
 *   same per document or per layer and sequence.
 * - No call aborts, throws or traps.  Errors come back as an ipttt_status.
 *   Arguments are checked before any launch: null pointers, non-positive or
 *   inconsistent sizes, L not a multiple of B, misaligned pointers, host
 *   pointers where device pointers are required, a device that is not
 *   compute capability 10.3.
 * - Constraints of the IPTTT_BF16 mode: d and d_ff multiples of 8 (16-byte row
 *   strides for the tensor-memory-accelerator copies) and B a multiple of 16
 *   (the tensor-core K step over tokens).  IPTTT_FP32 takes any sizes >= 1.
 */
#ifndef IPTTT_H
#define IPTTT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IPTTT_VERSION 100 /* 0.1.0 */

typedef enum ipttt_status {
  IPTTT_OK = 0,
  IPTTT_ERR_INVALID_ARG = 1, /* null/misaligned/host pointer, bad size, L % B != 0, ... */
  IPTTT_ERR_UNSUPPORTED = 2, /* no CUDA device, or not compute capability 10.3 */
  IPTTT_ERR_ALLOC = 3,       /* the scratch pool could not grow */
  IPTTT_ERR_LAUNCH = 4,      /* a kernel launch was rejected */
  IPTTT_ERR_TIMEOUT = 5,     /* a capped device-side wait ran out (from ipttt_sync_status) */
  IPTTT_ERR_CUDA = 6         /* another CUDA runtime error (sticky context errors included) */
} ipttt_status;

typedef enum ipttt_dtype { IPTTT_FP32 = 0, IPTTT_BF16 = 1 } ipttt_dtype;

typedef enum ipttt_rule {
  IPTTT_RULE_MSE = 0, /* W <- W - (eta/B) Z_k^T (Z_k W - V_k): sequential over chunks */
  IPTTT_RULE_ADD = 1, /* W <- W + (eta/B) Z_k^T V_k: chunk-parallel prefix scan */
  /* The additive rule's outputs from its block-causal quadratic form, without a
   * fast weight per chunk: O = Z W_0 + (eta/B) mask(Z Z^T) V with mask keeping
   * the tokens of earlier chunks, and W_final = W_0 + (eta/B) Z^T V (itsolotime
   * §2.3: the additive rule is associative; §3.2: parallel equals serial).  The
   * same results as IPTTT_RULE_ADD; work and scratch grow as L^2 per sequence
   * (batch*L*(d_ff+L) act elements of scratch), so it pays at small B, where
   * the scan streams a fast weight per chunk.  Packed documents
   * (ipttt_layer_forward_varlen) run it as IPTTT_RULE_ADD. */
  IPTTT_RULE_ADD_BLOCKCAUSAL = 2
} ipttt_rule;

/* Sizes shared by the calls.  batch = independent sequences; d = model width;
 * d_ff = gated-MLP hidden width; dtype = ipttt_dtype of the "act" arrays;
 * w0_per_seq = 0: W_o0 is one d_ff x d matrix shared by all sequences,
 *              1: W_o0 is batch x d_ff x d (for example the W_final of a
 *                 previous call, to resume a sequence where it stopped). */
typedef struct ipttt_dims {
  int64_t batch;
  int64_t d;
  int64_t d_ff;
  int32_t dtype;
  int32_t w0_per_seq;
} ipttt_dims;

typedef void* ipttt_stream; /* a cudaStream_t */

/*
 * Whole layer: gated activation, targets and the chunk loop, for dims->batch
 * sequences of L tokens.  (In-Place TTT: gated MLP itsolotime §2.1, target
 * §2.3, chunk-wise apply-then-update §2.2 / Fig. 1.)
 *
 *   X      [batch*L, d]      act   hidden states entering the MLP
 *   E      [batch*L, d]      act   token embeddings of the same tokens
 *   W_g    [d, d_ff]         act   frozen gate projection
 *   W_u    [d, d_ff]         act   frozen up projection
 *   W_o0   [d_ff, d] fp32          initial fast weight (or [batch, d_ff, d] if
 *                                  dims->w0_per_seq); not modified
 *   conv_w [d, 4] fp32             depthwise conv taps, conv_w[c][j] for E[t+j][c]
 *   P      [d, d]            act   target projection
 *   L, B                           tokens per sequence, tokens per chunk; L % B == 0
 *   eta                            step size (the step is eta/B times the chunk sum)
 *   rule                           IPTTT_RULE_MSE, IPTTT_RULE_ADD or IPTTT_RULE_ADD_BLOCKCAUSAL
 *   O      [batch*L, d]      act   out: O_k = Z_k W_k, chunk by chunk
 *   W_final[batch, d_ff, d] fp32   out: the fast weight after the last chunk
 *
 * O and W_final must not overlap any input.  L == 0 copies W_o0 to W_final.
 *
 * In bf16 mode the MSE rule takes chunks below 1024 tokens a window of m = W/B
 * chunks at a time when d, d_ff are multiples of 256, a window W (1024, 768,
 * 512 or 256 tokens) holds m >= 2 chunks and divides L, and d (m - 1) >= 2 W:
 * within a window the m steps unroll to one triangular solve for the
 * residuals, so the fast weight is read and written once per window.  O and
 * W_final are those of the m chunk steps, up to rounding.
 */
ipttt_status ipttt_layer_forward(const void* X, const void* E, const void* W_g, const void* W_u,
                                 const float* W_o0, const float* conv_w, const void* P, int64_t L,
                                 int64_t B, float eta, ipttt_rule rule, void* O, float* W_final,
                                 const ipttt_dims* dims, ipttt_stream stream);

/*
 * Whole layer over packed documents of different lengths, the fast weight
 * reset to W_o0 at every document boundary (In-Place TTT, itsolotime §3.2,
 * "boundary reset": no document sees another's updates).
 *
 *   cu_seqlens [n_docs+1] int64, HOST array: document i holds rows
 *                  cu_seqlens[i] .. cu_seqlens[i+1]-1; cu_seqlens[0] == 0 and
 *                  the values rise strictly (every document has a token).
 *                  Read during the call only.
 *   X, E   [T, d]            act   T = cu_seqlens[n_docs], documents back to back
 *   W_g, W_u, conv_w, P            as in ipttt_layer_forward
 *   W_o0   [d_ff, d] fp32          shared initial fast weight, or [n_docs, d_ff, d]
 *                                  if dims->w0_per_seq (document order)
 *   B                              tokens per chunk (a multiple of 16 in bf16 mode)
 *   O      [T, d]            act   out: O_k = Z_k W_k, chunk by chunk per document
 *   W_final[n_docs, d_ff, d] fp32  out: each document's fast weight after its last chunk
 *
 * dims->batch is ignored.  Chunks are counted from each document's first
 * token; a document's last chunk holds the n <= B tokens left, its step is
 * normalised by n (the chunk mean, as for full chunks), and the conv reads
 * zeros past the document's end as past any chunk's end.  Both rules run
 * chunk by chunk here.  Errors: IPTTT_ERR_INVALID_ARG for a bad cu_seqlens, B
 * or pointer (nothing is queued), else as ipttt_layer_forward.
 */
ipttt_status ipttt_layer_forward_varlen(const void* X, const void* E, const void* W_g, const void* W_u,
                                        const float* W_o0, const float* conv_w, const void* P,
                                        const int64_t* cu_seqlens, int64_t n_docs, int64_t B, float eta,
                                        ipttt_rule rule, void* O, float* W_final,
                                        const ipttt_dims* dims, ipttt_stream stream);

/*
 * Several layers' fast-weight MLPs over the same tokens in one call: every
 * step is one launch for all layers (the gate and projection GEMMs batched over
 * the layers, one conv launch, and the chunk loop over all layers and sequences:
 * in bf16 mode with d, d_ff and B multiples of 256 one persistent kernel for
 * the whole MSE loop, else each chunk's apply / residual / update).  Layer l takes its own hidden states and weights;
 * every layer's target is built from the same token embeddings E (the In-Place
 * TTT layer is the MLP block of each layer it is put in, itsolotime §2.1; its
 * target reads the token embeddings, §2.3).  Layers do not interact.
 *
 *   X      [n_layers, batch*L, d]     act   hidden states entering each layer's MLP
 *   E      [batch*L, d]               act   token embeddings, shared by the layers
 *   W_g    [n_layers, d, d_ff]        act   per-layer gate projections
 *   W_u    [n_layers, d, d_ff]        act   per-layer up projections
 *   W_o0   [n_layers, d_ff, d] fp32         per-layer initial fast weight, or
 *                                           [n_layers, batch, d_ff, d] if dims->w0_per_seq
 *   conv_w [n_layers, d, 4] fp32            per-layer conv taps
 *   P      [n_layers, d, d]           act   per-layer target projections
 *   O      [n_layers, batch*L, d]     act   out
 *   W_final[n_layers, batch, d_ff, d] fp32  out (also the scratch that holds each
 *                                           sequence's start when W_o0 is per layer)
 *
 * L, B, eta, rule and errors as in ipttt_layer_forward; n_layers == 0 does
 * nothing.  W_o0 must not overlap W_final.
 */
ipttt_status ipttt_layers_forward(const void* X, const void* E, const void* W_g, const void* W_u,
                                  const float* W_o0, const float* conv_w, const void* P, int64_t n_layers,
                                  int64_t L, int64_t B, float eta, ipttt_rule rule, void* O, float* W_final,
                                  const ipttt_dims* dims, ipttt_stream stream);

/*
 * Targets only: V = Proj(Conv(E)) with the conv zero-padded at every chunk's
 * end (itsolotime §2.3; the next-token case is conv one-hot at tap 1, P = I).
 *
 *   E [batch*L, d] act, conv_w [d, 4] fp32, P [d, d] act, V [batch*L, d] act (out).
 */
ipttt_status ipttt_make_targets(const void* E, const float* conv_w, const void* P, void* V,
                                int64_t L, int64_t B, const ipttt_dims* dims, ipttt_stream stream);

/*
 * Gated activation only: Z = SiLU(X W_g) * (X W_u) (itsolotime §2.1), for
 * n_tokens rows.  X [n_tokens, d] act, W_g W_u [d, d_ff] act, Z [n_tokens, d_ff]
 * act (out).  dims->batch is ignored.
 */
ipttt_status ipttt_gate_up(const void* X, const void* W_g, const void* W_u, void* Z,
                           int64_t n_tokens, const ipttt_dims* dims, ipttt_stream stream);

/*
 * Chunk engine only, on precomputed Z [batch*L, d_ff] act and V [batch*L, d]
 * act: the apply / residual / update loop (MSE rule) or the chunk-parallel
 * prefix scan (additive rule) of itsolotime §2.2 and §2.3.  Other arguments as
 * in ipttt_layer_forward.
 */
ipttt_status ipttt_chunk_forward(const void* Z, const void* V, const float* W_o0, int64_t L,
                                 int64_t B, float eta, ipttt_rule rule, void* O, float* W_final,
                                 const ipttt_dims* dims, ipttt_stream stream);

/*
 * Targets without any allocation: the same result as ipttt_make_targets (same
 * kernels), but the conv output it needs as scratch lives in a fixed array
 * inside this library rather than in the pool that ipttt_make_targets grows
 * with cudaMalloc.  The pages have no counterpart of this call; it is for
 * callers that cannot allocate device memory at this point -- a process whose
 * GPU memory is already handed out by another allocator (where a new
 * cudaMalloc can fail or break that allocator's bookkeeping), or a service
 * that cannot pay for cudaMalloc / cudaFree, which may synchronise the device.
 *
 * - Limit: batch*L*d elements of the act type must fit in
 *   IPTTT_NOALLOC_SCRATCH_BYTES (16 MiB, e.g. 3276 tokens at d = 2560 in
 *   bf16); larger calls return IPTTT_ERR_INVALID_ARG and do nothing.  Split
 *   the tokens into chunk-aligned pieces (the conv never reads past a chunk).
 * - The array takes IPTTT_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 *   library, until the process exits.
 * - Every call looks the array's device address up for the current device
 *   and CUDA context (cudaGetSymbolAddress), so a device reset or another
 *   device never sees a stale address.  The first call on a device also loads
 *   the library's kernels there: make that first call before any stream
 *   capture.
 * - Every call shares the array: calls that overlap on the GPU (unordered
 *   streams) race on it.  Nothing in it needs clearing between calls.
 * - Arguments, layouts and errors otherwise as ipttt_make_targets; no
 *   cudaMalloc, cudaFree or other allocating call is made.
 */
#define IPTTT_NOALLOC_SCRATCH_BYTES (16u << 20)
ipttt_status ipttt_make_targets_noalloc(const void* E, const float* conv_w, const void* P, void* V,
                                        int64_t L, int64_t B, const ipttt_dims* dims,
                                        ipttt_stream stream);

/*
 * Pieces of the additive rule over one sequence split across GPUs (context
 * parallelism: each rank holds a run of whole chunks).  The rule's weight after
 * a run of chunks is the weight before it plus (eta/B) times the run's sum of
 * Z_k^T V_k (itsolotime §2.3: the additive rule is associative), so a rank
 * starts from W_0 plus the sums of the ranks before it and then runs its chunks
 * with ipttt_chunk_forward (rule IPTTT_RULE_ADD, per-sequence W_o0).
 *
 * ipttt_additive_sums: S[s] = Z_s^T V_s over the L tokens of each sequence s.
 *   Z [batch*L, d_ff] act, V [batch*L, d] act, S [batch, d_ff, d] fp32 (out).
 *   In IPTTT_BF16 mode L must be a multiple of 16.  L == 0 writes zeros.
 * ipttt_weight_axpy: W[i] += alpha * S[i] for i < n, fp32 device arrays.
 */
ipttt_status ipttt_additive_sums(const void* Z, const void* V, int64_t L, float* S, const ipttt_dims* dims,
                                 ipttt_stream stream);
ipttt_status ipttt_weight_axpy(float* W, const float* S, float alpha, int64_t n, ipttt_stream stream);

/* Bytes of pool scratch ipttt_layer_forward (with_activations = 1) or
 * ipttt_chunk_forward (with_activations = 0) needs for these sizes.  Host only. */
ipttt_status ipttt_workspace_size(const ipttt_dims* dims, int64_t L, int64_t B, ipttt_rule rule,
                                  int32_t with_activations, size_t* bytes);

/* Synchronise `stream`, then read and clear the device error word of the
 * current device: IPTTT_ERR_TIMEOUT if a capped wait ran out since the last
 * check, IPTTT_ERR_CUDA for a CUDA error, else IPTTT_OK. */
ipttt_status ipttt_sync_status(ipttt_stream stream);

/* Soft limit, in nanoseconds, of the pipeline waits inside the tensor-core
 * kernels on the current device (0 restores the default, the 2 s hard limit;
 * larger values are clamped to it).  No counterpart on the pages: it is the
 * failure-detection hook of the library.  A wait that lasts longer records
 * IPTTT_ERR_TIMEOUT for ipttt_sync_status(); its CTA then issues no more
 * tensor-core work and writes no more results, but keeps every handshake of
 * its pipeline until the copies and MMAs already in flight have completed, so
 * that the kernel still ends cleanly and the context stays usable.  The
 * outputs of such a call are unspecified.  Only a wait that reaches the hard
 * limit gives up outright.  Set it below the length of a real wait (a few
 * hundred ns) to make the detection fire on purpose; every later call on the
 * device uses the new value until it is restored.  Synchronous; do not call
 * it while kernels of the library run on the device.
 * Errors: IPTTT_ERR_UNSUPPORTED (no compute capability 10.3 device),
 * IPTTT_ERR_CUDA. */
ipttt_status ipttt_set_wait_limit(uint64_t ns);

/* Free the scratch pool of every device the library has used.  The caller
 * must make sure no queued call still uses it (synchronise first). */
ipttt_status ipttt_release(void);

/* Cap the scratch one call may take from the pool (bytes; 0 = no cap, the
 * default): a call that needs more returns IPTTT_ERR_ALLOC before queuing
 * anything.  For processes that share the GPU with another allocator.  It does
 * not shrink a pool grown before; ipttt_release() does.  Host only. */
ipttt_status ipttt_set_pool_limit(size_t bytes);

/* Kernels queued by the last call made from this host thread (a count of this
 * library's launches, for profiling).  Host only. */
int64_t ipttt_last_launch_count(void);

/* Per-kernel timing, a profiling aid that is off by default.  While enabled,
 * every kernel this library launches is bracketed by two CUDA events on its
 * stream (no synchronisation is added).  ipttt_kernel_timing(1) clears the
 * totals and starts recording, (0) stops.  ipttt_kernel_timing_read waits
 * for the recorded events and returns, for one kernel kind, the launches and
 * their summed device time in milliseconds since the last start.  Kinds:
 * 0 gate_up, 1 conv, 2 proj, 3 apply, 4 residual, 5 update, 6 group_sum,
 * 7 scan, 8 weight_copy, 9 scores, 10 engine, 11 window (names from
 * ipttt_kernel_name).  Host only. */
ipttt_status ipttt_kernel_timing(int32_t enable);
ipttt_status ipttt_kernel_timing_read(int32_t kind, int64_t* launches, double* total_ms);
const char* ipttt_kernel_name(int32_t kind);

const char* ipttt_status_string(ipttt_status status);
int ipttt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IPTTT_H */
