/*
 * gdn.h -- C ABI of libgdn, the GB300 (sm_103a) gated delta rule library.
 *
 * The gated delta rule, per (sequence, value head h) with a K x V fp32 state S:
 *
 *     S   <- exp(g_t) * S
 *     S   <- S + k_t * (beta_t * (v_t - S^T k_t))^T
 *     o_t  = scale * S^T q_t
 *
 * q_t, k_t optionally L2-normalised in-kernel (x / sqrt(sum x^2 + 1e-6)), value
 * head h reading query/key head h / (Hv / Hqk).  Sources: the GDN mixer and its
 * torch-native chunked rule on "Megatron-Core API: core.ssm.gated_delta_net.gdn"
 * (GatedDeltaNet, GatedDeltaNet._compute_gates "per-head log-decay g and the
 * write strength beta", torch_chunk_gated_delta_rule); the inference contract on
 * "Megatron-Core API: core.ssm.gated_delta_product" (GatedDeltaProductMixer.
 * ssm_decode, ssm_prefill, ssm_inference_chunk_size); and the -1 padding rule on
 * "Add GDN dynamic inference" (Megatron-LM pull request 6499, review thread).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument named as device memory must be device memory
 *     allocated by the caller; the library allocates, frees and synchronises
 *     nothing.  All work is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and the call returns before it finishes, so the
 *     calls can be captured in a CUDA graph (ssm_decode and ssm_prefill on the
 *     gated_delta_product page require graph-safe steps: no host sync, no
 *     data-dependent shapes, device-side indices).
 *   - Argument errors are detected on the host before anything is launched and
 *     returned as a gdn_status_t; nothing is enqueued then.  A failed launch
 *     returns GDN_ERR_CUDA.
 *   - Bad data that only the device can see (a slot outside [-1, num_slots), a
 *     non-monotone cu_seqlens) is skipped by the kernels, never trapped on, and
 *     reported by OR-ing GDN_DEV_* bits into *dev_status when dev_status is a
 *     non-NULL device int.
 *   - Dense tensors are contiguous, row-major, in the layouts given per
 *     argument; q, k, v and o must start on 16-byte boundaries (g and beta on their element size).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_NULL = 1,        /* a required pointer is NULL                         */
  GDN_ERR_SHAPE = 2,       /* a size is out of range or sizes disagree           */
  GDN_ERR_DTYPE = 3,       /* unknown dtype code                                 */
  GDN_ERR_LAYOUT = 4,      /* a pointer is not aligned as required               */
  GDN_ERR_UNSUPPORTED = 5, /* well-formed but not provided (e.g. chunk_size 32)  */
  GDN_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed        */
  GDN_ERR_WORKSPACE = 7    /* workspace missing or smaller than required         */
} gdn_status_t;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define GDN_DEV_BAD_SLOT 1        /* a slot index >= num_slots or < -1 was skipped */
#define GDN_DEV_BAD_CU_SEQLENS 2  /* cu_seqlens not monotone / out of [0, T]       */
#define GDN_DEV_TIMEOUT 4         /* a bounded in-kernel wait gave up (unit skipped) */

/* Largest head dimensions the library accepts (K, V). */
#define GDN_MAX_HEAD_DIM 128

/*
 * gdn_chunk_fwd -- chunkwise forward (training / prefill) of the gated delta rule.
 *
 * Arguments follow torch_chunk_gated_delta_rule (q, k, v, g, beta, scale,
 * chunk_size, initial_state, output_final_state, use_qk_l2norm_in_kernel,
 * cu_seqlens) on "Megatron-Core API: core.ssm.gated_delta_net.gdn"; the packed
 * layout with cu_seqlens follows GatedDeltaProductMixer._run_gdp_kernel and
 * ssm_prefill on "Megatron-Core API: core.ssm.gated_delta_product".
 *
 *   q, k        [B, T, Hqk, K] io_dtype, device.
 *   v           [B, T, Hv, V] io_dtype, device.          Hv % Hqk == 0.
 *   g           [B, T, Hv] fp32 log-decay, device; every value finite.
 *   beta        [B, T, Hv] beta_dtype, device.
 *   B, T        batch and tokens per batch row.  With cu_seqlens, B must be 1 and
 *               T is the packed token count.
 *   K, V        head dims, 1..GDN_MAX_HEAD_DIM (K * sizeof(io_dtype) and
 *               V * sizeof(io_dtype) multiples of 16 bytes).
 *   io_dtype    GDN_F32 or GDN_BF16 (q, k, v, o); beta_dtype GDN_F32 or io_dtype.
 *   scale       read-out scale; NaN selects the default 1/sqrt(K) (the page's
 *               "scale defaults to 1 / sqrt(K)").
 *   chunk_size  must be 64 (the inference kernels "chunk at a fixed 64",
 *               ssm_inference_chunk_size); anything else: GDN_ERR_UNSUPPORTED.
 *   initial_state  fp32, device, or NULL (zero state).  Without state_indices:
 *               [N, Hv, K, V], N = B or num_seqs.  With state_indices: a slot
 *               cache [num_slots, Hv, K, V].
 *   output_final_state, final_state  when the flag is set, final_state (fp32,
 *               device, same shape rule as initial_state) receives the state
 *               after the last token; it may be the same pointer as
 *               initial_state (in-place slot update).
 *   use_qk_l2norm  L2-normalise q and k inside the kernels.
 *   cu_seqlens  [num_seqs + 1] int32, device, or NULL: sequence n is the packed
 *               tokens [cu_seqlens[n], cu_seqlens[n+1]); chunks restart at every
 *               sequence start; empty sequences are allowed and leave their
 *               state unchanged.
 *   state_indices  [N] int32, device, or NULL.  Sequence n reads its initial
 *               state from slot state_indices[n] and writes its final state back
 *               to that slot ("each request enters carrying whatever state its
 *               cache slot holds and leaves having written the slot back",
 *               ssm_prefill).  Slot -1 is padding: the sequence's output rows are
 *               zero and no state is read or written.  Slots must be distinct.
 *   num_slots   slots in the cache when state_indices is given.
 *   o           [B, T, Hv, V] io_dtype, device, written completely.
 *   workspace, workspace_bytes  device scratch of at least
 *               gdn_chunk_fwd_workspace_size(...) bytes, 256-byte aligned for the
 *               tensor-core path.  Not read before it is written; may be reused
 *               once the call's work on `stream` has finished.  The tensor-core
 *               path also runs without it (NULL or smaller than that size): it
 *               then skips its launch plan -- longest sequences first, and, when
 *               the batch has fewer than a third as many (sequence, head) chains
 *               as the GPU has SMs, every sequence of at least 2 s chunks split
 *               into s segments that run concurrently and are joined exactly
 *               through the linearity of the chunk map (a per-segment transition
 *               and contribution, a scan, and a second pass from each segment's
 *               entry state).  The plan is built on the device from cu_seqlens,
 *               so a captured graph replays it for any lengths.
 *   dev_status  NULL or a device int receiving GDN_DEV_* bits.
 *   stream      cudaStream_t.
 */
gdn_status_t gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                           const void* beta, int B, int T, int Hqk, int Hv, int K, int V,
                           gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                           int chunk_size, const float* initial_state, int output_final_state,
                           float* final_state, int use_qk_l2norm, const int32_t* cu_seqlens,
                           int num_seqs, const int32_t* state_indices, int num_slots, void* o,
                           void* workspace, size_t workspace_bytes, int* dev_status,
                           void* stream);

/*
 * Device scratch (bytes) gdn_chunk_fwd needs for these sizes: the CUDA-core
 * path's scratch, or the tensor-core path's launch plan (unit tables and, when
 * sequences split, 64 KB per segment matrix), sized for the SM count of the
 * current device.  num_seqs is N (B when cu_seqlens is NULL).  Returns
 * (size_t)-1 for sizes gdn_chunk_fwd would reject.
 */
size_t gdn_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int K, int V, int num_seqs,
                                    gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype);

/*
 * Which kernel family gdn_chunk_fwd uses for these sizes: 1 = the fused
 * tcgen05 / TMEM / TMA kernel (bf16, K = V = 128), 0 = the fp32 CUDA-core
 * chunk kernels (every other accepted case), -1 = rejected.
 */
int gdn_chunk_fwd_path(int K, int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype);

/*
 * gdn_decode -- one token per request on a slot-indexed state cache, in place.
 *
 * Follows GatedDeltaNet.ssm_decode ("one CUDA-graph-compatible GDN decode token
 * per request", "Megatron-Core API: core.ssm.gated_delta_net.gdn") and
 * GatedDeltaProductMixer.ssm_decode ("Megatron-Core API:
 * core.ssm.gated_delta_product": states read and written in place at the slots
 * named by batch_indices, -1 marks padding whose output is zeroed,
 * batch_indices=None means the cache is already in request order).  Padding
 * slots are skipped inside the kernel rather than clamped to slot 0 ("Add GDN
 * dynamic inference" review thread: writes ignore -1; the Mamba2-style in-kernel
 * skip writes zeros).
 *
 *   q, k        [n, Hqk, K] io_dtype, device.
 *   v           [n, Hv, V] io_dtype, device.
 *   g           [n, Hv] fp32, device.      beta [n, Hv] beta_dtype, device.
 *   ssm_state   [num_slots, Hv, K, V] fp32, device, updated in place.
 *   batch_indices  [n] int32, device, or NULL (request i uses slot i; then
 *               n <= num_slots).  -1: output row zero, state untouched.  Slots
 *               outside [-1, num_slots): skipped like -1 and reported through
 *               GDN_DEV_BAD_SLOT.  Non-negative slots must be distinct.
 *   scale       NaN selects 1/sqrt(K).    use_qk_l2norm: normalise q, k.
 *   o           [n, Hv, V] io_dtype, device.
 *   dev_status, stream  as above.
 * Slot selection, padding and untouched slots are exact: a padding row is +0.0
 * and a slot not named in batch_indices is never accessed.
 */
gdn_status_t gdn_decode(const void* q, const void* k, const void* v, const float* g,
                        const void* beta, float* ssm_state, int num_slots,
                        const int32_t* batch_indices, int n, int Hqk, int Hv, int K, int V,
                        gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                        int use_qk_l2norm, void* o, int* dev_status, void* stream);

/*
 * gdn_decode_multi -- L tokens per request on the slot-indexed cache (multi-token
 * decode, e.g. verifying speculative tokens), with optional per-token states.
 *
 * GatedDeltaProductMixer.ssm_decode ("Megatron-Core API:
 * core.ssm.gated_delta_product") takes [n, seq_len, ...] inputs per request and
 * optional intermediate_ssm_state / intermediate_conv_state outputs; the GDN mixer's
 * ssm_decode has the same arguments ("Megatron-Core API: core.ssm.gated_delta_net.gdn").
 * Request i applies its tokens t = 0..L-1 in order to slot batch_indices[i]:
 *   q, k        [n, L, Hqk, K];  v, o [n, L, Hv, V];  g, beta [n, L, Hv]  (token-major per request)
 *   intermediate_states  NULL, or [n, L, Hv, K, V] fp32 receiving the state after
 *               every token (the last one equals the slot's new state).
 * The slot receives the state after token L - 1.  Padding (-1) and invalid slots:
 * all L output rows zero, no state read or written, intermediate rows untouched.
 * Every other rule as gdn_decode (which is this call with L = 1 and no intermediates).
 */
gdn_status_t gdn_decode_multi(const void* q, const void* k, const void* v, const float* g,
                              const void* beta, float* ssm_state, int num_slots,
                              const int32_t* batch_indices, int n, int L, int Hqk, int Hv, int K,
                              int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                              int use_qk_l2norm, void* o, float* intermediate_states,
                              int* dev_status, void* stream);

/*
 * Fused gates.  The GDN mixer computes "the per-head log-decay g and the write
 * strength beta" from its gate features and the per-head parameters A_log and
 * dt_bias ("Megatron-Core API: core.ssm.gated_delta_net.gdn",
 * GatedDeltaNet._compute_gates; "_prepare_inference_inputs ... leaving
 * normalization and gates fused in-kernel").  These two entry points take the
 * raw features instead of g and beta and evaluate, inside the kernels,
 *
 *     g = -exp(A_log[h]) * softplus(a + dt_bias[h]),     beta = sigmoid(b),
 *
 * so g and beta never exist in device memory.
 *   a, b        [B, T, Hv] (chunk) or [n, Hv] (decode), ab_dtype = GDN_F32 or io_dtype.
 *   A_log, dt_bias  [Hv] fp32, device.
 * Every other argument, layout and error behaviour is that of gdn_chunk_fwd /
 * gdn_decode (beta_dtype is implied).
 */
gdn_status_t gdn_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* a,
                                 const void* b, gdn_dtype_t ab_dtype, const float* A_log,
                                 const float* dt_bias, int B, int T, int Hqk, int Hv, int K, int V,
                                 gdn_dtype_t io_dtype, float scale, int chunk_size,
                                 const float* initial_state, int output_final_state,
                                 float* final_state, int use_qk_l2norm,
                                 const int32_t* cu_seqlens, int num_seqs,
                                 const int32_t* state_indices, int num_slots, void* o,
                                 void* workspace, size_t workspace_bytes, int* dev_status,
                                 void* stream);

gdn_status_t gdn_decode_gated(const void* q, const void* k, const void* v, const void* a,
                              const void* b, gdn_dtype_t ab_dtype, const float* A_log,
                              const float* dt_bias, float* ssm_state, int num_slots,
                              const int32_t* batch_indices, int n, int Hqk, int Hv, int K, int V,
                              gdn_dtype_t io_dtype, float scale, int use_qk_l2norm, void* o,
                              int* dev_status, void* stream);

/*
 * Gated Delta Product ("Megatron-Core API: core.ssm.gated_delta_product",
 * GatedDeltaProductMixer: each token is projected into the V, K, Q, beta and decay terms
 * of a sequence of Householder updates, num_householder = n_h of them; the forked
 * inference kernels chunk at a fixed 64, ssm_inference_chunk_size).  Per token t, with
 * the decay applied once before the first write and the token's single query reading the
 * state after the last write:
 *
 *     S <- exp(g_t) S;   for j = 0..n_h-1:  S <- S + k_tj (beta_tj (v_tj - S^T k_tj))^T;
 *     o_t = scale * S^T q_t
 *
 * (q_t and every k_tj L2-normalised in-kernel when use_qk_l2norm).  n_h = 1 is the gated
 * delta rule.  Layouts, writes of a token consecutive:
 *   q [B, T, Hqk, K];  k [B, T, n_h, Hqk, K];  v [B, T, n_h, Hv, V];  g [B, T, Hv] fp32;
 *   beta [B, T, n_h, Hv] (fp32 or io_dtype);  o [B, T, Hv, V].
 * Every other argument -- scale, chunk_size (64), initial / final states, cu_seqlens (in
 * tokens), state_indices slot caching, dev_status, stream -- and every error rule as in
 * gdn_chunk_fwd.  The workspace (gdn_product_chunk_fwd_workspace_size bytes, 256-byte
 * aligned, caller-owned) holds the query and decay of every write, the outputs of all
 * writes and the chunk kernels' own scratch; n_h = 1 needs only the latter.
 */
size_t gdn_product_chunk_fwd_workspace_size(int B, int T, int n_h, int Hqk, int Hv, int K, int V,
                                            int num_seqs, gdn_dtype_t io_dtype,
                                            gdn_dtype_t beta_dtype);

gdn_status_t gdn_product_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                                   const void* beta, int B, int T, int n_h, int Hqk, int Hv, int K,
                                   int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype,
                                   float scale, int chunk_size, const float* initial_state,
                                   int output_final_state, float* final_state, int use_qk_l2norm,
                                   const int32_t* cu_seqlens, int num_seqs,
                                   const int32_t* state_indices, int num_slots, void* o,
                                   void* workspace, size_t workspace_bytes, int* dev_status,
                                   void* stream);

/*
 * One Gated Delta Product token per request on the slot cache (the decode step of
 * GatedDeltaProductMixer.ssm_decode, same page):
 *   q [n, Hqk, K];  k [n, n_h, Hqk, K];  v [n, n_h, Hv, V];  g [n, Hv] fp32;
 *   beta [n, n_h, Hv];  o [n, Hv, V];
 *   intermediate_states  NULL, or [n, n_h, Hv, K, V] fp32: the state after every write.
 * Slots, padding (-1: zero output row, no state access), defaults and errors as in
 * gdn_decode.
 */
gdn_status_t gdn_product_decode(const void* q, const void* k, const void* v, const float* g,
                                const void* beta, float* ssm_state, int num_slots,
                                const int32_t* batch_indices, int n, int n_h, int Hqk, int Hv,
                                int K, int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype,
                                float scale, int use_qk_l2norm, void* o,
                                float* intermediate_states, int* dev_status, void* stream);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd without caller-provided scratch.
 *
 * The sources have no counterpart for this entry point; it exists for callers
 * that cannot allocate device memory: plugins running inside another runtime
 * whose device memory that runtime has already reserved, C callers without an
 * allocator of their own, and code that must not call cudaMalloc mid-step
 * because cudaMalloc can synchronise the device.
 *
 * Arguments, layouts and results are those of gdn_chunk_fwd without
 * `workspace` / `workspace_bytes`: the scratch the CUDA-core chunk kernels need
 * comes from one static device array of GDN_NOALLOC_SCRATCH_BYTES (64 MiB) that
 * every GPU loading the library holds until the process exits.  Nothing is
 * allocated or freed per call.
 *   - Sizes whose scratch need (gdn_chunk_fwd_workspace_size) exceeds
 *     GDN_NOALLOC_SCRATCH_BYTES are rejected with GDN_ERR_WORKSPACE before
 *     anything is launched when the CUDA-core path serves them; other argument
 *     errors as in gdn_chunk_fwd.
 *   - Cases the tensor-core kernel serves (bf16, K = V = 128) get the static
 *     array as their workspace and run exactly as through gdn_chunk_fwd (without
 *     the launch plan when it does not fit).
 *   - Every call looks up the array's device address in the current context
 *     (cudaGetSymbolAddress; nothing is cached, so a context created again after
 *     cudaDeviceReset is handled and a failed lookup is retried on the next call).
 *     The first call on a device may load the module: make it before any stream
 *     capture.  `stream` must belong to the current device (NULL: the current
 *     device's default stream); a stream of another device is rejected with
 *     GDN_ERR_CUDA before any launch.
 *   - Every call on a device shares the one array.  No scratch contents need to
 *     start at zero (each launch writes everything it later reads), but calls
 *     whose work overlaps on the GPU (different streams, or concurrent host
 *     threads) race on it: serialise them.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status_t gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                   const void* beta, int B, int T, int Hqk, int Hv, int K, int V,
                                   gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                                   int chunk_size, const float* initial_state,
                                   int output_final_state, float* final_state, int use_qk_l2norm,
                                   const int32_t* cu_seqlens, int num_seqs,
                                   const int32_t* state_indices, int num_slots, void* o,
                                   int* dev_status, void* stream);

/*
 * gdn_chunk_bwd -- backward (training) of the chunkwise gated delta rule.
 *
 * Training runs the chunked rule ("Megatron-Core API: core.ssm.gated_delta_net.gdn",
 * torch_chunk_gated_delta_rule, whose deterministic mode is the reason it exists;
 * "Megatron-Core API: core.ssm.gated_delta_product", _gdp_chunk_forward, shared by
 * training and prefill).  The sources print no backward: this returns the exact
 * gradients of gdn_chunk_fwd's outputs, computed chunkwise with fp32 accumulation
 * (bf16 I/O with K = V = 128: every product on the tcgen05 tensor cores with bf16
 * operands; otherwise fp32 on the CUDA cores), with no atomics (bitwise identical
 * from run to run).
 *
 * Forward arguments (q, k, v, g, beta, B, T, Hqk, Hv, K, V, io_dtype, beta_dtype,
 * scale, chunk_size = 64, initial_state [N, Hv, K, V] or NULL, use_qk_l2norm,
 * cu_seqlens, num_seqs) are those of the forward call being differentiated, with
 * the same layouts and rules as gdn_chunk_fwd; there is no slot cache here
 * (state_indices) and g / beta are given (not the fused gates).
 *   d_o          [B, T, Hv, V] io_dtype, device: gradient of the loss w.r.t. o.
 *   d_final_state  [N, Hv, K, V] fp32, device, or NULL (zero): gradient w.r.t.
 *                the final states.
 *   dq, dk       [B, T, Hqk, K] io_dtype, device, written completely (the value
 *                heads sharing a query/key head are summed).
 *   dv           [B, T, Hv, V] io_dtype, device, written completely.
 *   dg, dbeta    [B, T, Hv] fp32, device, written completely.
 *   d_initial_state  [N, Hv, K, V] fp32, device, or NULL (not computed).
 * Tokens past the last sequence (cu_seqlens[N] < T) get zero gradients.  A
 * non-monotone cu_seqlens is reported as GDN_DEV_BAD_CU_SEQLENS and every
 * gradient is written as zero.
 *   workspace, workspace_bytes  device scratch of at least
 *                gdn_chunk_bwd_workspace_size(...) bytes, 16-byte aligned, owned
 *                by the caller: per chunk of C = 64 tokens and value head, about
 *                2 (2 K V + 2 C V) + 4 (C C + 4 C + 320) bytes on the tensor-core path,
 *                4 (3 K V + 3 C V + C K + C C + 5 C) bytes on the CUDA-core path, which
 *                also keeps 8 Hv K bytes per token.
 * Errors as gdn_chunk_fwd: host-side checks return a status before any launch.
 */
gdn_status_t gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                           const void* beta, int B, int T, int Hqk, int Hv, int K, int V,
                           gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                           int chunk_size, const float* initial_state, int use_qk_l2norm,
                           const int32_t* cu_seqlens, int num_seqs, const void* d_o,
                           const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                           float* dbeta, float* d_initial_state, void* workspace,
                           size_t workspace_bytes, int* dev_status, void* stream);

/* Device scratch (bytes) gdn_chunk_bwd needs; (size_t)-1 for rejected sizes. */
size_t gdn_chunk_bwd_workspace_size(int B, int T, int Hqk, int Hv, int K, int V, int num_seqs,
                                    gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype);

/*
 * gdn_chunk_bwd_gated -- backward of gdn_chunk_fwd_gated: the gradients reach the gate
 * features and the per-head gate parameters ("Megatron-Core API: core.ssm.gated_delta_net.gdn",
 * GatedDeltaNet._compute_gates: "the per-head log-decay g and the write strength beta" from
 * A_log and dt_bias).  With x = a + dt_bias[h] and the chunked backward's dg, dbeta:
 *     da = dg * (-exp(A_log[h]) * sigmoid(x)),       db = dbeta * beta * (1 - beta),
 *     dA_log[h] = sum over every token of dg * g,     ddt_bias[h] = sum over every token of da,
 * the derivative of g = -exp(A_log) softplus(x) and beta = sigmoid(b).  g and beta are evaluated
 * in fp32 as the fused forward evaluates them; the two sums are deterministic (fixed-order
 * per-CTA partials added in block order in fp64), so the whole call is bitwise reproducible.
 *
 * Arguments: those of gdn_chunk_bwd with the fused-gate inputs of gdn_chunk_fwd_gated (a, b
 * [B, T, Hv] ab_dtype = GDN_F32 or io_dtype; A_log, dt_bias [Hv] fp32) in place of g and beta.
 *   dq, dk, dv, d_initial_state  as gdn_chunk_bwd.
 *   da, db        [B, T, Hv] fp32, device, written completely (zero past the last sequence).
 *   dA_log, ddt_bias  [Hv] fp32, device.
 *   workspace     gdn_chunk_bwd_gated_workspace_size(...) bytes, 256-byte aligned: the chunked
 *                 backward's scratch followed by g, beta, dg, dbeta (4 bytes per token and head
 *                 each) and the partial sums.
 * Hv must be at most 256 (GDN_ERR_UNSUPPORTED).  Other errors as gdn_chunk_bwd.
 */
gdn_status_t gdn_chunk_bwd_gated(const void* q, const void* k, const void* v, const void* a,
                                 const void* b, gdn_dtype_t ab_dtype, const float* A_log,
                                 const float* dt_bias, int B, int T, int Hqk, int Hv, int K, int V,
                                 gdn_dtype_t io_dtype, float scale, int chunk_size,
                                 const float* initial_state, int use_qk_l2norm,
                                 const int32_t* cu_seqlens, int num_seqs, const void* d_o,
                                 const float* d_final_state, void* dq, void* dk, void* dv,
                                 float* da, float* db, float* dA_log, float* ddt_bias,
                                 float* d_initial_state, void* workspace, size_t workspace_bytes,
                                 int* dev_status, void* stream);

/* Workspace (bytes) of gdn_chunk_bwd_gated; (size_t)-1 for sizes it would reject. */
size_t gdn_chunk_bwd_gated_workspace_size(int B, int T, int Hqk, int Hv, int K, int V,
                                          int num_seqs, gdn_dtype_t io_dtype);

/*
 * gdn_selftest_wait_timeout -- the bounded wait of the fused kernels, run on its own.
 *
 * The sources have no counterpart for this entry point: it tests the failure detection of
 * this library.  Every mbarrier wait inside the tensor-core kernels has a time limit; a wait
 * that runs out sets GDN_DEV_TIMEOUT in *dev_status and the kernel returns instead of
 * hanging.  This launches one thread that waits, with the same helper and nothing else in
 * flight, on an mbarrier that nobody arrives on (arrive_first = 0: the wait gives up after
 * limit_ns and GDN_DEV_TIMEOUT is OR-ed into *dev_status) or that the thread has already
 * arrived on (arrive_first = 1: the wait succeeds, nothing is reported).
 *
 *   dev_status  device int (required) receiving GDN_DEV_* bits.
 *   limit_ns    the wait's limit, 1 ns .. 100 ms (else GDN_ERR_SHAPE).
 *   waited_ns   NULL or a device unsigned long long receiving the time the wait took
 *               (global timer).
 *   stream      CUDA stream (cudaStream_t) of the current device; the call is asynchronous.
 */
gdn_status_t gdn_selftest_wait_timeout(int* dev_status, unsigned long long limit_ns,
                                       int arrive_first, unsigned long long* waited_ns,
                                       void* stream);

/* Static, NUL-terminated name of a status code ("GDN_OK", ...). */
const char* gdn_status_string(gdn_status_t status);

/* Library version as major * 10000 + minor * 100 + patch. */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
