// gdn_internal.h -- launchers behind the C ABI (not part of the public header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Where the log-decay g and the write strength beta come from.  kGatesGiven: the
// g / beta tensors.  kGatesFused: computed in the kernels from the raw gate
// features a, b and the per-head parameters A_log, dt_bias:
//   g = -exp(A_log[h]) * softplus(a + dt_bias[h]),   beta = sigmoid(b).
enum { kGatesGiven = 0, kGatesFused = 1 };

struct GateArgs {
  int mode;
  const void* a;           // [.., Hv], ab_dtype
  const void* b;           // [.., Hv], ab_dtype
  int ab_dtype;
  const float* A_log;      // [Hv]
  const float* dt_bias;    // [Hv]
};

// One unit of work of the tensor-core forward when it runs from a unit table (the planned
// launch): value head h of the token range [bos, eos) of sequence n, chunked from bos.
// init / fin: the [K][V] fp32 state entering / leaving the range (NULL: a zero entry state /
// no exit state written).  flags: kUnit* below.
struct TcUnit {
  const float* init;
  float* fin;
  int n, h, bos, eos;
  int flags;
  int pad_;
};
enum {
  kUnitZeroV = 1,      // v read as zero (no V loads): the transition run of a segment
  kUnitIdentity = 2,   // entry state = identity (K = V): with kUnitZeroV, the segment's K x K map
  kUnitNoOut = 4,      // o not written
  kUnitPadding = 8,    // padding sequence: o rows of the range zeroed, no state access
  kUnitSkip = 16,      // rejected sequence (bad cu_seqlens): nothing written
  kUnitFinT = 32       // exit state written transposed ([V][K])
};

// The reverse pass's per-(chunk, value head) vectors (zero at tokens past the chunk end):
//   [kRvCq + i]    scale gamma_i r_q,i      the q rows of the dS update
//   [kRvW + j]     lambda_j r_k,j           the columns of Y^T = dS^T K^T over raw k rows
//   [kRvF + i]     -gamma_i beta_i r_k,i    the dX^T operand of the dS update (raw k rows)
//   [kRvBeta + i]  beta_i                   dv = diag(beta) dX
//   [kRvGl]        gamma_L = e^{G_{L-1}}    the decay of dS across the chunk
// with r_q, r_k the l2-norm reciprocals (1 without the norm), G the in-chunk cumulative
// log-decay and lambda_j = e^{G_{L-1} - G_j}.
constexpr int kRvCq = 0, kRvW = 64, kRvF = 128, kRvBeta = 192, kRvGl = 256, kRvFloats = 320;

struct ChunkArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const void* beta;
  int B, T, Hqk, Hv, K, V;
  int io_dtype, beta_dtype;
  float scale;
  const float* initial_state;
  float* final_state;  // NULL when no final state is requested
  int use_qk_l2norm;
  const int32_t* cu_seqlens;  // NULL: uniform rows of T tokens
  int num_seqs;               // N
  const int32_t* state_indices;
  int num_slots;
  void* o;
  void* workspace;
  size_t workspace_bytes;
  int* dev_status;
  cudaStream_t stream;
  GateArgs gates;
  // Record mode of the tensor-core kernel (the backward's forward recompute): when set, the
  // state entering every chunk and U' go out as bf16 operand tiles of the backward's
  // tensor-core grad pass (128-byte swizzled, K-major: rows dk resp. tokens, dv along the
  // rows in two 64-element halves), one per chunk and head in slots of K V / 2 resp. 64 V / 2
  // floats (32 KB / 16 KB) of rec_states / rec_u; chunk numbering from the device chunk table
  // rec_chunk_off.
  float* rec_states = nullptr;
  float* rec_u = nullptr;
  const int32_t* rec_chunk_off = nullptr;
  // and, for the reverse pass, per chunk and head: T = (I + A)^{-1} transposed (element (i, j)
  // = T[j][i], the layout of a K-major B operand) and P (element (i, j) = P[i][j]), both bf16
  // 128-byte swizzled [64][64] tiles, together in a 16 KB slot of rec_tp; the per-token vectors
  // of the reverse pass (kRv* below) in a slot of kRvFloats floats of rec_vec
  float* rec_tp = nullptr;
  float* rec_vec = nullptr;
  // Planned launch: CTA i runs units[i] when i < *unit_count (device memory), else exits.
  const TcUnit* units = nullptr;
  const int* unit_count = nullptr;
  int unit_cap = 0;   // CTAs launched (an upper bound of *unit_count)
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const void* beta;
  float* state;
  int num_slots;
  const int32_t* batch_indices;
  int n, Hqk, Hv, K, V;
  int io_dtype, beta_dtype;
  float scale;
  int use_qk_l2norm;
  void* o;
  int* dev_status;
  cudaStream_t stream;
  GateArgs gates;
  int L;                // tokens per request (1 for the single-token step)
  float* intermediate;  // [n, L, Hv, K, V] state after every token, or NULL
  int product;          // 1: Gated Delta Product -- the L entries of a request are the
                        // writes of one token: q [n, Hqk, K] and g [n, Hv] per request,
                        // decay on the first write, output [n, Hv, V] after the last
};

// Upper bound on the number of 64-token chunks over all sequences.
inline long long max_chunks(int T_total, int num_seqs) {
  return ((long long)T_total + 63) / 64 + (long long)num_seqs;
}

// fp32 CUDA-core chunk path (any accepted K, V, dtype).
size_t chunk_generic_workspace_bytes(int T_total, int num_seqs, int Hv, int K, int V);
cudaError_t launch_chunk_generic(const ChunkArgs& a);

// The serial state pass of the fp32 chunk path on caller-provided buffers: from the
// per-chunk W = T diag(beta exp G) K, U = T diag(beta) V and in-chunk cumulative G
// ([NC][Hv][C][K], [NC][Hv][C][V], [NC][Hv][C]), records the state at every chunk
// entry in S [NC][Hv][K][V] and overwrites U with U' = U - W S.  chunk_off is the
// device chunk table (launch_chunk_table).
cudaError_t launch_chunk_states(const ChunkArgs& a, int32_t* chunk_off, float* W, float* U,
                                float* G, float* S);
// The prep pass of the fp32 chunk path on caller-provided buffers: W, U and G per chunk.
cudaError_t launch_chunk_prep(const ChunkArgs& a, int32_t* chunk_off, float* W, float* U,
                              float* G);

// Gradients for the backward of the chunkwise rule (all device pointers).
struct BwdArgs {
  const void* d_o;        // [T_total, Hv, V] io dtype
  const float* d_final;   // [N, Hv, K, V] or NULL (zero)
  void* dq;               // [T_total, Hqk, K] io dtype
  void* dk;               // [T_total, Hqk, K] io dtype
  void* dv;               // [T_total, Hv, V] io dtype
  float* dg;              // [T_total, Hv]
  float* dbeta;           // [T_total, Hv]
  float* d_initial;       // [N, Hv, K, V] or NULL
};

// Backward of the chunkwise rule (given gates, no slot cache): every product on the tensor
// cores for bf16 with K = V = 128 (tc), else fp32 on the CUDA cores; the two paths lay their
// scratch out differently.
bool chunk_bwd_uses_tc(int K, int V, int io_dtype, int beta_dtype);
size_t chunk_bwd_workspace_bytes(int T_total, int num_seqs, int Hv, int K, int V, bool tc);
cudaError_t launch_chunk_bwd(const ChunkArgs& a, const BwdArgs& b);

// Fused tcgen05 / TMEM / TMA path (bf16, K = V = 128).
bool chunk_tc_supported(int K, int V, int io_dtype, int beta_dtype);
// TMA map of a [T_total, H, 128] bf16 tensor with 64 x 1 x 64 boxes (64 features of one head
// for 64 tokens, 128-byte swizzled), zero fill past the last token.
bool encode_rows_map_bf16(CUtensorMap* m, const void* base, int H, int T_total);
cudaError_t launch_chunk_tc(const ChunkArgs& a);
// The planned forward (a.workspace): sequences sorted longest first, and, when the batch has
// too few (sequence, head) chains to fill the GPU, sequences of at least 2 s chunks split into
// s segments joined through the linearity of the chunk map S -> M S + B (a transition and a
// contribution run per middle segment, a scan, then every segment run from its exact entry
// state).  Falls back to launch_chunk_tc when the workspace is smaller than
// chunk_tc_plan_bytes.  num_sms: the SM count the plan is sized for.
int chunk_tc_segments(int num_seqs, int Hv, int num_sms);
// SM count of device dev (cached per device), 0 if it cannot be read.
int device_sm_count(int dev);
size_t chunk_tc_plan_bytes(int num_seqs, int Hv, int segments);
cudaError_t launch_chunk_tc_planned(const ChunkArgs& a);

cudaError_t launch_decode(const DecodeArgs& a);

// Backward through the fused gates: g and beta materialised (fp32) from the gate features, and
// the chain rule from dg, dbeta to da, db ([T_total, Hv] fp32) and dA_log, ddt_bias ([Hv],
// deterministic sums).  Hv <= 256.  gates_bwd_extra_bytes: the scratch for g, beta, dg, dbeta
// and the per-CTA partial sums (each part 256-byte aligned, in that order).
size_t gates_bwd_extra_bytes(long long T_total, int Hv);
cudaError_t launch_gates_materialise(const GateArgs& ga, long long T_total, int Hv, float* g,
                                     float* beta, cudaStream_t stream);
cudaError_t launch_gates_bwd(const GateArgs& ga, const float* dg, const float* dbeta,
                             long long T_total, int Hv, float* da, float* db, float* dA_log,
                             float* ddt_bias, float* partial, cudaStream_t stream);

// Gated Delta Product as the gated delta rule over the sequence of writes: q' (the query on
// the last write of each token), g' (the decay on the first), n_h * cu_seqlens, and the
// output rows of the last writes gathered back.
cudaError_t launch_product_expand(const void* q, const float* g, void* q_exp, float* g_exp,
                                  const int32_t* cu, int32_t* cu_exp, long long T_total, int n_h,
                                  int Hqk, int Hv, int K, int io_dtype, int num_seqs,
                                  cudaStream_t stream);
cudaError_t launch_product_gather(const void* o_exp, void* o, long long T_total, int n_h, int Hv,
                                  int V, int io_dtype, cudaStream_t stream);

}  // namespace gdn
