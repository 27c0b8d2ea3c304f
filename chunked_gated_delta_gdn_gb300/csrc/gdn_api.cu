// gdn_api.cu -- the extern "C" boundary of libgdn: argument validation and
// dispatch to the kernels.  Declarations and the full contract are in gdn.h.
#include <math.h>
#include <stdint.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

bool is_dtype(int d) { return d == GDN_F32 || d == GDN_BF16; }
size_t elem_size(int d) { return d == GDN_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

float resolve_scale(float scale, int K) {
  return isnan(scale) ? 1.0f / sqrtf((float)K) : scale;
}

// Shape / dtype checks shared by the chunk entry point and its size queries.
gdn_status_t check_chunk_shapes(int B, int T, int Hqk, int Hv, int K, int V, int io_dtype,
                                int beta_dtype) {
  if (!is_dtype(io_dtype) || !is_dtype(beta_dtype)) return GDN_ERR_DTYPE;
  if (beta_dtype != GDN_F32 && beta_dtype != io_dtype) return GDN_ERR_DTYPE;
  if (B < 0 || T < 0 || Hqk <= 0 || Hv <= 0 || Hv % Hqk != 0) return GDN_ERR_SHAPE;
  if (K <= 0 || V <= 0 || K > GDN_MAX_HEAD_DIM || V > GDN_MAX_HEAD_DIM) return GDN_ERR_SHAPE;
  if ((K * elem_size(io_dtype)) % 16 != 0 || (V * elem_size(io_dtype)) % 16 != 0)
    return GDN_ERR_SHAPE;
  if ((long long)B * T > 0x7fffffffLL) return GDN_ERR_SHAPE;
  return GDN_OK;
}

// Arguments of the fused-gate entry points (checked before anything else).
gdn_status_t check_gate_args(const void* a, const void* b, int ab_dtype, const float* A_log,
                             const float* dt_bias, int io_dtype, long long count) {
  if (!is_dtype(ab_dtype) || (ab_dtype != GDN_F32 && ab_dtype != io_dtype)) return GDN_ERR_DTYPE;
  if (count > 0 && (!a || !b || !A_log || !dt_bias)) return GDN_ERR_NULL;
  if (((uintptr_t)a & (elem_size(ab_dtype) - 1)) || ((uintptr_t)b & (elem_size(ab_dtype) - 1)) ||
      ((uintptr_t)A_log & 3u) || ((uintptr_t)dt_bias & 3u))
    return GDN_ERR_LAYOUT;
  return GDN_OK;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status_t s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_NULL: return "GDN_ERR_NULL";
    case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE";
    case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE";
    case GDN_ERR_LAYOUT: return "GDN_ERR_LAYOUT";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
  }
  return "GDN_ERR_UNKNOWN";
}

int gdn_version(void) { return 100; }

int gdn_chunk_fwd_path(int K, int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype) {
  if (check_chunk_shapes(1, 1, 1, 1, K, V, io_dtype, beta_dtype) != GDN_OK) return -1;
  return gdn::chunk_tc_supported(K, V, io_dtype, beta_dtype) ? 1 : 0;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// SM count of the current device, 0 when there is none.
static int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return gdn::device_sm_count(dev);
}

size_t gdn_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int K, int V, int num_seqs,
                                    gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype) {
  if (check_chunk_shapes(B, T, Hqk, Hv, K, V, io_dtype, beta_dtype) != GDN_OK || num_seqs < 0)
    return (size_t)-1;
  if (gdn::chunk_tc_supported(K, V, io_dtype, beta_dtype)) {
    const int N = num_seqs > 0 ? num_seqs : B;
    return gdn::chunk_tc_plan_bytes(N, Hv, gdn::chunk_tc_segments(N, Hv, current_sm_count()));
  }
  const long long T_total = (long long)B * T;
  return gdn::chunk_generic_workspace_bytes((int)T_total, num_seqs, Hv, K, V);
}

static gdn_status_t chunk_impl(const void* q, const void* k, const void* v, const float* g,
                               const void* beta, int B, int T, int Hqk, int Hv, int K, int V,
                               gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                               int chunk_size, const float* initial_state, int output_final_state,
                               float* final_state, int use_qk_l2norm, const int32_t* cu_seqlens,
                               int num_seqs, const int32_t* state_indices, int num_slots, void* o,
                               void* workspace, size_t workspace_bytes, int* dev_status,
                               void* stream, const gdn::GateArgs& gates) {
  gdn_status_t st = check_chunk_shapes(B, T, Hqk, Hv, K, V, io_dtype, beta_dtype);
  if (st != GDN_OK) return st;
  if (chunk_size != 64) return GDN_ERR_UNSUPPORTED;
  if (cu_seqlens) {
    if (B != 1 || num_seqs < 0) return GDN_ERR_SHAPE;
  } else {
    num_seqs = B;
  }
  const long long T_total = (long long)B * T;
  if (T_total > 0 && (!q || !k || !v || !o)) return GDN_ERR_NULL;
  if (T_total > 0 && gates.mode == gdn::kGatesGiven && (!g || !beta)) return GDN_ERR_NULL;
  if (output_final_state && !final_state) return GDN_ERR_NULL;
  if (state_indices) {
    if (num_slots <= 0) return GDN_ERR_SHAPE;
  }
  if (T_total > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
                      ((uintptr_t)beta & (elem_size(beta_dtype) - 1)) || ((uintptr_t)g & 3u)))
    return GDN_ERR_LAYOUT;
  if ((initial_state && !aligned16(initial_state)) ||
      (output_final_state && !aligned16(final_state)))
    return GDN_ERR_LAYOUT;
  if (num_seqs == 0) return GDN_OK;

  gdn::ChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.B = B; a.T = T; a.Hqk = Hqk; a.Hv = Hv; a.K = K; a.V = V;
  a.io_dtype = io_dtype; a.beta_dtype = beta_dtype;
  a.scale = resolve_scale(scale, K);
  a.initial_state = initial_state;
  a.final_state = output_final_state ? final_state : nullptr;
  a.use_qk_l2norm = use_qk_l2norm ? 1 : 0;
  a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs;
  a.state_indices = state_indices;
  a.num_slots = num_slots;
  a.o = o;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.dev_status = dev_status;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.gates = gates;

  cudaError_t err;
  if (gdn::chunk_tc_supported(K, V, io_dtype, beta_dtype)) {
    err = gdn::launch_chunk_tc_planned(a);
  } else {
    const size_t need = gdn::chunk_generic_workspace_bytes((int)T_total, num_seqs, Hv, K, V);
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GDN_ERR_LAYOUT;
    err = gdn::launch_chunk_generic(a);
  }
  return err == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                           const void* beta, int B, int T, int Hqk, int Hv, int K, int V,
                           gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                           int chunk_size, const float* initial_state, int output_final_state,
                           float* final_state, int use_qk_l2norm, const int32_t* cu_seqlens,
                           int num_seqs, const int32_t* state_indices, int num_slots, void* o,
                           void* workspace, size_t workspace_bytes, int* dev_status,
                           void* stream) {
  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesGiven;
  return chunk_impl(q, k, v, g, beta, B, T, Hqk, Hv, K, V, io_dtype, beta_dtype, scale,
                    chunk_size, initial_state, output_final_state, final_state, use_qk_l2norm,
                    cu_seqlens, num_seqs, state_indices, num_slots, o, workspace,
                    workspace_bytes, dev_status, stream, gates);
}

gdn_status_t gdn_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* a,
                                 const void* b, gdn_dtype_t ab_dtype, const float* A_log,
                                 const float* dt_bias, int B, int T, int Hqk, int Hv, int K, int V,
                                 gdn_dtype_t io_dtype, float scale, int chunk_size,
                                 const float* initial_state, int output_final_state,
                                 float* final_state, int use_qk_l2norm,
                                 const int32_t* cu_seqlens, int num_seqs,
                                 const int32_t* state_indices, int num_slots, void* o,
                                 void* workspace, size_t workspace_bytes, int* dev_status,
                                 void* stream) {
  gdn_status_t st = check_gate_args(a, b, ab_dtype, A_log, dt_bias, io_dtype, (long long)B * T);
  if (st != GDN_OK) return st;
  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesFused;
  gates.a = a;
  gates.b = b;
  gates.ab_dtype = ab_dtype;
  gates.A_log = A_log;
  gates.dt_bias = dt_bias;
  // beta_dtype only selects the kernel family here; the fused gates replace g / beta.
  return chunk_impl(q, k, v, nullptr, nullptr, B, T, Hqk, Hv, K, V, io_dtype, io_dtype, scale,
                    chunk_size, initial_state, output_final_state, final_state, use_qk_l2norm,
                    cu_seqlens, num_seqs, state_indices, num_slots, o, workspace,
                    workspace_bytes, dev_status, stream, gates);
}

size_t gdn_chunk_bwd_workspace_size(int B, int T, int Hqk, int Hv, int K, int V, int num_seqs,
                                    gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype) {
  if (check_chunk_shapes(B, T, Hqk, Hv, K, V, io_dtype, beta_dtype) != GDN_OK || num_seqs < 0)
    return (size_t)-1;
  return gdn::chunk_bwd_workspace_bytes((int)((long long)B * T), num_seqs, Hv, K, V,
                                        gdn::chunk_bwd_uses_tc(K, V, io_dtype, beta_dtype));
}

gdn_status_t gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                           const void* beta, int B, int T, int Hqk, int Hv, int K, int V,
                           gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                           int chunk_size, const float* initial_state, int use_qk_l2norm,
                           const int32_t* cu_seqlens, int num_seqs, const void* d_o,
                           const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                           float* dbeta, float* d_initial_state, void* workspace,
                           size_t workspace_bytes, int* dev_status, void* stream) {
  gdn_status_t st = check_chunk_shapes(B, T, Hqk, Hv, K, V, io_dtype, beta_dtype);
  if (st != GDN_OK) return st;
  if (chunk_size != 64) return GDN_ERR_UNSUPPORTED;
  if (cu_seqlens) {
    if (B != 1 || num_seqs < 0) return GDN_ERR_SHAPE;
  } else {
    num_seqs = B;
  }
  const long long T_total = (long long)B * T;
  if (T_total > 0 && (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta))
    return GDN_ERR_NULL;
  if (T_total > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(d_o) ||
                      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
                      ((uintptr_t)beta & (elem_size(beta_dtype) - 1)) || ((uintptr_t)g & 3u) ||
                      ((uintptr_t)dg & 3u) || ((uintptr_t)dbeta & 3u)))
    return GDN_ERR_LAYOUT;
  if ((initial_state && !aligned16(initial_state)) || (d_final_state && !aligned16(d_final_state)) ||
      (d_initial_state && !aligned16(d_initial_state)))
    return GDN_ERR_LAYOUT;
  if (num_seqs == 0 && T_total == 0) return GDN_OK;
  const size_t need = gdn::chunk_bwd_workspace_bytes((int)T_total, num_seqs, Hv, K, V,
                                                     gdn::chunk_bwd_uses_tc(K, V, io_dtype, beta_dtype));
  if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return GDN_ERR_LAYOUT;

  gdn::ChunkArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.B = B; a.T = T; a.Hqk = Hqk; a.Hv = Hv; a.K = K; a.V = V;
  a.io_dtype = io_dtype; a.beta_dtype = beta_dtype;
  a.scale = resolve_scale(scale, K);
  a.initial_state = initial_state;
  a.final_state = nullptr;
  a.use_qk_l2norm = use_qk_l2norm ? 1 : 0;
  a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs;
  a.state_indices = nullptr;
  a.num_slots = 0;
  a.o = nullptr;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.dev_status = dev_status;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.gates.mode = gdn::kGatesGiven;
  gdn::BwdArgs b;
  b.d_o = d_o;
  b.d_final = d_final_state;
  b.dq = dq; b.dk = dk; b.dv = dv; b.dg = dg; b.dbeta = dbeta;
  b.d_initial = d_initial_state;
  return gdn::launch_chunk_bwd(a, b) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t gdn_chunk_bwd_gated_workspace_size(int B, int T, int Hqk, int Hv, int K, int V,
                                          int num_seqs, gdn_dtype_t io_dtype) {
  const size_t inner = gdn_chunk_bwd_workspace_size(B, T, Hqk, Hv, K, V, num_seqs, io_dtype, GDN_F32);
  if (inner == (size_t)-1 || Hv > 256) return (size_t)-1;
  return ((inner + 255) & ~(size_t)255) + gdn::gates_bwd_extra_bytes((long long)B * T, Hv);
}

gdn_status_t gdn_chunk_bwd_gated(const void* q, const void* k, const void* v, const void* a,
                                 const void* b, gdn_dtype_t ab_dtype, const float* A_log,
                                 const float* dt_bias, int B, int T, int Hqk, int Hv, int K, int V,
                                 gdn_dtype_t io_dtype, float scale, int chunk_size,
                                 const float* initial_state, int use_qk_l2norm,
                                 const int32_t* cu_seqlens, int num_seqs, const void* d_o,
                                 const float* d_final_state, void* dq, void* dk, void* dv,
                                 float* da, float* db, float* dA_log, float* ddt_bias,
                                 float* d_initial_state, void* workspace, size_t workspace_bytes,
                                 int* dev_status, void* stream) {
  gdn_status_t st = check_chunk_shapes(B, T, Hqk, Hv, K, V, io_dtype, GDN_F32);
  if (st != GDN_OK) return st;
  if (Hv > 256) return GDN_ERR_UNSUPPORTED;
  const long long T_total = (long long)B * T;
  st = check_gate_args(a, b, ab_dtype, A_log, dt_bias, io_dtype, T_total);
  if (st != GDN_OK) return st;
  if (!A_log || !dt_bias || !dA_log || !ddt_bias || (T_total > 0 && (!da || !db)))
    return GDN_ERR_NULL;
  if (((uintptr_t)da & 3u) || ((uintptr_t)db & 3u) || ((uintptr_t)dA_log & 3u) ||
      ((uintptr_t)ddt_bias & 3u))
    return GDN_ERR_LAYOUT;
  if (chunk_size != 64) return GDN_ERR_UNSUPPORTED;
  if (cu_seqlens && (B != 1 || num_seqs < 0)) return GDN_ERR_SHAPE;
  const int N = cu_seqlens ? num_seqs : B;
  const size_t need = gdn_chunk_bwd_gated_workspace_size(B, T, Hqk, Hv, K, V, N, io_dtype);
  if (need == (size_t)-1) return GDN_ERR_SHAPE;
  if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return GDN_ERR_LAYOUT;
  const size_t inner = gdn_chunk_bwd_workspace_size(B, T, Hqk, Hv, K, V, N, io_dtype, GDN_F32);
  uint8_t* w = reinterpret_cast<uint8_t*>(workspace);
  const size_t part = align256((size_t)T_total * Hv * sizeof(float));
  size_t off = align256(inner);
  float* g = reinterpret_cast<float*>(w + off); off += part;
  float* beta = reinterpret_cast<float*>(w + off); off += part;
  float* dg = reinterpret_cast<float*>(w + off); off += part;
  float* dbeta = reinterpret_cast<float*>(w + off); off += part;
  float* partial = reinterpret_cast<float*>(w + off);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesFused;
  gates.a = a;
  gates.b = b;
  gates.ab_dtype = ab_dtype;
  gates.A_log = A_log;
  gates.dt_bias = dt_bias;
  if (gdn::launch_gates_materialise(gates, T_total, Hv, g, beta, s) != cudaSuccess) return GDN_ERR_CUDA;
  st = gdn_chunk_bwd(q, k, v, g, beta, B, T, Hqk, Hv, K, V, io_dtype, GDN_F32, scale, chunk_size,
                     initial_state, use_qk_l2norm, cu_seqlens, num_seqs, d_o, d_final_state, dq,
                     dk, dv, dg, dbeta, d_initial_state, workspace, inner, dev_status, stream);
  if (st != GDN_OK) return st;
  return gdn::launch_gates_bwd(gates, dg, dbeta, T_total, Hv, da, db, dA_log, ddt_bias, partial,
                               s) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

static gdn_status_t decode_impl(const void* q, const void* k, const void* v, const float* g,
                                const void* beta, float* ssm_state, int num_slots,
                                const int32_t* batch_indices, int n, int Hqk, int Hv, int K, int V,
                                gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                                int use_qk_l2norm, void* o, int* dev_status, void* stream,
                                const gdn::GateArgs& gates, int L = 1,
                                float* intermediate = nullptr, int product = 0) {
  gdn_status_t st = check_chunk_shapes(1, 1, Hqk, Hv, K, V, io_dtype, beta_dtype);
  if (st != GDN_OK) return st;
  if (n < 0 || num_slots < 0 || L < 0) return GDN_ERR_SHAPE;
  if ((long long)n * L > 0x7fffffffLL) return GDN_ERR_SHAPE;
  if (!batch_indices && n > num_slots) return GDN_ERR_SHAPE;
  if (n == 0 || L == 0) return GDN_OK;
  if (!q || !k || !v || !o || !ssm_state) return GDN_ERR_NULL;
  if (intermediate && !aligned16(intermediate)) return GDN_ERR_LAYOUT;
  if (gates.mode == gdn::kGatesGiven && (!g || !beta)) return GDN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(ssm_state))
    return GDN_ERR_LAYOUT;
  if (gates.mode == gdn::kGatesGiven &&
      (((uintptr_t)g & 3u) || ((uintptr_t)beta & (elem_size(beta_dtype) - 1))))
    return GDN_ERR_LAYOUT;
  gdn::DecodeArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.state = ssm_state;
  a.num_slots = num_slots;
  a.batch_indices = batch_indices;
  a.n = n; a.Hqk = Hqk; a.Hv = Hv; a.K = K; a.V = V;
  a.io_dtype = io_dtype; a.beta_dtype = beta_dtype;
  a.scale = resolve_scale(scale, K);
  a.use_qk_l2norm = use_qk_l2norm ? 1 : 0;
  a.o = o;
  a.dev_status = dev_status;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.gates = gates;
  a.L = L;
  a.intermediate = intermediate;
  a.product = product;
  return gdn::launch_decode(a) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t gdn_decode(const void* q, const void* k, const void* v, const float* g,
                        const void* beta, float* ssm_state, int num_slots,
                        const int32_t* batch_indices, int n, int Hqk, int Hv, int K, int V,
                        gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                        int use_qk_l2norm, void* o, int* dev_status, void* stream) {
  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesGiven;
  return decode_impl(q, k, v, g, beta, ssm_state, num_slots, batch_indices, n, Hqk, Hv, K, V,
                     io_dtype, beta_dtype, scale, use_qk_l2norm, o, dev_status, stream, gates);
}

gdn_status_t gdn_decode_multi(const void* q, const void* k, const void* v, const float* g,
                              const void* beta, float* ssm_state, int num_slots,
                              const int32_t* batch_indices, int n, int L, int Hqk, int Hv, int K,
                              int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype, float scale,
                              int use_qk_l2norm, void* o, float* intermediate_states,
                              int* dev_status, void* stream) {
  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesGiven;
  return decode_impl(q, k, v, g, beta, ssm_state, num_slots, batch_indices, n, Hqk, Hv, K, V,
                     io_dtype, beta_dtype, scale, use_qk_l2norm, o, dev_status, stream, gates, L,
                     intermediate_states);
}

gdn_status_t gdn_decode_gated(const void* q, const void* k, const void* v, const void* a,
                              const void* b, gdn_dtype_t ab_dtype, const float* A_log,
                              const float* dt_bias, float* ssm_state, int num_slots,
                              const int32_t* batch_indices, int n, int Hqk, int Hv, int K, int V,
                              gdn_dtype_t io_dtype, float scale, int use_qk_l2norm, void* o,
                              int* dev_status, void* stream) {
  gdn_status_t st = check_gate_args(a, b, ab_dtype, A_log, dt_bias, io_dtype, n);
  if (st != GDN_OK) return st;
  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesFused;
  gates.a = a;
  gates.b = b;
  gates.ab_dtype = ab_dtype;
  gates.A_log = A_log;
  gates.dt_bias = dt_bias;
  return decode_impl(q, k, v, nullptr, nullptr, ssm_state, num_slots, batch_indices, n, Hqk, Hv,
                     K, V, io_dtype, io_dtype, scale, use_qk_l2norm, o, dev_status, stream, gates);
}

// ---- Gated Delta Product ("Megatron-Core API: core.ssm.gated_delta_product")


// Workspace of the product's chunk forward: q', g', o' over the T * n_h writes, the scaled
// cu_seqlens, then the chunk kernels' own workspace for the write sequence.
static size_t product_ws_parts(int B, int T, int n_h, int Hqk, int Hv, int K, int V, int num_seqs,
                               int io_dtype, int beta_dtype, size_t* inner_off) {
  const size_t te = (size_t)B * T * n_h, es = elem_size(io_dtype);
  size_t off = align256(te * Hqk * K * es) + align256(te * Hv * 4) + align256(te * Hv * V * es) +
               align256(((size_t)num_seqs + 1) * 4);
  *inner_off = off;
  return off + gdn_chunk_fwd_workspace_size(B, T * n_h, Hqk, Hv, K, V, num_seqs,
                                            (gdn_dtype_t)io_dtype, (gdn_dtype_t)beta_dtype);
}

size_t gdn_product_chunk_fwd_workspace_size(int B, int T, int n_h, int Hqk, int Hv, int K, int V,
                                            int num_seqs, gdn_dtype_t io_dtype,
                                            gdn_dtype_t beta_dtype) {
  if (n_h < 1 || B < 0 || T < 0 || num_seqs < 0 || (long long)B * T * n_h > 0x7fffffffLL)
    return (size_t)-1;
  if (check_chunk_shapes(B, T * n_h, Hqk, Hv, K, V, io_dtype, beta_dtype) != GDN_OK)
    return (size_t)-1;
  if (n_h == 1) return gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, K, V, num_seqs, io_dtype, beta_dtype);
  size_t inner;
  return product_ws_parts(B, T, n_h, Hqk, Hv, K, V, num_seqs, io_dtype, beta_dtype, &inner);
}

gdn_status_t gdn_product_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                                   const void* beta, int B, int T, int n_h, int Hqk, int Hv, int K,
                                   int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype,
                                   float scale, int chunk_size, const float* initial_state,
                                   int output_final_state, float* final_state, int use_qk_l2norm,
                                   const int32_t* cu_seqlens, int num_seqs,
                                   const int32_t* state_indices, int num_slots, void* o,
                                   void* workspace, size_t workspace_bytes, int* dev_status,
                                   void* stream) {
  if (n_h < 1 || B < 0 || T < 0 || (long long)B * T * n_h > 0x7fffffffLL) return GDN_ERR_SHAPE;
  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesGiven;
  if (n_h == 1)   // one write per token: the gated delta rule itself
    return chunk_impl(q, k, v, g, beta, B, T, Hqk, Hv, K, V, io_dtype, beta_dtype, scale,
                      chunk_size, initial_state, output_final_state, final_state, use_qk_l2norm,
                      cu_seqlens, num_seqs, state_indices, num_slots, o, workspace,
                      workspace_bytes, dev_status, stream, gates);
  gdn_status_t st = check_chunk_shapes(B, T * n_h, Hqk, Hv, K, V, io_dtype, beta_dtype);
  if (st != GDN_OK) return st;
  if (chunk_size != 64) return GDN_ERR_UNSUPPORTED;
  if (cu_seqlens) {
    if (B != 1 || num_seqs < 0) return GDN_ERR_SHAPE;
  } else {
    num_seqs = B;
  }
  const long long T_total = (long long)B * T;
  if (T_total > 0 && (!q || !k || !v || !o || !g || !beta)) return GDN_ERR_NULL;
  if (T_total > 0 && (!aligned16(q) || !aligned16(o) || ((uintptr_t)g & 3u)))
    return GDN_ERR_LAYOUT;
  size_t inner_off;
  const size_t need = product_ws_parts(B, T, n_h, Hqk, Hv, K, V, num_seqs, io_dtype, beta_dtype,
                                       &inner_off);
  if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return GDN_ERR_LAYOUT;
  const size_t te = (size_t)T_total * n_h, es = elem_size(io_dtype);
  uint8_t* w = reinterpret_cast<uint8_t*>(workspace);
  void* q_exp = w;
  float* g_exp = reinterpret_cast<float*>(w + align256(te * Hqk * K * es));
  void* o_exp = w + align256(te * Hqk * K * es) + align256(te * Hv * 4);
  int32_t* cu_exp = reinterpret_cast<int32_t*>(w + align256(te * Hqk * K * es) +
                                               align256(te * Hv * 4) + align256(te * Hv * V * es));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (gdn::launch_product_expand(q, g, q_exp, g_exp, cu_seqlens, cu_exp, T_total, n_h, Hqk, Hv,
                                 K, io_dtype, num_seqs, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  st = chunk_impl(q_exp, k, v, g_exp, beta, B, T * n_h, Hqk, Hv, K, V, io_dtype, beta_dtype,
                  scale, chunk_size, initial_state, output_final_state, final_state,
                  use_qk_l2norm, cu_seqlens ? cu_exp : nullptr, num_seqs, state_indices,
                  num_slots, o_exp, w + inner_off, workspace_bytes - inner_off, dev_status,
                  stream, gates);
  if (st != GDN_OK) return st;
  return gdn::launch_product_gather(o_exp, o, T_total, n_h, Hv, V, io_dtype, s) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

gdn_status_t gdn_product_decode(const void* q, const void* k, const void* v, const float* g,
                                const void* beta, float* ssm_state, int num_slots,
                                const int32_t* batch_indices, int n, int n_h, int Hqk, int Hv,
                                int K, int V, gdn_dtype_t io_dtype, gdn_dtype_t beta_dtype,
                                float scale, int use_qk_l2norm, void* o,
                                float* intermediate_states, int* dev_status, void* stream) {
  if (n_h < 1) return GDN_ERR_SHAPE;
  gdn::GateArgs gates{};
  gates.mode = gdn::kGatesGiven;
  return decode_impl(q, k, v, g, beta, ssm_state, num_slots, batch_indices, n, Hqk, Hv, K, V,
                     io_dtype, beta_dtype, scale, use_qk_l2norm, o, dev_status, stream, gates,
                     n_h, intermediate_states, 1);
}

}  // extern "C"
