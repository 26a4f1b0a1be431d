// kda_api.cu -- the C ABI of libkda.so: argument checks, path selection and
// the device status word.  Every check runs on the host before anything is
// enqueued; a rejected call launches nothing.
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {

// Written by device code when a bounded wait gives up (KDA_ERR_TIMEOUT).
__device__ int g_status_word = 0;

unsigned long long current_context_id() {
  // The driver's context queries, reached through the runtime so that the
  // library needs no link against the driver library.
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int* status_word() {
  // looked up once per (device, context): a device reset makes a new context,
  // in which the word has a new address
  static std::mutex m;
  static unsigned long long ctx_of[64] = {0};
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> g(m);
  if (id != 0 && ctx_of[dev] == id && cached[dev]) return cached[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || !p) return nullptr;
  cached[dev] = static_cast<int*>(p);
  ctx_of[dev] = current_context_id();
  return cached[dev];
}

}  // namespace kda

using namespace kda;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// beta is read one element at a time: element alignment is enough
bool beta_aligned(const void* p, int dtype) {
  return (reinterpret_cast<uintptr_t>(p) & (dtype == KDA_BF16 ? 1u : 3u)) == 0;
}
bool supported_d(int d) { return d == 32 || d == 64 || d == 128; }
// log_alpha: required unless there is no decay; a per-head array is read one
// element at a time
bool log_alpha_ok(const float* la, int mode) {
  return mode == KDA_DECAY_NONE || la != nullptr;
}
bool log_alpha_aligned(const float* la, int mode) {
  if (!la || mode == KDA_DECAY_NONE) return true;
  return mode == KDA_DECAY_HEAD ? (reinterpret_cast<uintptr_t>(la) & 3u) == 0 : aligned16(la);
}

const kda_options* opts_or_default(const kda_options* opt, kda_options* storage) {
  if (opt) return opt;
  kda_options_init(storage);
  return storage;
}

int check_common_opts(const kda_options* o) {
  if (o->l2norm_qk != 0 && o->l2norm_qk != 1) return KDA_ERR_ARG;
  if (o->beta_is_logit != 0 && o->beta_is_logit != 1) return KDA_ERR_ARG;
  // The chunked paths rely on the floor: 16 steps of at least e^-5 keep the
  // rescale factors inside fp32/bf16 range.  A higher floor is also safe.
  if (!(o->g_min >= -5.0f && o->g_min <= 0.0f)) return KDA_ERR_ARG;
  if (!(o->eps_l2 >= 0.0f) || !(o->eps_norm >= 0.0f)) return KDA_ERR_ARG;
  if (o->q_scale != o->q_scale) return KDA_ERR_ARG;
  if (o->decay_mode < KDA_DECAY_CHANNEL || o->decay_mode > KDA_DECAY_NONE) return KDA_ERR_ARG;
  if (o->gate && !aligned16(o->gate)) return KDA_ERR_ALIGN;
  if (o->norm_weight && !aligned16(o->norm_weight)) return KDA_ERR_ALIGN;
  if (o->decay_from_logit != 0 && o->decay_from_logit != 1) return KDA_ERR_ARG;
  if (o->decay_from_logit && o->decay_mode != KDA_DECAY_CHANNEL) return KDA_ERR_ARG;
  if ((o->decay_scale && (reinterpret_cast<uintptr_t>(o->decay_scale) & 3u)) ||
      (o->decay_bias && (reinterpret_cast<uintptr_t>(o->decay_bias) & 3u)))
    return KDA_ERR_ALIGN;
  if (o->conv_weight && !aligned16(o->conv_weight)) return KDA_ERR_ALIGN;
  if (o->conv_state && !aligned16(o->conv_state)) return KDA_ERR_ALIGN;
  return KDA_OK;
}

int prefill_path(const kda_options* o, int d, int dtype) {
  if (o->impl == KDA_IMPL_SIMT) return KDA_IMPL_SIMT;
  const bool tc_ok = tc_prefill_supported(d, dtype, o->chunk);
  if (o->impl == KDA_IMPL_TC) return tc_ok ? KDA_IMPL_TC : -1;
  if (o->impl != KDA_IMPL_AUTO) return -1;
  if (o->chunk == 16) return KDA_IMPL_SIMT;
  return tc_ok ? KDA_IMPL_TC : KDA_IMPL_SIMT;
}

}  // namespace

namespace kda {

int check_prefill(const void* q, const void* k, const void* v, const float* log_alpha,
                  const void* beta, const float* S0, const int32_t* cu_seqlens, int N,
                  const void* o, const float* S_T, int T_total, int H, int d_k, int d_v,
                  int dtype, const kda_options* op, int* path_out, int* snap_slots_out) {
  if (N < 1 || H < 1 || T_total < 0) return KDA_ERR_SHAPE;
  // token arrays may be NULL only when there are no tokens
  if (!S_T || (T_total > 0 && (!q || !k || !v || !log_alpha_ok(log_alpha, op->decay_mode) ||
                               !beta || !o)))
    return KDA_ERR_ARG;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
  if (!cu_seqlens && (T_total % N) != 0) return KDA_ERR_SHAPE;
  if (op->max_seqlen < 0 || op->max_seqlen > T_total) return KDA_ERR_SHAPE;
  if (op->chunk != 0 && op->chunk != 16 && op->chunk != 64) return KDA_ERR_ARG;
  const void* ptrs[] = {q, k, v, o, S_T};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_ALIGN;
  if (!log_alpha_aligned(log_alpha, op->decay_mode)) return KDA_ERR_ALIGN;
  if (beta && !beta_aligned(beta, dtype)) return KDA_ERR_ALIGN;
  if ((S0 && !aligned16(S0)) || (cu_seqlens && !aligned16(cu_seqlens))) return KDA_ERR_ALIGN;
  int rc = check_common_opts(op);
  if (rc != KDA_OK) return rc;
  // 64-bit extents: every index below 2^62
  const long long tok_elems = (long long)T_total * H * d_k;
  if (tok_elems < 0) return KDA_ERR_SHAPE;
  // state snapshots every snapshot_every tokens (a multiple of the chunk)
  int snap_slots = 0;
  if (op->snapshot_every < 0 || (op->snapshot_every > 0 && op->snapshot_every % 64 != 0))
    return KDA_ERR_ARG;
  if (op->snapshot_every > 0) {
    if (!op->snapshots) return KDA_ERR_ARG;
    if (!aligned16(op->snapshots)) return KDA_ERR_ALIGN;
    const int L = op->max_seqlen > 0 ? op->max_seqlen : (cu_seqlens ? T_total : T_total / N);
    snap_slots = L / op->snapshot_every;
  }
  const int path = prefill_path(op, d_k, dtype);
  if (path < 0) return KDA_ERR_UNSUPPORTED;
  if (path == KDA_IMPL_SIMT && op->chunk == 64) return KDA_ERR_UNSUPPORTED;
  if (path_out) *path_out = path;
  if (snap_slots_out) *snap_slots_out = snap_slots;
  return KDA_OK;
}

}  // namespace kda

extern "C" {

void kda_options_init(kda_options* opt) {
  if (!opt) return;
  memset(opt, 0, sizeof(*opt));
  opt->chunk = 0;
  opt->l2norm_qk = 1;
  opt->beta_is_logit = 0;
  opt->g_min = -5.0f;
  opt->q_scale = 1.0f;
  opt->eps_l2 = 1e-6f;
  opt->eps_norm = 1e-6f;
  opt->impl = KDA_IMPL_AUTO;
  opt->decay_mode = KDA_DECAY_CHANNEL;
}

int kda_abi_version(void) { return 3; }

const char* kda_status_string(int s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_ARG: return "invalid argument";
    case KDA_ERR_SHAPE: return "inconsistent sizes";
    case KDA_ERR_DTYPE: return "unknown dtype";
    case KDA_ERR_ALIGN: return "pointer not aligned as required";
    case KDA_ERR_UNSUPPORTED: return "unsupported head size or option";
    case KDA_ERR_CUDA: return "CUDA runtime error";
    case KDA_ERR_TIMEOUT: return "a bounded device wait gave up";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

size_t kda_prefill_workspace_size(int T_total, int N, int H, int d_k, int d_v,
                                  const kda_options* opt) {
  kda_options def;
  const kda_options* o = opts_or_default(opt, &def);
  if (T_total < 0 || N < 1 || H < 1 || d_k != d_v || !supported_d(d_k)) return 0;
  const int path = prefill_path(o, d_k, KDA_BF16);
  if (path != KDA_IMPL_TC) return 0;
  return tc_workspace_bytes(T_total, N, H, d_k, o);
}

int kda_prefill_path(int T_total, int N, int H, int d_k, int d_v, int dtype,
                     const kda_options* opt, int* launches, int* chunk) {
  kda_options def;
  const kda_options* op = opts_or_default(opt, &def);
  if (N < 1 || H < 1 || T_total < 0) return KDA_ERR_SHAPE;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
  if (op->chunk != 0 && op->chunk != 16 && op->chunk != 64) return KDA_ERR_ARG;
  const int rc = check_common_opts(op);
  if (rc != KDA_OK) return rc;
  const int path = prefill_path(op, d_k, dtype);
  if (path < 0 || (path == KDA_IMPL_SIMT && op->chunk == 64)) return KDA_ERR_UNSUPPORTED;
  if (launches) *launches = path == KDA_IMPL_TC ? tc_launches(T_total, N, H, d_k, op) : 1;
  if (chunk) *chunk = path == KDA_IMPL_TC ? tc_chunk(op) : 16;
  return path;
}

int kda_prefill(const void* q, const void* k, const void* v, const float* log_alpha,
                const void* beta, const float* S0, const int32_t* cu_seqlens, int N, void* o,
                float* S_T, int T_total, int H, int d_k, int d_v, int dtype,
                const kda_options* opt, kda_stream_t stream) {
  kda_options def;
  const kda_options* op = opts_or_default(opt, &def);
  int path = 0, snap_slots = 0;
  int rc = kda::check_prefill(q, k, v, log_alpha, beta, S0, cu_seqlens, N, o, S_T, T_total, H,
                              d_k, d_v, dtype, op, &path, &snap_slots);
  if (rc != KDA_OK) return rc;

  int* status = status_word();
  if (!status) return KDA_ERR_CUDA;

  PrefillArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta;
  a.S0 = S0; a.cu_seqlens = cu_seqlens; a.o = o; a.S_T = S_T;
  a.gate = op->gate; a.norm_weight = op->norm_weight; a.status = status;
  a.N = N; a.T_total = T_total; a.H = H; a.d = d_k;
  a.l2norm_qk = op->l2norm_qk; a.beta_is_logit = op->beta_is_logit;
  a.decay_mode = op->decay_mode;
  a.g_min = op->g_min; a.q_scale = op->q_scale; a.eps_l2 = op->eps_l2;
  a.eps_norm = op->eps_norm;
  a.snapshots = snap_slots > 0 ? op->snapshots : nullptr;
  a.snapshot_every = op->snapshot_every;
  a.snapshot_slots = snap_slots;
  a.decay_from_logit = op->decay_from_logit;
  a.decay_scale = op->decay_scale;
  a.decay_bias = op->decay_bias;
  a.conv_weight = op->conv_weight;
  a.conv_state = op->conv_weight ? op->conv_state : nullptr;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (path == KDA_IMPL_TC) {
    const size_t need = tc_workspace_bytes(T_total, N, H, d_k, op);
    if (!op->workspace || op->workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(op->workspace)) return KDA_ERR_ALIGN;
    e = launch_prefill_tc(a, op, s);
  } else {
    cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(op->phase_events);
    if (ev && cudaEventRecord(ev[0], s) != cudaSuccess) return KDA_ERR_CUDA;
    e = launch_prefill_simt(a, dtype, s);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[1], s);
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_step(const void* q, const void* k, const void* v, const float* log_alpha,
                    const void* beta, float* S, void* o, int N, int H, int d_k, int d_v,
                    int dtype, const kda_options* opt, kda_stream_t stream) {
  kda_options def;
  const kda_options* op = opts_or_default(opt, &def);
  if (!q || !k || !v || !log_alpha_ok(log_alpha, op->decay_mode) || !beta || !S || !o)
    return KDA_ERR_ARG;
  if (N < 1 || H < 1) return KDA_ERR_SHAPE;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  if (d_k != d_v || !supported_d(d_k)) return KDA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, S, o};
  for (const void* p : ptrs)
    if (!aligned16(p)) return KDA_ERR_ALIGN;
  if (!log_alpha_aligned(log_alpha, op->decay_mode)) return KDA_ERR_ALIGN;
  if (!beta_aligned(beta, dtype)) return KDA_ERR_ALIGN;
  int rc = check_common_opts(op);
  if (rc != KDA_OK) return rc;
  if ((long long)N * H > 0x7fffffffLL) return KDA_ERR_SHAPE;

  DecodeArgs a;
  a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.S = S; a.o = o;
  a.gate = op->gate; a.norm_weight = op->norm_weight;
  a.N = N; a.H = H; a.d = d_k;
  a.l2norm_qk = op->l2norm_qk; a.beta_is_logit = op->beta_is_logit;
  a.decay_mode = op->decay_mode;
  a.g_min = op->g_min; a.q_scale = op->q_scale; a.eps_l2 = op->eps_l2;
  a.eps_norm = op->eps_norm;
  a.decay_from_logit = op->decay_from_logit;
  a.decay_scale = op->decay_scale;
  a.decay_bias = op->decay_bias;
  a.conv_weight = op->conv_weight;
  a.conv_state = op->conv_weight ? op->conv_state : nullptr;
  cudaError_t e = launch_decode(a, dtype, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_gated_rmsnorm(const void* o, const void* gate, const float* w, void* y, int rows,
                      int H, int d_v, float eps, int dtype, kda_stream_t stream) {
  if (!o || !gate || !y) return KDA_ERR_ARG;
  if (rows < 0 || H < 1) return KDA_ERR_SHAPE;
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
  if (!supported_d(d_v)) return KDA_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f)) return KDA_ERR_ARG;
  if (!aligned16(o) || !aligned16(gate) || !aligned16(y) || (w && !aligned16(w)))
    return KDA_ERR_ALIGN;
  const long long units = (long long)rows * H;
  if (units / 32 > 0x7fffffffLL) return KDA_ERR_SHAPE;
  cudaError_t e = launch_gated_rmsnorm(o, gate, w, y, units, d_v, eps, dtype,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_get_last_error(kda_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KDA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
  const int zero = 0;
  if (v != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess)
    return KDA_ERR_CUDA;
  return v;
}

}  // extern "C"
