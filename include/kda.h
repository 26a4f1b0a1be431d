/*
 * kda.h -- C ABI of libkda.so, the GB300 (sm_103a) Kimi Delta Attention core.
 *
 * The operation (stated on "Kimi K3's hybrid block, from first principles",
 * section "From linear attention to the delta rule"; "Kimi K3, explained",
 * section "Kimi Delta Attention: making the radical option work"; "Kimi K3",
 * section "Forgetting different features at different rates"), per sequence,
 * per head h, per token t:
 *
 *     q, k  <- q / sqrt(|q|^2 + eps_l2), k / sqrt(|k|^2 + eps_l2)   (optional)
 *     beta  <- sigmoid(beta)                                         (optional)
 *     a     =  exp(clamp(log_alpha, g_min, 0))          one factor per key channel
 *     S_t   =  (I - beta k k^T) Diag(a) S_{t-1} + beta k v^T         [d_k x d_v]
 *     o_t   =  q_scale * S_t^T q                   (reads the UPDATED state)
 *     y_t   =  o_t / sqrt(mean(o_t^2) + eps_norm) * w * sigmoid(gate_t)  (optional)
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them.  Outputs are written in place.
 *   - Layouts are dense row-major with the shapes given per argument.  Token
 *     arrays are "packed": [T_total][H][d] with the tokens of sequence n at rows
 *     cu_seqlens[n] .. cu_seqlens[n+1]-1.
 *   - dtype selects the element type of q, k, v, beta, gate and o/y:
 *     KDA_F32 or KDA_BF16.  log_alpha, the states and norm_weight are always
 *     fp32.  Pointers must be 16-byte aligned, except beta, which only needs
 *     the alignment of its element type.
 *   - Work is enqueued on `stream` and returns before it finishes.  A negative
 *     return value means the arguments were rejected and NOTHING was launched.
 *     Errors that can only be seen on the device (a bounded wait that gave up)
 *     are recorded in a device status word read by kda_get_last_error().
 *   - Supported head sizes: d_k == d_v in {32, 64, 128}.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* kda_stream_t;

/* Status codes.  0 = success, negative = error. */
enum {
  KDA_OK = 0,
  KDA_ERR_ARG = -1,         /* null pointer, bad option or count           */
  KDA_ERR_SHAPE = -2,       /* sizes inconsistent or cu_seqlens malformed   */
  KDA_ERR_DTYPE = -3,       /* unknown dtype code                           */
  KDA_ERR_ALIGN = -4,       /* a pointer is not aligned as required         */
  KDA_ERR_UNSUPPORTED = -5, /* head size or option combination not built    */
  KDA_ERR_CUDA = -6,        /* the CUDA runtime reported an error           */
  KDA_ERR_TIMEOUT = -7,     /* a bounded device-side wait gave up           */
  KDA_ERR_WORKSPACE = -8    /* workspace missing or smaller than required   */
};

/* Element types of q, k, v, beta, gate, o/y. */
enum { KDA_F32 = 0, KDA_BF16 = 1 };

/* Prefill implementations. */
enum {
  KDA_IMPL_AUTO = 0, /* tensor-core path when built for the shape, else SIMT */
  KDA_IMPL_SIMT = 1, /* fp32 CUDA-core chunked path (chunk 16)              */
  KDA_IMPL_TC = 2    /* tcgen05 tensor-core chunked path                    */
};

/* Decay modes.  KDA keeps one decay per key channel; Gated DeltaNet shrinks the
 * whole state by one factor per head, and DeltaNet has no decay ("Kimi K3",
 * section "Forgetting different features at different rates"; "Kimi K3's
 * hybrid block, from first principles", section "From linear attention to the
 * delta rule").  The recurrence is otherwise the same. */
enum {
  KDA_DECAY_CHANNEL = 0, /* log_alpha [..][H][d_k]: one decay per key channel   */
  KDA_DECAY_HEAD = 1,    /* log_alpha [..][H]: one decay per token and head    */
  KDA_DECAY_NONE = 2     /* alpha = 1; log_alpha is not read and may be NULL   */
};

/*
 * Options.  Always initialise with kda_options_init() and then override.
 */
typedef struct kda_options {
  int chunk;             /* tokens per chunk: 16 or 64; 0 = the path's default   */
  int l2norm_qk;         /* 1 (default): L2-normalise q and k per head per token */
  int beta_is_logit;     /* 0 (default): beta is already in (0,1); 1: sigmoid    */
  float g_min;           /* floor of log alpha, default -5                       */
  float q_scale;         /* read-out multiplier, default 1                       */
  float eps_l2;          /* L2-norm epsilon, default 1e-6                        */
  float eps_norm;        /* RMSNorm epsilon, default 1e-6                        */
  const void* gate;      /* NULL: return o.  Else gate logits [T][H][d_v] (dtype)
                            and the output is y = RMSNorm(o) * w * sigmoid(gate) */
  const float* norm_weight; /* RMSNorm weight [d_v] fp32, NULL = ones            */
  void* workspace;       /* device scratch, >= kda_prefill_workspace_size()      */
  size_t workspace_bytes;
  int max_seqlen;        /* host-side bound on the longest sequence, 0 = T_total */
  int impl;              /* KDA_IMPL_*                                           */
  int debug_timeout;     /* test hook: 1 = the first bounded device wait gives up
                            immediately and reports KDA_ERR_TIMEOUT              */
  long long timeout_spins; /* spin limit of bounded device waits, 0 = default   */
  void* const* phase_events; /* NULL, or (launches + 1) cudaEvent_t handles that
                            kda_prefill records on `stream` before each of its
                            kernels and after the last (per-kernel timing)      */
  int decay_mode;        /* KDA_DECAY_*, default KDA_DECAY_CHANNEL.  With
                            KDA_DECAY_HEAD, log_alpha needs only 4-byte
                            alignment                                            */
  int snapshot_every;    /* 0 (default): off.  Else a positive multiple of 64:
                            kda_prefill also writes the state after every
                            prefix of m * snapshot_every tokens of each
                            sequence, for prefix caching ("What's new in Kimi
                            K3", section "What it costs to serve": a KDA prefix
                            can only be reused where its state was saved)     */
  float* snapshots;      /* with snapshot_every: fp32
                            [N][L / snapshot_every][H][d_k][d_v], L =
                            max_seqlen (or T_total / N without cu_seqlens,
                            T_total with them); slot m of sequence n holds
                            the state after (m + 1) * snapshot_every of its
                            tokens, slots past its length are not written   */
  /* The prologue from raw projections ("Kimi K3's hybrid block, from first
   * principles", section "From linear attention to the delta rule"; section
   * "What changed": the decay mapping became a bounded sigmoid). */
  int decay_from_logit;  /* 0 (default): log_alpha holds log decays.  1: it holds
                            the decay logits z [T][H][d_k] (KDA_DECAY_CHANNEL
                            only) and log alpha = g_min * sigmoid(A_h (z + b))  */
  const float* decay_scale; /* with decay_from_logit: A [H] fp32, NULL = ones   */
  const float* decay_bias;  /* with decay_from_logit: b [H][d_k] fp32, NULL = 0 */
  const float* conv_weight; /* NULL (default): q, k, v are used as given.  Else
                            fp32 [3 (q, k, v)][H][d][4], 16-byte aligned: each
                            of q, k, v first passes through a causal depthwise
                            convolution of width 4 over the tokens of its
                            sequence (tap 0 weighs the row 3 tokens back, tap 3
                            the token's own row), then Swish x * sigmoid(x);
                            q and k are L2-normalised after that            */
  void* conv_state;      /* with conv_weight: the raw q, k, v rows of the 3
                            tokens before each sequence, [N][3 (q, k, v)][3
                            (oldest first)][H][d] (dtype), 16-byte aligned;
                            NULL = zeros.  kda_prefill only reads it (after a
                            prefill, the next window is the last 3 raw rows
                            of the sequence); kda_decode_step reads it and
                            writes the window that ends with this token      */
} kda_options;

/* Fill *opt with the defaults listed above. */
void kda_options_init(kda_options* opt);

/*
 * kda_prefill -- chunkwise-parallel prefill over packed sequences.
 *
 * The chunked form reaches the same result as the token recurrence above
 * (parallel inside a chunk, recurrent across chunks: "Kimi K3", section
 * "Forgetting different features at different rates"; "Kimi K3's hybrid
 * block", section "From linear attention to the delta rule").
 *
 *   q, k        [T_total][H][d_k]  dtype
 *   v           [T_total][H][d_v]  dtype
 *   log_alpha   [T_total][H][d_k]  fp32 (clamped to [g_min, 0] inside);
 *               [T_total][H] with KDA_DECAY_HEAD, unused with KDA_DECAY_NONE
 *   beta        [T_total][H]       dtype
 *   S0          [N][H][d_k][d_v]   fp32 initial states, NULL = zeros
 *   cu_seqlens  [N+1] int32 on the device, cu_seqlens[0] = 0,
 *               non-decreasing, cu_seqlens[N] = T_total.  NULL = N sequences
 *               of T_total/N tokens each.  Zero-length sequences are allowed
 *               and return S_T = S0.  The values are not checked on the host
 *               (they live on the device); opt->max_seqlen must bound them.
 *   o           [T_total][H][d_v]  dtype out (y when opt->gate is set)
 *   S_T         [N][H][d_k][d_v]   fp32 final states out (may alias S0)
 *   The token arrays may be NULL when T_total == 0 (then S_T = S0).
 *
 * The tensor-core path needs opt->workspace of kda_prefill_workspace_size()
 * bytes (KDA_ERR_WORKSPACE otherwise); the SIMT path needs none.
 */
int kda_prefill(const void* q, const void* k, const void* v, const float* log_alpha,
                const void* beta, const float* S0, const int32_t* cu_seqlens, int N,
                void* o, float* S_T, int T_total, int H, int d_k, int d_v, int dtype,
                const kda_options* opt, kda_stream_t stream);

/* Bytes of device workspace kda_prefill needs for these sizes and options
 * (0 when the selected path needs none). */
size_t kda_prefill_workspace_size(int T_total, int N, int H, int d_k, int d_v,
                                  const kda_options* opt);

/*
 * The implementation kda_prefill runs for these sizes and options: returns
 * KDA_IMPL_SIMT or KDA_IMPL_TC (> 0), or a negative status if kda_prefill
 * would reject them.  *launches (if not NULL) receives the number of kernels
 * one call enqueues with cu_seqlens (the tensor-core path enqueues one fewer
 * for equal-length sequences, cu_seqlens NULL: it needs no chunk-base prefix
 * sum, and the first phase_events interval is then empty), *chunk (if not
 * NULL) the chunk length it uses.
 */
int kda_prefill_path(int T_total, int N, int H, int d_k, int d_v, int dtype,
                     const kda_options* opt, int* launches, int* chunk);

/*
 * kda_decode_step -- one recurrent token for N independent sequences, with the
 * state updated in place ("Kimi K3, explained", section "Kimi Delta Attention:
 * making the radical option work": k and v update S(t-1), q reads S(t)).
 *
 *   q, k        [N][H][d_k]  dtype
 *   v           [N][H][d_v]  dtype
 *   log_alpha   [N][H][d_k]  fp32
 *   beta        [N][H]       dtype
 *   S           [N][H][d_k][d_v] fp32, read and overwritten
 *   o           [N][H][d_v]  dtype out (y when opt->gate is set; gate [N][H][d_v])
 * Each state is read once and written once.
 */
int kda_decode_step(const void* q, const void* k, const void* v, const float* log_alpha,
                    const void* beta, float* S, void* o, int N, int H, int d_k, int d_v,
                    int dtype, const kda_options* opt, kda_stream_t stream);

/*
 * kda_gated_rmsnorm -- per-head RMSNorm times a sigmoid gate ("Kimi K3's
 * hybrid block", section "From linear attention to the delta rule": the
 * output is RMSNorm'd per head and multiplied by a full-rank sigmoid gate).
 *
 *   o, y  [rows][H][d_v] dtype (y may alias o);  gate [rows][H][d_v] dtype;
 *   w     [d_v] fp32 or NULL (= ones).
 *   y = o / sqrt(mean_j o_j^2 + eps) * w * sigmoid(gate)
 */
int kda_gated_rmsnorm(const void* o, const void* gate, const float* w, void* y, int rows,
                      int H, int d_v, float eps, int dtype, kda_stream_t stream);

/*
 * kda_prefill_noalloc -- the same prefill as kda_prefill on the tensor-core
 * path, for callers that cannot allocate device memory: for example host code
 * that must never call cudaMalloc while it serves requests (an allocation can
 * synchronise the device or fail half way through a step), or runtimes that
 * own every device byte through their own pool and forbid raw allocations.
 * The pages have no counterpart; it is a convenience of this library.
 *
 * Arguments, layouts and results are those of kda_prefill, except that
 * opt->workspace is ignored: the scratch is a fixed array of
 * KDA_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that loads
 * it until the process exits.  Errors, all returned before anything is
 * launched:
 *   - the argument checks of kda_prefill come first, with its status codes
 *     (KDA_ERR_ARG, _SHAPE, _DTYPE, _ALIGN, ...);
 *   - KDA_ERR_UNSUPPORTED for anything the tensor-core path does not take:
 *     opt->impl other than KDA_IMPL_AUTO / KDA_IMPL_TC, opt->chunk other than
 *     0 / 64, fp32 data, or d_k = d_v other than 128;
 *   - KDA_ERR_WORKSPACE for sizes whose scratch (kda_prefill_workspace_size)
 *     exceeds the array.
 * Nothing is allocated.
 *
 * The first call on a device looks up the array's device address (again after
 * the device's context is replaced, e.g. by a device reset, since the array
 * then lives at a new address); make that first call before any stream
 * capture.  All calls share the one array, so calls that can overlap on the
 * GPU (different streams, or other threads) race: order them, e.g. on one
 * stream.  No state carries over between calls.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u << 20)
int kda_prefill_noalloc(const void* q, const void* k, const void* v, const float* log_alpha,
                        const void* beta, const float* S0, const int32_t* cu_seqlens, int N,
                        void* o, float* S_T, int T_total, int H, int d_k, int d_v, int dtype,
                        const kda_options* opt, kda_stream_t stream);

/*
 * Synchronise `stream`, then return and clear the device status word of the
 * current device: KDA_OK, KDA_ERR_TIMEOUT (a bounded device wait gave up),
 * KDA_ERR_SHAPE (a kernel found cu_seqlens out of range and skipped that
 * sequence), or KDA_ERR_CUDA if the stream itself reports an error.
 */
int kda_get_last_error(kda_stream_t stream);

/* Static English text for a status code. */
const char* kda_status_string(int status);

/* ABI version of this header (bumped on any incompatible change). */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
