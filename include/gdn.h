/*
 * gdn.h -- C ABI of the KDA / Gated DeltaNet step on NVIDIA GB300 (sm_103a).
 *
 * The step (per sequence b, per token t, per value head h), as stated in
 * "Thirty tiny kernels per layer" (the decode-step list and the pure step
 * function) and in the delta-rule definition of Kimi Delta Attention /
 * Gated DeltaNet:
 *   1. X = [conv_state[b] (K-1 rows, oldest first); qkv[b,t]];
 *      xhat[c] = silu(sum_j conv_w[c][j] * X[j][c]); conv_state[b] = X[1..K-1]
 *   2. q, k, v = split(xhat) (channel order: q of every qk head, k of every qk
 *      head, v of every value head); q <- q * q_scale / sqrt(|q|^2 + eps_l2),
 *      k <- k / sqrt(|k|^2 + eps_l2).  Value head h reads qk head h / (H_v/H_qk).
 *   3. g = -exp(A_log[h]) * softplus(f + dt_bias)  (per key channel for
 *      GDN_GATE_PER_CHANNEL, one per head for GDN_GATE_PER_HEAD), or
 *      g = dt_bias[h] * sigmoid(-A_log[h] * f) per key channel for
 *      GDN_GATE_LOWER_BOUND (the GLM KDA's bounded "safe" decay, "llama.cpp
 *      PR #84", the KDA decay precompute); alpha = exp(g)
 *   4. beta = sigmoid(beta_logit)
 *   5. S <- (I - beta k k^T) Diag(alpha) S + beta k v^T     (S is [d_k, d_v], fp32)
 *   6. o = S^T q
 *   7. y = o / sqrt(mean(o^2) + eps_norm) * norm_w * silu(z), or * sigmoid(z)
 *      with GDN_FLAG_SIGMOID_GATE (the GLM KDA's output gate, "llama.cpp PR #84",
 *      the gated-norm fusion)
 *
 * Ownership: the caller owns every buffer.  The library allocates nothing,
 * keeps no state between calls, makes no host<->device copy and never
 * synchronises: work is queued on `stream` in stream order.  Every pointer is
 * a device pointer.  state, state_hist, conv_w and out must be 16-byte
 * aligned; every other pointer must be aligned to its element size.
 *
 * Errors: argument and shape errors return a negative status before anything
 * is launched.  A failed launch returns GDN_ERR_CUDA (the CUDA error is left
 * for cudaGetLastError).  Faults inside a kernel surface at the caller's next
 * synchronisation.  There is no CPU fallback: a shape without a GPU kernel
 * returns GDN_ERR_UNSUPPORTED.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = -1,        /* a required pointer is NULL                       */
    GDN_ERR_ALIGN = -2,       /* a pointer is misaligned (see Ownership)         */
    GDN_ERR_SHAPE = -3,       /* sizes are negative, inconsistent or out of range */
    GDN_ERR_UNSUPPORTED = -4, /* valid, but no kernel instance for these sizes    */
    GDN_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required       */
    GDN_ERR_CUDA = -6,        /* the CUDA runtime refused a launch                */
    GDN_ERR_TIMEOUT = -7      /* a bounded device wait gave up (gdn_device_status) */
} gdn_status_t;

typedef enum {
    GDN_GATE_PER_HEAD = 0,    /* Gated DeltaNet: f [B,T,H_v],     dt_bias [H_v]     */
    GDN_GATE_PER_CHANNEL = 1, /* KDA:            f [B,T,H_v,d_k], dt_bias [H_v,d_k] */
    GDN_GATE_LOWER_BOUND = 2  /* KDA, bounded:   f [B,T,H_v,d_k]; A_log [H_v] holds
                                 the scale a (used as is), dt_bias [H_v] the bound
                                 lb <= 0 of the log-decay                          */
} gdn_gate_mode_t;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype_t;

/* Launch flags (gdn_shape_t.flags). */
enum {
    /*
     * Launch with programmatic dependent launch: the kernel reads `state`,
     * `conv_state` and the parameters before it waits for the previous kernel
     * on the stream, and lets the next kernel start once its own wait has
     * returned.  The caller asserts that the kernel queued just before this
     * call on the stream does not write `state`, `conv_state` or the
     * parameters (for example, the previous layer of a model).  If that kernel
     * lets its dependents start before its own dependency wait, the same must
     * hold for the kernels before it that may still be running.  This
     * library's kernels let their dependents start only after their own wait,
     * so a chain of its calls needs the promise for the immediately preceding
     * call alone.  Inputs q/k/v/f/beta/z are read after the wait.  Without
     * this flag launches are plain stream-ordered.
     */
    GDN_FLAG_PDL = 1,
    /* Output gate sigmoid(z) in place of silu(z). */
    GDN_FLAG_SIGMOID_GATE = 2
};

typedef struct {
    int32_t B;          /* sequences                                              */
    int32_t T;          /* tokens per sequence in this call                       */
    int32_t H_qk;       /* query/key heads                                        */
    int32_t H_v;        /* value heads, a multiple of H_qk                        */
    int32_t d_k;        /* key width (state rows)                                 */
    int32_t d_v;        /* value width (state columns)                            */
    int32_t conv_K;     /* conv taps; conv_state keeps conv_K - 1 rows            */
    int32_t chunk;      /* chunk length of gdn_prefill_chunked (64)               */
    int32_t gate_mode;  /* gdn_gate_mode_t                                        */
    int32_t in_dtype;   /* gdn_dtype_t of qkv, f, beta, z                         */
    int32_t out_dtype;  /* gdn_dtype_t of out                                     */
    int32_t flags;      /* GDN_FLAG_*                                             */
    float q_scale;      /* d_k^-1/2 rounded to fp32 by the caller                 */
    float eps_l2;       /* epsilon of the q/k L2 norm                             */
    float eps_norm;     /* epsilon of the gated RMSNorm                           */
} gdn_shape_t;

/*
 * Tensors, all row-major and contiguous.  C = 2*H_qk*d_k + H_v*d_v.
 */
typedef struct {
    const void *qkv;       /* [B,T,C] in_dtype: pre-conv q|k|v rows               */
    const void *f;         /* [B,T,H_v,d_k] or [B,T,H_v] in_dtype: gate logits    */
    const void *beta;      /* [B,T,H_v] in_dtype: beta logits                     */
    const void *z;         /* [B,T,H_v,d_v] in_dtype: output-gate rows            */
    const float *conv_w;   /* [C,conv_K]                                          */
    const float *A_log;    /* [H_v]                                               */
    const float *dt_bias;  /* [H_v,d_k] or [H_v]                                  */
    const float *norm_w;   /* [d_v]                                               */
    float *conv_state;     /* [B,conv_K-1,C], oldest row first                    */
    float *state;          /* [B,H_v,d_k,d_v]; row = key channel                  */
    void *out;             /* [B,T,H_v*d_v] out_dtype                             */
    float *state_hist;     /* verify: [T,B,H_v,d_k,d_v]; prefill: [min(T,4),B,H_v,d_k,d_v]
                              (snapshot tails); or NULL; unused elsewhere        */
    float *conv_hist;      /* verify: [T,B,conv_K-1,C]; prefill: [min(T,4),B,conv_K-1,C];
                              or NULL; unused elsewhere                          */
} gdn_tensors_t;

/*
 * One decode step (T must be 1): steps 1-7 for every sequence and value head.
 * conv_state and state are advanced in place; out receives y.
 * Kernel instances: d_k == d_v in {16, 32, 64, 128}, conv_K == 4.
 */
GDN_API gdn_status_t gdn_decode_step(const gdn_shape_t *shape, const gdn_tensors_t *t,
                             gdn_stream_t stream);

/*
 * Multi-token verify (1 <= T <= 4): steps 1-7 for tokens 0..T-1 in order, as T
 * decode steps would (the arithmetic per token is the decode step's, so the
 * outputs and per-token states equal T gdn_decode_step calls bit for bit).
 * state and conv_state are only read.  state_hist[t], when not NULL, receives
 * the state after token t; conv_hist[t], when not NULL, the conv window after
 * token t.  With both NULL only out is written (the state is read once).  To
 * commit k accepted tokens the caller either adopts state_hist[k-1] and
 * conv_hist[k-1] or calls gdn_commit_accepted ("opus_gdn_qsa" audit, the
 * gdn_step commit / verify modes and history output).
 */
GDN_API gdn_status_t gdn_verify_T(const gdn_shape_t *shape, const gdn_tensors_t *t,
                          gdn_stream_t stream);

/*
 * In-place commit of accepted tokens (1 <= T <= 4 rows per sequence in
 * qkv/f/beta/z): sequence b takes its first accepted[b] tokens (clamped to
 * 0..T; accepted == NULL takes all T) through steps 1-7, and state and
 * conv_state are advanced in place to the state and window after them -- the
 * values verify would have written to state_hist[k-1] and conv_hist[k-1], bit
 * for bit, and k = 0 leaves the sequence untouched.  out may be NULL; when it
 * is not, the rows of the taken tokens receive y and the other rows are left
 * alone.  state_hist and conv_hist are ignored.  accepted is a device array
 * of B int32 read by the kernel after its dependency wait, so the kernel
 * queued before this call may write it ("opus_gdn_qsa" audit, the gdn_step
 * commit modes: commit all, none, or the first k tokens).
 */
GDN_API gdn_status_t gdn_commit_accepted(const gdn_shape_t *shape, const gdn_tensors_t *t,
                                 const int32_t *accepted, gdn_stream_t stream);

/*
 * Chunked prefill of T >= 1 tokens per sequence: the same result as T decode
 * steps, computed in the chunked WY/UT form ("llama.cpp PR #84", chunked
 * KDA prefill).  conv_state and state are advanced in place; out receives y
 * for every token.  Kernels, by shape (shape->chunk must be > 0):
 *   - per-head decay, bf16 rows, d = 128, chunk == 64: one tensor-core kernel
 *     in 64-token chunks, every dense product on tcgen05, no workspace;
 *   - the same with chunk == 32: one tensor-core kernel in 32-token chunks;
 *   - any other shape with d = 128 and T > 4 (per-channel decay, fp32 rows,
 *     other chunk lengths): the two-kernel form, an intra-chunk pass over all
 *     16-token chunks into the workspace, then a tcgen05 state pass;
 *   - everything else: the recurrent step kernel.
 * workspace must hold gdn_prefill_workspace_bytes(shape) bytes, 16-byte aligned
 * (may be 0 bytes; then NULL is accepted); the call owns it until the work
 * queued on `stream` completes.
 *
 * Snapshot tails ("llama.cpp PR #84", the chunked prefill's snapshot slots):
 * when state_hist or conv_hist is not NULL, the first T - n tokens (n =
 * min(T, 4)) run as above and the last n on the recurrent step kernel from the
 * state and window they leave; state_hist[k] ([n,B,H_v,d_k,d_v], 16-byte
 * aligned) then receives the state after token T - n + k and conv_hist[k]
 * ([n,B,conv_K-1,C]) the conv window after it, so index n - 1 holds the final
 * state and window (also left in state and conv_state).  A caller rolls back
 * to any of the last n tokens by adopting those entries.
 */
GDN_API gdn_status_t gdn_prefill_chunked(const gdn_shape_t *shape, const gdn_tensors_t *t,
                                 void *workspace, size_t workspace_bytes,
                                 gdn_stream_t stream);

/* Bytes of device workspace gdn_prefill_chunked needs for this shape (0 on a bad shape). */
GDN_API size_t gdn_prefill_workspace_bytes(const gdn_shape_t *shape);

/* Bytes of the scratch gdn_prefill_chunked_static uses in place of a workspace. */
#define GDN_PREFILL_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * gdn_prefill_chunked with no workspace argument, for callers that cannot
 * allocate device memory around the call: a C host with no device allocator
 * of its own, or a serving loop in which a cudaMalloc (which synchronises the
 * device) would stall the work queued on its other streams.
 *
 * The scratch is one static device array of GDN_PREFILL_STATIC_SCRATCH_BYTES
 * per device, reserved when the library's module loads in the device's context
 * (with lazy module loading, at the first call on that device).  The first call
 * on a device, and the first after its context was destroyed and made again
 * (cudaDeviceReset), looks up the array's device address and keeps it with the
 * context; make that first call before any stream capture.  The call allocates
 * and frees nothing.  A shape whose
 * gdn_prefill_workspace_bytes exceeds the scratch returns GDN_ERR_WORKSPACE
 * before anything is queued (one sequence of 32 heads fits 480 tokens).
 * Nothing in the scratch has to start at zero: the first kernel writes every
 * word the second one uses.
 *
 * Every call on a device shares that one scratch.  Two calls whose work
 * overlaps in time (on different streams, or from different host threads
 * without ordering) race on it and produce wrong results; calls queued on one
 * stream run in order and are safe.  Arguments, results and the other errors
 * are those of gdn_prefill_chunked.  The pages describe no such entry point;
 * it is a deployment convenience around the same kernels.
 */
GDN_API gdn_status_t gdn_prefill_chunked_static(const gdn_shape_t *shape, const gdn_tensors_t *t,
                                        gdn_stream_t stream);

/*
 * Weights of one KDA layer's projections, all bf16, row-major, 16-byte
 * aligned.  C = 2*H_qk*d_k + H_v*d_v as for qkv.
 */
typedef struct {
    int32_t d_model;     /* width of the layer input x and output x_out (% 8 == 0)   */
    int32_t rank;        /* width of the low-rank gate chains (% 8 == 0)             */
    const void *w_qkv;   /* [C][d_model]: q of every qk head, k, then v rows          */
    const void *w_fa;    /* [rank][d_model]: f_a                                      */
    const void *w_fb;    /* [H_v*d_k][rank]: f_b, the per-channel gate logits         */
    const void *w_ga;    /* [rank][d_model]: g_a                                      */
    const void *w_gb;    /* [H_v*d_v][rank]: g_b, the output-gate rows z              */
    const void *w_beta;  /* [H_v][d_model]: beta logits                               */
    const void *w_o;     /* [d_model][H_v*d_v]: output projection                     */
} gdn_layer_weights_t;

/*
 * One decode step of a whole KDA layer for B sequences (T = 1): the
 * projections around the step fused into three or four launches.  From the
 * layer input x ([B][d_model] bf16, 16-byte aligned):
 *   qkv = x w_qkv^T, f_a = x w_fa^T, g_a = x w_ga^T, beta = x w_beta^T   (one launch)
 *   f = f_a w_fb^T, z = g_a w_gb^T              (one launch, or inside the step when
 *                                                the step runs on the column-slab kernel)
 *   the step of gdn_decode_step on those rows                            (the step)
 *   x_out = y w_o^T                                                      (one launch)
 * "Thirty tiny kernels per layer" (the decode budget: these projections are
 * ~90% of a KDA layer's decode time, as weight streaming) and "llama.cpp PR
 * #84" (f_a with g_a and beta, f_b with g_b, as single launches) describe the
 * chain.  Activations stay fp32 between the launches: t->qkv, f, beta, z and out
 * are caller scratch in the step's layouts with shape->in_dtype and
 * shape->out_dtype GDN_F32, 16-byte aligned; conv_w, A_log, dt_bias, norm_w,
 * conv_state and state are the step's.  gate_mode must be a per-channel gate.
 * workspace holds gdn_layer_workspace_bytes bytes (the low-rank rows),
 * 16-byte aligned.  x_out is [B][d_model] fp32.
 *
 * The launches use programmatic dependent launch whatever shape->flags
 * holds: each kernel reads activations and writes its outputs only after the
 * previous kernel on the stream has completed, and before that touches nothing
 * but read-only weights (asked into L2) and, for the step, its own state,
 * window and parameters.  The first projection therefore needs no promise from
 * the caller about the kernel before it.
 */
GDN_API gdn_status_t gdn_layer_decode(const gdn_shape_t *shape, const gdn_layer_weights_t *w,
                              const void *x, float *x_out, const gdn_tensors_t *t,
                              void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Bytes of workspace gdn_layer_decode needs (0 on bad arguments). */
GDN_API size_t gdn_layer_workspace_bytes(const gdn_shape_t *shape, const gdn_layer_weights_t *w);

/*
 * Reads and clears the library's device error word on the current device.
 * Kernels that wait on an mbarrier give up after about two seconds instead of
 * hanging and record the time-out there; their outputs are then invalid.
 * Returns GDN_OK, GDN_ERR_TIMEOUT, or GDN_ERR_CUDA if the word could not be
 * read.  Synchronises with the current device (a debugging aid, not for the
 * hot path).
 */
GDN_API gdn_status_t gdn_device_status(void);

/* Static, NUL-terminated name of a status code. */
GDN_API const char *gdn_status_string(gdn_status_t status);

/*
 * Name of the kernel variant a call with this shape would launch for `op`
 * (0 decode, 1 verify, 2 prefill), e.g. "step<128,16>" (d = 128, 16-column slabs).  Lets tests check that
 * the intended fast path runs.  Returns NULL for an unsupported shape.
 */
GDN_API const char *gdn_kernel_variant(const gdn_shape_t *shape, int op);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
