/*
 * la_chunked.h -- C ABI of the chunkwise-parallel causal linear attention forward pass
 * (GB300, sm_103a).  Library: chunkwise_causal_linear_gb300/liblachunked.so.
 *
 * What is computed (per (b, h) head, rows t = 0..L-1, phi applied row-wise):
 *
 *     num_t = sum_{s <= t} M[t,s] (phi(q_t) . phi(k_s)) v_s
 *     den_t = sum_{s <= t} M[t,s] (phi(q_t) . phi(k_s))
 *     out_t = normalize ? num_t / den_t : num_t
 *
 * with M[t,s] = 1 (causal linear attention), or M[t,s] = lambda_t^(l(t,s)),
 * l = 0 if s == t else 1 + floor(log2(t XOR s)) (Fenwick-level log-linear mask).
 *
 * Sources:
 *   "attention と線形の間" (sharin-2a1.pages.dev, parts/chunked.html), section 2:
 *       Chunked(q, k, v, c) -- chunks of c rows; inside a chunk the causally masked
 *       scores (diagonal kept), across chunks a d_k x d_v state carried forward;
 *       c <= 0 means 1; a partial last chunk is allowed.  Section 3: Shape cost model.
 *   "Linear Attention / Performerの理論と実装" (disassemble-channel.com): the ELU
 *       feature map, FAVOR+ positive random features, the normalised output y_t and the
 *       (S_t, z_t) recurrence.
 *   "論文紹介：Log Linear Attention" (docswell slides): Fenwick buckets (slides 15-21),
 *       level weights lambda (slide 17), chunkwise level-0 block plus per-level
 *       inter-chunk states (slides 34-35).
 *
 * Conventions for every entry point:
 *   - Layout: q, k [B, H, L, dk]; v, out [B, H, L, dv]; contiguous row-major.
 *   - All tensor pointers are DEVICE pointers unless the name says _host.  The caller
 *     owns every buffer; the library allocates no device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream) and return after the launches are queued.
 *   - Host-detectable errors return a negative la_status before anything is launched.
 *     Errors found on the device (a bounded wait that timed out, an index check) are
 *     recorded in a device error word that la_last_device_status() reads.
 *   - Concurrent calls on different streams are safe if they use different workspaces
 *     (the device error word is shared by all calls).
 */
#ifndef LA_CHUNKED_H
#define LA_CHUNKED_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------- */
enum la_status {
    LA_OK = 0,
    LA_ERR_NULL = -1,        /* a required pointer is NULL                               */
    LA_ERR_SHAPE = -2,       /* a dimension is <= 0, or sizes overflow                   */
    LA_ERR_UNSUPPORTED = -3, /* combination not supported (dtype, dims, feature map, C)  */
    LA_ERR_WORKSPACE = -4,   /* workspace missing or smaller than la_chunked_workspace_bytes */
    LA_ERR_CUDA = -5,        /* a CUDA runtime call failed (launch, copy, attribute)      */
    LA_ERR_TIMEOUT = -6,     /* device: a bounded wait gave up (read via la_last_device_status) */
    LA_ERR_DEVICE = -7,      /* device: an index or shape check failed inside a kernel    */
    LA_ERR_SCRATCH_LIMIT = -8, /* la_chunked_fwd_noalloc: the problem needs more scratch than
                                  its fixed buffer holds (8 MiB)                          */
    LA_ERR_ARG = -9            /* an argument value is out of range (la_decay_*: gamma)    */
};

/* ---- feature maps phi -------------------------------------------------------------- */
enum la_fm_kind {
    LA_FM_IDENTITY = 0, /* phi(x) = x                                                     */
    LA_FM_ELU1 = 1,     /* phi(x) = elu(x) + 1 = (x >= 0 ? x + 1 : e^x)                   */
    LA_FM_FAVOR = 2     /* FAVOR+: x^ = x / dk^(1/4); phi(x) = exp(omega x^ - |x^|^2/2)/sqrt(m) */
};

typedef struct la_feature_map {
    int kind;            /* enum la_fm_kind                                              */
    int m;               /* FAVOR+: number of random features (the feature dimension);
                            other kinds: ignored (the feature dimension is dk)            */
    const float *omega;  /* FAVOR+: device [m, dk] fp32 row-major random matrix, owned by
                            the caller and read during the call; other kinds: ignored     */
} la_feature_map;

/* ---- storage dtypes of q, k, v, out ---------------------------------------------- */
enum la_dtype {
    LA_BF16 = 0,  /* bfloat16 storage; arithmetic in fp32 with bf16 tensor-core operands  */
    LA_F32 = 1    /* fp32 storage; arithmetic in fp32 (exact on small-integer inputs)     */
};

/* ---- execution paths ---------------------------------------------------------------- */
enum la_path {
    LA_PATH_AUTO = 0,    /* the library picks (see la_chunked_plan)                       */
    LA_PATH_SIMT = 1,    /* generic fp32 CUDA-core path: any C, any supported dims         */
    LA_PATH_TC = 2       /* tcgen05/TMEM tensor-core single-pass path (subset of shapes)   */
};

/*
 * la_chunked_fwd -- the forward pass.
 *
 *   q, k          device [B, H, L, dk], dtype `dtype`
 *   v             device [B, H, L, dv], dtype `dtype`
 *   out           device [B, H, L, dv], dtype `dtype`; fully overwritten
 *   C             chunk size: C <= 0 means 1, C >= L means one chunk ("attention and
 *                 linear order meet at the two ends", chunked page section 2)
 *   feature_map   NULL means identity
 *   normalize     0: out = num; 1: out = num / den
 *   level_weights NULL, or device [B, H, L, num_levels] fp32 lambda_t^(l) (log-linear).
 *                 num_levels must cover 1 + ceil(log2 L) levels, and with more than one
 *                 chunk C must be a power of two (chunk edges are then Fenwick edges).
 *   workspace     device scratch of at least la_chunked_workspace_bytes(...) bytes (may
 *                 be NULL when that is 0); contents on entry are ignored.
 *   stream        cudaStream_t as void*.
 * Returns LA_OK or a negative la_status (nothing launched on error).
 */
int la_chunked_fwd(const void *q, const void *k, const void *v, void *out,
                   int B, int H, int L, int dk, int dv, int C,
                   const la_feature_map *feature_map, int normalize,
                   const float *level_weights, int num_levels,
                   int dtype, void *workspace, size_t workspace_bytes, void *stream);

/* As la_chunked_fwd, with an explicit execution path (enum la_path).  LA_PATH_TC returns
 * LA_ERR_UNSUPPORTED for shapes the tensor-core path does not cover.  It covers bf16
 * storage, L >= 128, and:
 *   - identity / elu+1 features, with or without the normaliser, dk = D, (dk, dv) in
 *     {(64, 64), (64, 128), (128, 128)}, C in {16, 32, 64, 128, 256};
 *   - FAVOR+ features, dk = 64, m = 256, dv = 64, C = 64, with or without the normaliser;
 *   - the log-linear mask: identity features, no normaliser, dk = dv = 64, C = 64, at most
 *     4096 chunks, num_levels <= 32, L * num_levels a multiple of 4 and level_weights
 *     16-byte aligned (LA_PATH_AUTO falls back to LA_PATH_SIMT when it is not).
 * Few-head problems are split along the sequence into segments; their plan reports two
 * launches and a workspace for the segment totals. */
int la_chunked_fwd_path(const void *q, const void *k, const void *v, void *out,
                        int B, int H, int L, int dk, int dv, int C,
                        const la_feature_map *feature_map, int normalize,
                        const float *level_weights, int num_levels,
                        int dtype, void *workspace, size_t workspace_bytes, void *stream,
                        int path);

/*
 * la_chunked_fwd_host -- the same forward pass from HOST buffers: copies q, k, v (and
 * nothing else: omega and level_weights stay device pointers) from host memory into the
 * caller's device buffers q_dev, k_dev, v_dev, runs la_chunked_fwd on them into out_dev,
 * copies out_dev back into out_host.  Host buffers should be pinned (cudaHostAlloc /
 * page-locked) for the copies to be asynchronous; the host buffers must stay valid until
 * the stream reaches the end of the call.  Sizes and error behaviour as la_chunked_fwd.
 * When the plan is one unsplit launch and the step moves at least 64 MB, the call runs as a
 * pipeline over up to 8 groups of heads: copies in on one internal stream, the groups'
 * launches on `stream`, copies out on another internal stream, so the two copy directions
 * and the compute overlap.  Each head's arithmetic is that of la_chunked_fwd (identical
 * outputs).  Either way the work is ordered after what `stream` already holds, and `stream`
 * reaches the end of the call only after every copy.
 */
int la_chunked_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                        void *out_host, void *q_dev, void *k_dev, void *v_dev, void *out_dev,
                        int B, int H, int L, int dk, int dv, int C,
                        const la_feature_map *feature_map, int normalize,
                        const float *level_weights, int num_levels,
                        int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * la_chunked_fwd_noalloc -- the same forward pass, for callers that cannot allocate device
 * memory (code running inside an allocator or a memory-pool callback, plugins whose host
 * application owns every device allocation, real-time loops that must never call
 * cudaMalloc / cudaFree).  No counterpart on the pages: it is a deployment variant.
 *
 * It allocates nothing.  Every problem whose la_chunked_workspace_bytes is nonzero takes
 * that scratch from a fixed 8 MiB array compiled into the library: the segment totals of a
 * sequence cut into segments (few heads, on the tensor-core paths), and the log-linear
 * mask's per-level chunk states.  Every GPU that loads the library holds those 8 MiB until
 * the process exits.  Problems that need more return LA_ERR_SCRATCH_LIMIT before anything
 * is launched (la_chunked_workspace_bytes tells how much a problem needs).
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.  The address is kept for
 *     the life of the process: calls after cudaDeviceReset of that device are not
 *     supported.
 *   - All calls share the one array and it keeps the last call's contents; the kernel
 *     clears what it needs at the start of every call.  Calls that may overlap on the GPU
 *     (different streams, or different host threads) race on it: serialise them.
 * Arguments, layout and the other errors are those of la_chunked_fwd (no workspace).
 */
int la_chunked_fwd_noalloc(const void *q, const void *k, const void *v, void *out,
                           int B, int H, int L, int dk, int dv, int C,
                           const la_feature_map *feature_map, int normalize,
                           const float *level_weights, int num_levels,
                           int dtype, void *stream);

/* Bytes of device workspace la_chunked_fwd needs for this problem on the current device
 * (0 when none).  Returns 0 also for invalid arguments (la_chunked_fwd reports those). */
size_t la_chunked_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                  const la_feature_map *feature_map, int normalize,
                                  int num_levels, int dtype);

/* ---- plan introspection (host only; no device call when num_sms > 0) --------------- */
typedef struct la_plan_info {
    int path;              /* enum la_path actually chosen                               */
    int chunk;             /* effective chunk size after clamping                         */
    int n_chunks;          /* ceil(L / chunk)                                             */
    int feature_dim;       /* D: dk, or m for FAVOR+                                      */
    int grid_x, grid_y;    /* main kernel grid                                            */
    int block;             /* threads per CTA of the main kernel                          */
    int smem_bytes;        /* dynamic shared memory per CTA of the main kernel            */
    int n_launches;        /* kernel launches per call                                    */
    size_t workspace_bytes;
} la_plan_info;

/* Fills *info with the plan for the problem as la_chunked_fwd_path(path) would run it.
 * num_sms: SM count to plan for (0 = query the current device).  Returns LA_OK or the
 * status la_chunked_fwd_path would return for these arguments (pointers are not
 * checked). */
int la_chunked_plan(int B, int H, int L, int dk, int dv, int C,
                    const la_feature_map *feature_map, int normalize, int loglinear,
                    int num_levels, int dtype, int path, int num_sms, la_plan_info *info);

/* Waits for `stream`, then returns and clears the device error word: LA_OK, or the
 * first device-side error (LA_ERR_TIMEOUT, LA_ERR_DEVICE) recorded since the last call,
 * or LA_ERR_CUDA if the stream itself reports an error. */
int la_last_device_status(void *stream);

/* Static description of a status code (never NULL). */
const char *la_status_string(int status);

/*
 * la_cost_model -- "attention と線形の間", section 3, Shape{L, D, C}: multiply-add counts
 * of the chunked order.  *state_macs = 2 L D^2 (writing and reading the D x D state, the
 * same for every C); *score_macs = 2 L C D (making the in-chunk scores and mixing the
 * values, proportional to C).  Either output pointer may be NULL.  Returns LA_OK, or
 * LA_ERR_SHAPE for negative sizes.
 */
int la_cost_model(long long L, long long D, long long C, long long *state_macs,
                  long long *score_macs);

/*
 * la_decode_step -- one step of the recurrent (decoding) form for every (b, h) head, the
 * inference counterpart of the chunked state ("Linear Attention / Performerの理論と実装",
 * "再帰的な状態更新"; "論文紹介：Log Linear Attention", slides 17-22 for the level weights).
 *
 *   q, k          device [B, H, dk] (this token), dtype `dtype`
 *   v, out        device [B, H, dv], dtype `dtype`; out is overwritten
 *   state         device fp32, read and updated in place.  Without level weights:
 *                 [B, H, D, dv] = S, the sum of phi(k_s) v_s^T over the tokens so far.
 *                 With level weights: [B, H, num_levels - 1, D, dv], the Fenwick level
 *                 states S^(1), S^(2), ... (zeros before the first token).
 *   zstate        device fp32 normaliser, [B, H, D] or [B, H, num_levels - 1, D]; may be
 *                 NULL when normalize is 0.  Updated in place like `state`.
 *   level_weights NULL, or device [B, H, num_levels] fp32 lambda_t^(l) of this token.
 *   t             this token's position (0-based); used by the level update only.
 * D is dk, or m for FAVOR+.  Plain: state += phi(k) v^T, z += phi(k), then
 * out = phi(q)^T state (/ phi(q)^T z).  Level weights: out = lambda^(0) (phi(q).phi(k)) v +
 * sum_{l>=1} lambda^(l) phi(q)^T S^(l) from the states before the update; then, with r =
 * trailing zeros of t+1, S^(r+1) = phi(k) v^T + sum_{l<=r} S^(l) and S^(1..r) = 0.  Stepping
 * t = 0..L-1 reproduces la_chunked_fwd's rows (the same function of the sequence).
 * Returns LA_OK, LA_ERR_NULL, LA_ERR_SHAPE (sizes, or num_levels too small for position
 * t+1: the update needs num_levels >= 2 + trailing zeros of t+1, one more level than the
 * forward pass over positions 0..t uses), LA_ERR_UNSUPPORTED, LA_ERR_CUDA.  Asynchronous on `stream`; the caller owns every
 * buffer and must not run two steps of the same state concurrently.
 */
int la_decode_step(const void *q, const void *k, const void *v, void *out, float *state,
                   float *zstate, int B, int H, int dk, int dv,
                   const la_feature_map *feature_map, int normalize,
                   const float *level_weights, int num_levels, long long t, int dtype,
                   void *stream);

/* Number of fp32 elements of la_decode_step's state and zstate for these sizes (0 on an
 * invalid combination).  num_levels = 0 means no level weights. */
long long la_decode_state_elems(int B, int H, int dk, int dv, const la_feature_map *feature_map,
                                int num_levels, long long *z_elems);

/*
 * la_noncausal_fwd -- bidirectional (non-causal) linear attention: every query sees every
 * key ("Linear Attention / Performerの理論と実装", the non-causal normalised form, and the
 * Performer's bidirectional FAVOR+ attention; "attention と線形の間" section 1, StateFirst):
 *     S = sum_s phi(k_s) v_s^T,  z = sum_s phi(k_s),  out_t = phi(q_t)^T S (/ phi(q_t)^T z).
 * Arguments as la_chunked_fwd (no chunk size, no level weights: the mask is all ones).
 * D (dk, or m for FAVOR+) must be at most 256.  The workspace holds the per-head state:
 * at least la_noncausal_workspace_bytes(...) bytes.  Returns LA_OK or a negative status
 * before any launch.
 */
int la_noncausal_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                     int dk, int dv, const la_feature_map *feature_map, int normalize, int dtype,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes la_noncausal_fwd needs (0 on an invalid or unsupported combination). */
size_t la_noncausal_workspace_bytes(int B, int H, int L, int dk, int dv,
                                    const la_feature_map *feature_map, int normalize, int dtype);

/*
 * la_decay_fwd -- causal linear attention with the Retention decay ("Linear Attention /
 * Performerの理論と実装", the section on the RNN without forgetting):
 *     S_t = gamma S_{t-1} + phi(k_t) v_t^T,        out_t = phi(q_t)^T S_t,
 * i.e. out_t = sum_{s<=t} gamma^(t-s) (phi(q_t).phi(k_s)) v_s.  With normalize the
 * normaliser decays alike, z_t = gamma z_{t-1} + phi(k_t), and out_t = phi(q_t)^T S_t /
 * phi(q_t)^T z_t (a weighted mean of the values; the page gives the update of S only).
 *   gamma   0 < gamma <= 1, one value for every head; gamma = 1 is la_chunked_fwd's result.
 *           Outside that range (or NaN): LA_ERR_ARG.
 *   path    enum la_path.  LA_PATH_TC covers bf16, identity / elu+1 features, dk = D,
 *           (dk, dv) in {(64, 64), (64, 128), (128, 128)}, C = 64, L >= 128 and
 *           gamma >= 0.5 (gamma^64 >= 2^-64); LA_PATH_AUTO takes it there and the generic
 *           fp32 path elsewhere (any C, dtype, feature map).
 * Other arguments, layouts and errors as la_chunked_fwd (no level weights).  The workspace
 * must hold la_decay_workspace_bytes(...) bytes (the few-head sequence split's totals).
 */
int la_decay_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                 int dk, int dv, int C, const la_feature_map *feature_map, int normalize,
                 float gamma, int dtype, void *workspace, size_t workspace_bytes, void *stream,
                 int path);

/* la_decode_step with the Retention decay: state = gamma state + phi(k) v^T, zstate =
 * gamma zstate + phi(k), then out = phi(q)^T state (/ phi(q)^T zstate).  Stepping t =
 * 0..L-1 from zero state reproduces la_decay_fwd's rows.  Buffers as la_decode_step without
 * level weights ([B, H, D, dv] and [B, H, D] fp32).  gamma as la_decay_fwd (LA_ERR_ARG
 * outside 0 < gamma <= 1). */
int la_decay_decode_step(const void *q, const void *k, const void *v, void *out, float *state,
                         float *zstate, int B, int H, int dk, int dv,
                         const la_feature_map *feature_map, int normalize, float gamma,
                         int dtype, void *stream);

/* Workspace bytes la_decay_fwd needs (0 when none, or on invalid arguments). */
size_t la_decay_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                const la_feature_map *feature_map, int normalize, float gamma,
                                int dtype);

/* la_chunked_plan for la_decay_fwd: the plan la_decay_fwd(path) would run. */
int la_decay_plan(int B, int H, int L, int dk, int dv, int C, const la_feature_map *feature_map,
                  int normalize, float gamma, int dtype, int path, int num_sms, la_plan_info *info);

/*
 * la_chunked_bwd -- backward pass of the causal forward (la_chunked_fwd without level
 * weights, or la_decay_fwd): given dout = dL/dout, writes dq, dk, dv.  The pages give no
 * backward formulas; these follow from the chain rule on the causal definition (mask 1 or
 * gamma^(t-s), with or without the normaliser), then through the feature map.  They are
 * linear-attention passes with the roles swapped, two of them anti-causal:
 *   - LA_PATH_TC: bf16, L >= 128, 16-byte aligned q, k, v, dout and gradient buffers, and
 *     either identity / elu+1 features with (dk, dv) in {(64, 64), (128, 128)}, no decay or
 *     gamma >= 0.5 without the normaliser (the same gamma^|t-s| mask in every pass), or
 *     FAVOR+ with dk = dv = 64, m in {128, 256, 512} and no decay.  Every pass runs on the
 *     tensor-core forward with identity features (the anti-causal ones in its anti-causal
 *     mode, in place; FAVOR+ once per 128 features); the normaliser adds three passes and
 *     its feature-gradient passes keep fp32 rows;
 *   - LA_PATH_SIMT: every supported case, in fp32 on the generic kernel;
 *   - LA_PATH_AUTO picks the first that applies.
 *   q, k, v, dout   device, as la_chunked_fwd's q, k, v and out ([B, H, L, d], dtype).
 *                   The forward output is not an input: with the normaliser, dq is a small
 *                   difference of two large sums, so the pass recomputes the output in fp32
 *                   (a bf16-stored one would carry its rounding into dq about thirtyfold).
 *   grad_q, grad_k, grad_v  device outputs dq, dk, dv: same shapes and dtype as q, k, v;
 *                   fully overwritten
 *   gamma           1 for the plain mask, else the decay (0 < gamma < 1; LA_ERR_ARG outside)
 *   C               chunk size of the generic path's passes (any value; the result does
 *                   not depend on it beyond rounding); the tensor-core passes use 64
 *   workspace       at least la_chunked_bwd_workspace_bytes(...) bytes (intermediates:
 *                   about 4 (D + dv) floats per row on the generic route, at most about
 *                   6 (D + dv) on the tensor-core route, none there for identity features
 *                   without the normaliser)
 * D (dk, or m for FAVOR+) and dk must be at most 512 and dv below 512.  Returns LA_OK or a
 * negative status before any launch.
 */
int la_chunked_bwd(const void *q, const void *k, const void *v, const void *dout,
                   void *grad_q, void *grad_k, void *grad_v, int B, int H,
                   int L, int dk, int dv, int C, const la_feature_map *feature_map,
                   int normalize, float gamma, int dtype, void *workspace,
                   size_t workspace_bytes, void *stream, int path);

/* Workspace bytes la_chunked_bwd needs (0 on an invalid or unsupported combination). */
size_t la_chunked_bwd_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                      const la_feature_map *feature_map, int normalize,
                                      int dtype);

/*
 * la_chunked_bwd_ll -- backward pass of the causal forward under the log-linear mask
 * (la_chunked_fwd with level_weights; "論文紹介：Log Linear Attention", slide 17, mask
 * M_ts = lambda_t^(l(t,s))): given dout, writes dq, dk, dv.  The level weights are treated as
 * data: their own gradient is not formed.  By the chain rule, with G_ts = M_ts (dout_t . v_s)
 * (normalised: M_ts (dout_t . v_s - dout_t . out_t) / den_t):
 *   dphi(q)_t = sum_{s<=t} G_ts phi(k_s)    -- a causal log-linear pass with the roles swapped;
 *   dphi(k)_s = sum_{t>=s} G_ts phi(q_t),   dv_s = sum_{t>=s} M_ts (phi(q_t).phi(k_s)) dout_t
 *                                            (/ den_t) -- anti-causal sums in which each pair is
 *                                            weighted by the LATER row's lambda; they are grouped
 *                                            by the aligned dyadic blocks of the level rule, one
 *                                            weighted state per block,
 * then through the feature map.  Generic fp32 route (path LA_PATH_AUTO or LA_PATH_SIMT;
 * LA_PATH_TC returns LA_ERR_UNSUPPORTED), any feature map, with or without the normaliser.
 *   level_weights  device [B, H, L, num_levels] fp32, as la_chunked_fwd's (1 + ceil(log2 L)
 *                  levels at least)
 *   C              ignored beyond la_chunked_fwd's checks (the passes use 64-row chunks)
 *   workspace      at least la_chunked_bwd_ll_workspace_bytes(...) bytes (fp32 rows of about
 *                  4 (D + dv) floats per row, level states, and one D x dv state per aligned
 *                  block of chunks per head)
 * Other arguments and errors as la_chunked_bwd (no decay).
 */
int la_chunked_bwd_ll(const void *q, const void *k, const void *v, const void *dout,
                      void *grad_q, void *grad_k, void *grad_v, int B, int H, int L, int dk,
                      int dv, int C, const la_feature_map *feature_map, int normalize,
                      const float *level_weights, int num_levels, int dtype, void *workspace,
                      size_t workspace_bytes, void *stream, int path);

/* Workspace bytes la_chunked_bwd_ll needs (0 on an invalid or unsupported combination). */
size_t la_chunked_bwd_ll_workspace_bytes(int B, int H, int L, int dk, int dv, int C,
                                         const la_feature_map *feature_map, int normalize,
                                         int num_levels, int dtype);

/*
 * Carried state.  The state a causal pass ends with seeds a decoding loop (prefill, then
 * la_decode_step / la_decay_decode_step) or the next segment of a sequence cut into
 * segments (one per stream, thread or rank): each segment's own final state T_r, an
 * exclusive prefix P_r = gamma^len_{r-1} P_{r-1} + T_{r-1} over the earlier segments (the
 * "attention と線形の間" section 2 chunk scan at segment granularity), and the segment's pass
 * started from P_r give the same rows as one pass over the whole sequence.
 *
 * la_chunked_state -- the final state of a causal pass over k, v ([B, H, L, dk], [B, H, L,
 * dv], dtype): state[b,h,i,j] = sum_t w_t phi(k_t)_i v_t,j and zstate[b,h,i] = sum_t w_t
 * phi(k_t)_i, with w_t = 1, or gamma^(L-1-t) for the Retention decay (gamma as
 * la_decay_fwd; 1 = none).  state: device fp32 [B, H, D, dv], zstate: device fp32 [B, H, D]
 * or NULL (not computed); both fully overwritten, the la_decode_step layout.  D (dk, or m
 * for FAVOR+) at most 256; no level weights.  Generic path (fp32 accumulation).
 */
int la_chunked_state(const void *k, const void *v, float *state, float *zstate, int B, int H, int L,
                     int dk, int dv, const la_feature_map *feature_map, float gamma, int dtype,
                     void *stream);

/* state = factor * state + seg_state, zstate likewise (both NULL or both given): one step of
 * the prefix above.  [B, H, D, dv] and [B, H, D] fp32 device arrays; factor in [0, 1] (the
 * decay over seg_state's segment, gamma^len, or 1), else LA_ERR_ARG. */
int la_state_combine(float *state, float *zstate, const float *seg_state, const float *seg_zstate,
                     int B, int H, int D, int dv, float factor, void *stream);

/*
 * la_chunked_fwd_init -- the causal forward (plain mask, or the decay when gamma != 1)
 * starting from a given state: row t also reads gamma^(t+1) phi(q_t)^T state0 (and
 * zstate0 in the normaliser), as if the rows that produced state0 preceded row 0.
 * state0, zstate0: device fp32 [B, H, D, dv] and [B, H, D] (la_chunked_state's layout), or
 * NULL for zero.  Other arguments as la_decay_fwd; no level weights.  The tensor-core path
 * covers it for identity / elu+1 with C <= 64 (decay: C = 64); FAVOR+ and C > 64 run on the
 * generic path.  The workspace is la_chunked_workspace_bytes (gamma = 1) or
 * la_decay_workspace_bytes.
 */
int la_chunked_fwd_init(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                        int dk, int dv, int C, const la_feature_map *feature_map, int normalize,
                        float gamma, const float *state0, const float *zstate0, int dtype,
                        void *workspace, size_t workspace_bytes, void *stream, int path);

/* Library version string, e.g. "0.1.0". */
const char *la_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_CHUNKED_H */
