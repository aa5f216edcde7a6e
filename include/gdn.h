/*
 * gdn.h — C ABI of libgdn.so: chunked Gated DeltaNet prefill and the
 * one-token decode step on NVIDIA GB300 (sm_103a).
 *
 * The operation (per sequence and value head, fp32 state S of shape [dk, dv]):
 *
 *   S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   o_t = q_scale * S_t^T q_t
 *
 * A prompt is cut into chunks of at most 64 rows and every chunk is solved in
 * closed form: gamma = cumsum(g) within the chunk,
 *   (I + A) U = diag(beta) V - diag(beta exp(gamma)) K S_0,
 *       A_ij = beta_i exp(gamma_i - gamma_j) k_i.k_j  (j < i),
 *   O   = diag(exp(gamma)) Q S_0 + (exp(gamma_t - gamma_i) q_t.k_i)_{i<=t} U,
 *   S_S = exp(gamma_S) S_0 + (K * exp(min(gamma_S - gamma, 0)))^T U,
 * with gamma_S the chunk's last cumulative sum.  Source: "perf(qwen3_5):
 * prefill text prompts in multi-token chunks" (TensorRT-Model-Connect pull
 * request 2191), Implementation section and its gamma_S commit message.  The
 * state is carried from chunk to chunk on the device, as that page's runtime
 * advances the recurrent state after each chunk (run_prefill_chunks /
 * commit_prefill), and the prefill reads and writes the same recurrent-state
 * layout as the decode step.
 *
 * Conventions for every entry point
 * ---------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   allocates no memory, never synchronises the device or the stream, and
 *   enqueues all work on `stream` (NULL = the legacy default stream).
 * - Layouts are row-major and token-major over a packed variable-length
 *   batch: q, k [T, Hk, dk]; v [T, Hv, dv]; g, beta [T, Hv]; out [T, Hv, dv];
 *   state [B, Hv, dk, dv].  Value head h reads key head h / (Hv / Hk).
 * - "bf16" tensors hold __nv_bfloat16 values, "fp32" tensors float.
 * - g must be <= 0 (a decay); this is a precondition, not checked.
 * - Validation happens before anything is enqueued: a call that returns a
 *   non-zero status enqueued nothing.  A GDN_ERR_CUDA status after a launch
 *   leaves out, state_out and conv_state_out unspecified (there is no
 *   rollback, as on the page's runtime: the caller re-runs from its own copy
 *   of the state).  Nothing throws across the ABI.
 * - Concurrent calls on different streams are safe when they share no output
 *   buffer.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* gdn_stream_t;

/* Status codes returned by every entry point. */
enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, bad cu_seqlens length, ... */
    GDN_ERR_CHUNK = 2,       /* chunk outside 1..64 (the static 64-row padding of the solve) */
    GDN_ERR_UNSUPPORTED = 3, /* dk or dv not in {16, 32, 64, 128}, Hv % Hk != 0, bad dtype/act */
    GDN_ERR_ALIGN = 4,       /* a tensor pointer not 16-byte aligned */
    GDN_ERR_CUDA = 5,        /* a kernel launch failed (see gdn_last_cuda_error) */
    GDN_ERR_WORKSPACE = 6,   /* workspace missing, too small or not 256-byte aligned */
    GDN_ERR_TOO_LARGE = 7    /* a size beyond what the entry point supports */
};

/* Element type of q, k, v, conv_x and out. */
enum gdn_dtype { GDN_BF16 = 0, GDN_FP32 = 1 };

/* Activation after the short convolution. */
enum gdn_act { GDN_ACT_NONE = 0, GDN_ACT_SILU = 1 };

/*
 * Full description of one prefill call (gdn_prefill_ex) or decode step
 * (gdn_step_ex).  Zero-initialise, then fill; gdn_prefill_desc_init sets the
 * defaults (bf16, chunk 64, L2 norm on with eps 1e-6, q_scale 1, conv kernel 4,
 * no activation).
 */
typedef struct gdn_prefill_desc {
    int dtype;               /* enum gdn_dtype */
    int B;                   /* number of sequences (>= 0) */
    int Hk, Hv;              /* key and value heads, Hv % Hk == 0 */
    int dk, dv;              /* head dims, each in {16, 32, 64, 128} */
    int chunk;               /* rows per chunk, 1..64 (results do not depend on it) */
    int64_t T_total;         /* cu_seqlens[B]; required with conv_x, else may be -1.
                              * 0: no token in the batch; the token tensors may then
                              * be NULL and the call only returns every sequence's
                              * states (state_out <- state_in, conv_state_out <-
                              * conv_state_in, zeros without them) by stream-ordered
                              * device copies, launching no kernel */

    const void* q;           /* [T, Hk, dk] dtype; ignored when conv_x != NULL */
    const void* k;           /* [T, Hk, dk] dtype; ignored when conv_x != NULL */
    const void* v;           /* [T, Hv, dv] dtype; ignored when conv_x != NULL */
    const float* g;          /* [T, Hv] log-decay per token, <= 0 */
    const float* beta;       /* [T, Hv] delta-rule step size */
    const float* state_in;   /* [B, Hv, dk, dv]; NULL = zero state */
    float* state_out;        /* [B, Hv, dk, dv]; NULL = not written; may alias state_in */
    void* out;               /* [T, Hv, dv] dtype */
    const int32_t* cu_seqlens; /* device [B+1]: cu[0] = 0, non-decreasing */

    /* Optional depthwise causal short convolution in front ("perf(mamba):
     * prefill text prompts in multi-token chunks", Implementation,
     * add_short_conv_rows): channels c in [0, C), C = 2*Hk*dk + Hv*dv, ordered
     * q | k | v; y_t = act(sum_j w[c, j] * xx[t + j]) over
     * xx = [conv_state_in[n, c, :], x[seq n, c]]; the new conv state is the
     * last K-1 columns of xx. */
    const void* conv_x;      /* [T, C] dtype, or NULL for no convolution */
    const float* conv_w;     /* [C, K] */
    const float* conv_state_in; /* [B, C, K-1] oldest first; NULL = zeros */
    float* conv_state_out;   /* [B, C, K-1]; NULL = not written; may alias conv_state_in */
    int conv_kernel;         /* K, 2..8 */
    int conv_act;            /* enum gdn_act */

    int use_qk_l2norm;       /* q, k <- x / sqrt(sum x^2 + l2_eps) per head vector */
    float l2_eps;
    float q_scale;           /* o_t = q_scale * S_t^T q_t */

    void* workspace;         /* device scratch, >= gdn_workspace_bytes(desc), 256-aligned */
    size_t workspace_bytes;

    /* Segment-parallel chunk scan (bf16, dk = dv = 128, T_total known, and a
     * workspace): each sequence is cut into segments of this many chunks that
     * run in parallel.  Every later segment runs from a zero state (its
     * outputs O' and end state B_s) and from the identity with V = 0 (its
     * output map G and transition M_s); one more pass forms each segment's
     * incoming state S_s (S_{s+1} = M_s S_s + B_s) and its outputs
     * O = O' + G S_s on the tensor cores.  The workspace then also holds the
     * maps (3 x 64 KiB per value head and segment slot) and G (bf16, like
     * out).  0 = chosen from the shape by a cost model of the passes on the
     * current device's SMs (one pass when that is cheaper), < 0 = off.  The
     * chain kernels take the sequences longest first, so that with more
     * (sequence, head) units than one wave holds the longest chains start
     * first. */
    int segment_chunks;

    /* Split preparation (bf16, dk = dv = 128, T_total known, and a
     * workspace): the part of every chunk that does not depend on the
     * incoming state (q/k norms, the cumulative decay, the masked Gram
     * matrices, the blocked inverse T, U0 = T diag(beta) V,
     * W = T diag(beta exp(gamma)) K, the intra-chunk output weights and the
     * scaled queries) is solved first for all chunks in parallel and stored
     * as one 82432-byte record per (value head, chunk slot), Hv *
     * (T_total / chunk + B + 1) records; the state pass then streams the
     * records (chunk_state_kernel).  The results agree with those without
     * it within rounding.  >= 0 = on when the workspace holds the records
     * and there are fewer than 2^31 of them (else, as with < 0, off and
     * not asked for by gdn_workspace_bytes). */
    int split_prep;
} gdn_prefill_desc;

/* Fill *d with the defaults listed above (all pointers NULL). */
void gdn_prefill_desc_init(gdn_prefill_desc* d);

/*
 * gdn_prefill — chunked prefill, bf16 q/k/v/out, fp32 g/beta/state, q/k L2
 * normalisation on (eps 1e-6), q_scale 1, no convolution.  Grids are sized
 * from (B, Hv); cu_seqlens is read on the device, so the total length is not
 * needed.  Needs no workspace, and so runs neither the segment-parallel scan
 * nor the split preparation: one CTA per (sequence, value head) walks all of
 * its chunks in one kernel (chunk_tc_kernel for bf16, dk = dv = 128).  That
 * is several times slower than gdn_prefill_ex with a workspace on a long or
 * few-sequence batch (4096 tokens x 16 heads on a GB300: about 0.45 ms
 * against 0.095 ms); callers that can spare the workspace should use
 * gdn_prefill_ex.
 *   q, k      bf16 [T, Hk, dk]      v, out   bf16 [T, Hv, dv]
 *   g, beta   fp32 [T, Hv]          state_in / state_out  fp32 [B, Hv, dk, dv]
 *   cu_seqlens int32 [B+1] (device)  chunk in 1..64
 * Returns a gdn_status.
 */
int gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                const float* state_in, float* state_out, void* out, const int32_t* cu_seqlens,
                int B, int Hk, int Hv, int dk, int dv, int chunk, gdn_stream_t stream);

/* gdn_prefill_ex — the general prefill: dtype, short convolution, L2 norm,
 * q_scale and workspace as described in gdn_prefill_desc. */
int gdn_prefill_ex(const gdn_prefill_desc* d, gdn_stream_t stream);

/* Device workspace gdn_prefill_ex uses for *d, in bytes (0 if none), laid
 * out in this order: the output of the short convolution, the per-segment
 * maps and the output map G of the segment-parallel scan when that is
 * chosen, the chunk records of
 * the split preparation when that is on.  Reads only dtype, B, Hk, Hv, dk,
 * dv, chunk, T_total, segment_chunks, split_prep and whether conv_x is set;
 * returns (size_t)-1 when those are invalid.  Only the convolution's part is
 * required: a workspace too small for the maps and G runs the scan in one
 * pass, one too small for the records solves each chunk inside the state
 * pass (same results either way). */
size_t gdn_workspace_bytes(const gdn_prefill_desc* d);

/*
 * gdn_step — one decode token per sequence (the unchanged one-token step of
 * the page's runtime), bf16, L2 norm on, q_scale 1, no convolution:
 *   q, k bf16 [B, Hk, dk]; v bf16 [B, Hv, dv]; g, beta fp32 [B, Hv];
 *   state fp32 [B, Hv, dk, dv], updated in place; out bf16 [B, Hv, dv].
 */
int gdn_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
             float* state, void* out, int B, int Hk, int Hv, int dk, int dv,
             gdn_stream_t stream);

/* gdn_step_ex — decode step from a description: one token per sequence, so
 * q, k, v, conv_x, g, beta and out have B rows; cu_seqlens must be NULL and
 * T_total is ignored; chunk is ignored.  state_in / state_out may alias
 * (in-place update); conv_state_in / conv_state_out likewise.  No workspace. */
int gdn_step_ex(const gdn_prefill_desc* d, gdn_stream_t stream);

/* The kernels gdn_prefill_ex launches for *d, in launch order: writes up to
 * max_names pointers to static, NUL-terminated kernel names into names (which
 * may be NULL when max_names is 0) and returns how many kernels one call
 * launches, or minus a gdn_status when *d would be rejected.  Host-only: no
 * CUDA call, nothing enqueued. */
int gdn_prefill_plan(const gdn_prefill_desc* d, const char** names, int max_names);

/*
 * gdn_prefill_noalloc — gdn_prefill_ex for callers that cannot allocate
 * device memory (the pages have no counterpart: it is an addition for
 * users of this library).  Some callers cannot provide the scratch workspace
 * that a prefill with the short convolution needs: a serving runtime whose
 * device memory is all handed to its own pool and that may not call
 * cudaMalloc on the request path, or code that must not allocate because an
 * allocation can synchronise the device.  This entry point takes the same
 * description as gdn_prefill_ex (inputs and outputs still come from the
 * caller) but ignores d->workspace and uses a fixed scratch array inside the
 * library, gdn_noalloc_scratch_bytes() = 32 MiB, for the convolution's output
 * and, when they fit beside it, the chunk records and segment maps that make
 * a call faster (larger calls run the slower one-pass plan).  It allocates
 * nothing itself.
 *   - A description whose required workspace (the conv output: T_total * C *
 *     element size) exceeds the array is rejected with GDN_ERR_TOO_LARGE.
 *   - The array's device memory is reserved when the library's module that
 *     holds it is loaded on a device: with the CUDA runtime's default lazy
 *     module loading that is the first call on that device, which also looks
 *     up the array's address (cudaGetSymbolAddress, device current).  Make
 *     that first call at initialisation, before the caller's own pool takes
 *     the device's memory (else GDN_ERR_CUDA) and before any stream capture;
 *     later calls reserve nothing more.  The memory stays reserved until the
 *     process exits.
 *   - Every call shares the one array: calls whose work overlaps on the GPU
 *     (other streams, other host threads) race on it; serialise them.
 */
int gdn_prefill_noalloc(const gdn_prefill_desc* d, gdn_stream_t stream);

/* Size in bytes of the fixed scratch array gdn_prefill_noalloc uses. */
size_t gdn_noalloc_scratch_bytes(void);

/* ---- Selective-scan rows -------------------------------------------------
 * h_t = a_t h_{t-1} + b_t per channel over the rows of every sequence: the
 * add_selective_scan_rows recurrence of "perf(mamba): prefill text prompts in
 * multi-token chunks" (Implementation), in fp32 like the page.  The page runs
 * it on chunks of at most 64 rows by doubling rounds, the state carried from
 * chunk to chunk; one call here covers whole prompts (the result does not
 * depend on the chunking).
 *
 *   a, b        [T_total, C] fp32, token-major (the page's a_t are decays in
 *               (0, 1]; any finite values are accepted)
 *   h_in        [B, C] fp32 incoming state, or NULL for a zero state
 *   h_out       [B, C] fp32 state after each sequence's last row (h_in, or
 *               zero, for an empty sequence); may alias h_in
 *   h_rows      [T_total, C] fp32: h_t for every row
 *   cu_seqlens  [B+1] int32: cu[0] = 0, non-decreasing, cu[B] = T_total
 *   workspace   gdn_scan_workspace_bytes(C, T_total) bytes, 256-byte aligned,
 *               caller-owned; needs no initialisation; one call at a time
 * All pointers are device pointers; the call enqueues two kernels on
 * `stream`, allocates nothing and does not synchronise.  C must be a
 * multiple of 4 and a, b, h_rows 16-byte aligned.  Status: GDN_OK;
 * GDN_ERR_INVALID_ARG (NULL pointer or negative size); GDN_ERR_UNSUPPORTED
 * (C not a multiple of 4); GDN_ERR_ALIGN; GDN_ERR_WORKSPACE; GDN_ERR_TOO_LARGE
 * (more than 2^31 - 1 tiles of 256 rows x 32 channels); GDN_ERR_CUDA. */
size_t gdn_scan_workspace_bytes(int C, int64_t T_total);
int gdn_scan_rows(const float* a, const float* b, const float* h_in, float* h_out, float* h_rows,
                  const int32_t* cu_seqlens, int B, int C, int64_t T_total, void* workspace,
                  size_t workspace_bytes, gdn_stream_t stream);

/* ---- RWKV-4 WKV rows ------------------------------------------------------
 * The WKV of RWKV-4 time mixing over the rows of every sequence, as the
 * one-token decoder of "perf(rwkv): prefill text prompts in multi-token
 * chunks" (Implementation) computes it.  Per channel the state is
 * (num, den, max), A = num exp(max) and B = den exp(max), of
 *   A_t = exp(w) A_{t-1} + exp(k_t) v_t,   B_t = exp(w) B_{t-1} + exp(k_t),
 * and row t outputs
 *   wkv_t = (A_{t-1} + exp(u + k_t) v_t) / (B_{t-1} + exp(u + k_t)),
 * every exponential taken after subtracting the largest exponent of its sum.
 * The page builds each chunk of at most 64 rows as one exponent tensor; one
 * call here covers whole prompts (the result does not depend on chunking).
 *
 *   k, v        [T_total, C] fp32, token-major
 *   w, u        [C] fp32 per-channel decay exponent (exp(w) the decay) and bonus
 *   state_in    [B, 3, C] fp32 (num, den, max) or NULL for the empty state
 *               (0, 0, -1e38)
 *   state_out   [B, 3, C] fp32 state after each sequence's last row (state_in,
 *               or the empty state, for an empty sequence); may alias state_in.
 *               The triple is one representation of (A, B): (num c, den c,
 *               max - log c) is the same state.
 *   wkv         [T_total, C] fp32 outputs
 *   cu_seqlens  [B+1] int32: cu[0] = 0, non-decreasing, cu[B] = T_total
 *   workspace   gdn_wkv_workspace_bytes(C, T_total) bytes, 256-byte aligned,
 *               caller-owned; needs no initialisation; one call at a time
 * Device pointers; two kernels enqueued on `stream`; nothing allocated, no
 * synchronisation.  C must be a multiple of 4 and k, v, wkv 16-byte aligned.
 * Status codes as for gdn_scan_rows. */
size_t gdn_wkv_workspace_bytes(int C, int64_t T_total);
int gdn_wkv_rows(const float* k, const float* v, const float* w, const float* u,
                 const float* state_in, float* state_out, float* wkv, const int32_t* cu_seqlens,
                 int B, int C, int64_t T_total, void* workspace, size_t workspace_bytes,
                 gdn_stream_t stream);

/* ---- Full-attention rows over a KV cache ---------------------------------
 * The full-attention layers of a prefill chunk in "perf(qwen3_5): prefill
 * text prompts in multi-token chunks" (Implementation): the chunk's present
 * k / v rows are appended to the KV cache, and every query row attends over
 * the cache plus the chunk's causal prefix.  For sequence n with c =
 * cache_len[n] cached rows and chunk rows t = 0 .. L_n - 1:
 *   cache[n, kv, c + t] = (k_t, v_t) for every kv head (rows at or past the
 *                         capacity are dropped),
 *   o_t = softmax_j(scale q_t . K[j]) V[j] over cache rows j = 0 .. c + t,
 * with query head h reading kv head h / (Hq / Hkv).  bf16 tensors, fp32
 * scores, softmax and accumulation; head_dim must be 128.  cache_len is not
 * advanced (the caller commits the rows, as the page's runtime does).
 *
 *   q           [T_total, Hq, 128] bf16
 *   k, v        [T_total, Hkv, 128] bf16
 *   k_cache, v_cache  [B, Hkv, cache_capacity, 128] bf16, updated in place;
 *               cache_len[n] + L_n must not exceed cache_capacity
 *   cache_len   [B] int32 (device)
 *   o           [T_total, Hq, 128] bf16
 *   cu_seqlens  [B+1] int32: cu[0] = 0, non-decreasing, cu[B] = T_total
 *   scale       score scale; 0 selects 1 / sqrt(128)
 * Device pointers, 16-byte aligned; two kernels on `stream`; nothing
 * allocated.  Status: GDN_OK; GDN_ERR_INVALID_ARG; GDN_ERR_UNSUPPORTED
 * (head_dim != 128, Hq % Hkv != 0); GDN_ERR_ALIGN; GDN_ERR_TOO_LARGE;
 * GDN_ERR_CUDA. */
int gdn_attn_rows(const void* q, const void* k, const void* v, void* k_cache, void* v_cache,
                  const int32_t* cache_len, void* o, const int32_t* cu_seqlens, int B, int Hq, int Hkv,
                  int head_dim, int cache_capacity, int64_t T_total, float scale, gdn_stream_t stream);

/* Bounded device waits that ran out since the library was loaded (tensor-core
 * chunk kernel, selective scan, WKV rows and attention rows; a CTA whose wait runs out abandons its
 * work, so every result of the call that hit it is unspecified).  Waits for
 * the device to finish its work.  Returns the count, or -1 on a CUDA error. */
long long gdn_wait_timeouts(void);

/* ---- Launch timing ------------------------------------------------------
 * A host-side record of how long each kernel launch of the library took on
 * the GPU, for profiling without an external tool.  The pages define no such
 * call; it times the operations above.
 *
 * gdn_launch_timer_start(capacity) creates `capacity` pairs of CUDA events
 * (on the current device; capacity 1..1,000,000), forgets earlier records and
 * turns recording on: from then on every kernel the library launches, from
 * any entry point, is bracketed by a pair of events recorded on its stream.
 * Launches beyond the capacity run untimed and are counted as dropped.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG (capacity out of range) or
 * GDN_ERR_CUDA (event creation failed).  Not for use during stream capture.
 *
 * gdn_launch_timer_stop() turns recording off; the records stay readable.
 *
 * gdn_launch_timer_read(names, ms, max, dropped) waits for the recorded
 * events, writes the kernel name (static string) and duration in
 * milliseconds of the first min(count, max) launches in launch order, writes
 * the dropped count to *dropped (if non-NULL) and returns the number of
 * recorded launches (negative status on a CUDA error); a launch that was
 * begun but never made (its call failed) reads -1 ms.  names or ms may be
 * NULL to query the count.  The calls are thread-safe; launches made on
 * several streams at once are recorded on their own streams. */
int gdn_launch_timer_start(int capacity);
int gdn_launch_timer_stop(void);
int gdn_launch_timer_read(const char** names, float* ms, int max, int* dropped);

/* Static description of a status code. */
const char* gdn_status_string(int status);

/* The cudaError_t of the last failed launch on this thread (0 if none). */
int gdn_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
