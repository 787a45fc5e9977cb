/*
 * apex_attn.h -- C ABI of the GB300 (sm_103a) APEX-1 attention block.
 *
 * The block computes, for every batch b, query head h and query row r
 * (APEX-1 Mathematical Reference, Part 1 §4 and Part 2 §6, §8, §10):
 *
 *   m      = q_pos0 + r                       position of the query row
 *   g      = floor(h / G),  G = H_q / H_kv    KV head shared by the group
 *                                             (Part 2 §8.2; §8.4 example)
 *   q'     = RoPE(q[b,h,r], m)                interleaved pairs (2i, 2i+1)
 *   k'_j   = RoPE(k[b,g,j], j)                rotated by angle pos*theta_i,
 *                                             theta_i = base^(-2i/d_h)
 *                                             (Part 1 §4.2-§4.4)
 *   out    = sum_j softmax_j(<q', k'_j> / sqrt(d_h)) v[b,g,j]
 *            over the keys j visible from m   (Part 2 §6.2)
 *   visible(m, j) <=> j <= m  and  (window <= 0  or  m - j < window)
 *                                             (Part 2 §10.2)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are dense, row-major, bf16 (raw 16-bit patterns), in device
 *   memory, with the 4-D attention layout [B, H, S, d_h] (Part 1 §1 "Tensor
 *   Shape Convention").  Every pointer must be 16-byte aligned.
 * - The caller owns every buffer it passes, scratch included: the decode's
 *   split partials and the prefill's rotated keys live in workspaces the caller
 *   passes (sizes from the *_workspace_bytes functions).  The library owns only
 *   a per-device cache of RoPE cos/sin tables (fp32, built in double precision
 *   on the host), allocated on first use and grown on demand.  A call that has to build or
 *   grow that table allocates device memory and synchronises the device;
 *   apex_attn_rope_reserve() builds it ahead of time.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *   stream) and returns before it finishes.  Calls are thread-compatible:
 *   concurrent calls on one device serialise on an internal lock while they
 *   enqueue.
 * - Supported: d_h in {64, 128}; H_q % H_kv == 0 with G = H_q / H_kv in
 *   {1, 2, 4, 8, 16}; 1 <= S <= 2^24; q_pos0 >= 0 and q_pos0 + S_q <= S_k, so
 *   that every query row sees at least its own key.
 * - Arguments are validated before anything is launched: a rejected call
 *   launches nothing and returns APEX_ERR_INVALID_ARG (bad value) or
 *   APEX_ERR_UNSUPPORTED (valid but outside the supported set).  A CUDA
 *   failure while enqueuing returns APEX_ERR_CUDA; the CUDA error state is left
 *   as the runtime reports it.  No entry point prints, traps or exits.
 * - Every wait inside the kernels is bounded in time.  A wait that gives up
 *   records a code in a per-device status word and lets the kernel finish
 *   (with unspecified output); apex_attn_device_status() reads and clears it.
 */
#ifndef APEX_ATTN_H
#define APEX_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum apex_status {
    APEX_OK = 0,
    APEX_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or position */
    APEX_ERR_UNSUPPORTED = 2,  /* valid arguments outside the supported set     */
    APEX_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed             */
    APEX_ERR_NO_MEMORY = 4,    /* the RoPE table could not be allocated          */
    APEX_ERR_DEVICE_TIMEOUT = 5 /* a kernel's bounded wait gave up (see below)   */
} apex_status;

/* Opaque CUDA stream handle (same object as cudaStream_t / CUstream). */
typedef struct CUstream_st *apex_stream_t;

/*
 * Prefill: attention of S_q query rows against S_k keys.
 *
 *   q   [B, H_q,  S_q, d_h]  bf16, read      (query row r sits at q_pos0 + r)
 *   k   [B, H_kv, S_k, d_h]  bf16, read      (raw keys: RoPE is applied here,
 *   v   [B, H_kv, S_k, d_h]  bf16, read       key j at position j)
 *   out [B, H_q,  S_q, d_h]  bf16, written   (must not overlap q, k or v)
 *   window     <= 0: causal only; > 0: key j visible iff 0 <= m - j < window
 *   rope_base  RoPE base b of theta_i = b^(-2i/d_h) (10000 on the pages);
 *              must be finite and > 0
 *
 * Cites: Part 2 §6.2 (SDPA), §8.2 (GQA), §10.2 (mask); Part 1 §4 (RoPE).
 * Errors: see the conventions above.  Result: softmax in fp32 with exp2; Q, K
 * are rotated in fp32 and rounded to bf16 for the tensor cores, as is P.
 */
apex_status apex_attn_fwd(const void *q, const void *k, const void *v, void *out,
                          int B, int H_q, int H_kv, int S_q, int S_k, int d_h,
                          int window, int q_pos0, float rope_base, apex_stream_t stream);

/*
 * Options of the _ex entry points.  Zero-initialise the struct and set what is
 * needed: all zeros is the plain block with rope_base 10000.
 */
typedef struct apex_attn_options {
    int window;           /* <= 0: causal only; > 0: sliding window W            */
    int q_pos;            /* fwd: position of query row 0; decode: the query's   */
    float rope_base;      /* RoPE base b of theta_i = b^(-2i/d_h); 0 means 10000 */
    float yarn_scale;     /* YaRN factor s (Part 1 §5); <= 1: no YaRN            */
    float yarn_beta_fast; /* wavelength below which a pair is unscaled; 0: 32    */
    float yarn_beta_slow; /* beta_slow * s: wavelength above which theta/s; 0: 1 */
    int prefix_len;       /* P > 0: positions [0, P) attend to each other
                             bidirectionally (Part 2 §11.1); 0 <= P <= S_k       */
    int keys_prerotated;  /* non-zero: k / k_cache already hold RoPE(k_j, j)     */
} apex_attn_options;

/*
 * YaRN (Part 1 §5.3-§5.5), when yarn_scale > 1: with the wavelength
 * lambda_i = 2 pi / theta_i, pairs with lambda_i < beta_fast keep theta_i,
 * pairs with lambda_i > beta_slow * s use theta_i / s, the others use
 * theta_i / (t s + 1 - t), t = clamp((lambda_i / beta_slow - 1) / (s - 1), 0, 1);
 * the scores are multiplied by 0.1 ln(s) + 1.
 * Prefix (Part 2 §11.1), when prefix_len = P > 0: a query at m < P sees the keys
 * j < P and nothing else; queries at m >= P follow the causal/window rule.
 */

/*
 * Prefill with options: as apex_attn_fwd, with window, q_pos0 (= opt->q_pos)
 * and rope_base taken from *opt.  opt may not be NULL.
 */
apex_status apex_attn_fwd_ex(const void *q, const void *k, const void *v, void *out,
                             int B, int H_q, int H_kv, int S_q, int S_k, int d_h,
                             const apex_attn_options *opt, apex_stream_t stream);

/*
 * Bytes of caller-provided device workspace apex_attn_fwd_ws will use for this
 * call (same arguments): one rotated copy of the keys, B * H_kv * S_k * d_h bf16
 * values, when the library's cost model rotates the keys before the prefill;
 * 0 when it would not (then no workspace is needed), when opt->keys_prerotated
 * is set, and when the arguments are invalid.  Host-only, no CUDA call.
 */
size_t apex_attn_fwd_workspace_bytes(int B, int H_q, int H_kv, int S_q, int S_k, int d_h,
                                     const apex_attn_options *opt);

/*
 * Prefill with options and a workspace: the same result as apex_attn_fwd_ex
 * (same arguments, layouts, masks and rounding up to the order of fp32 sums),
 * computed faster on long or wide problems.  The pages rotate every key by its
 * position (Part 1 §4.2-§4.5); the prefill rotates each 128-key tile in shared
 * memory once for every work item that reaches it, which on long windows or
 * wide head groups means tens of times.  Given a workspace, the library may
 * instead rotate the keys once, RoPE(k_j, j) in bf16 as apex_attn_rope_keys
 * computes it, into the workspace and run the prefill on those (it does so when
 * its cost model -- key-tile visits against one read and write of K -- says
 * that is faster; otherwise the workspace is left untouched).
 *
 *   workspace, workspace_bytes: NULL (then this is apex_attn_fwd_ex), or device
 *     memory of at least apex_attn_fwd_workspace_bytes(...) bytes for the same
 *     arguments, 16-byte aligned, owned by the caller, not overlapping q, k, v
 *     or out, not read before written; a smaller or misaligned workspace gives
 *     APEX_ERR_INVALID_ARG before any launch.
 *   The pass is a second kernel on `stream` before the prefill; with
 *   opt->keys_prerotated no pass runs.
 * Errors as for apex_attn_fwd_ex.
 */
apex_status apex_attn_fwd_ws(const void *q, const void *k, const void *v, void *out,
                             int B, int H_q, int H_kv, int S_q, int S_k, int d_h,
                             const apex_attn_options *opt, void *workspace, size_t workspace_bytes,
                             apex_stream_t stream);

/*
 * Prefill of multi-head latent attention with decoupled RoPE (Part 2 §9.3):
 * query and key rows are [content | rope part], the rope part alone is
 * rotated, and values keep the content length.
 *
 *   q   [B, H_q,  S_q, d_h + d_r] bf16, read     (row: q_content | q_rope)
 *   k   [B, H_kv, S_k, d_h + d_r] bf16, read     (row: k_content | k_rope)
 *   v   [B, H_kv, S_k, d_h]       bf16, read
 *   out [B, H_q,  S_q, d_h]       bf16, written  (must not overlap q, k or v)
 *
 * The rope part is rotated as a d_r-dimensional RoPE vector (pairs numbered
 * from its start, theta_i = b^(-2i/d_r), with the options' YaRN rule); the
 * content part is used as it is.  Scores are the dot products of the whole
 * rows divided by sqrt(d_h + d_r) (times the YaRN temperature).  With
 * opt->keys_prerotated the rope part of k is taken as already rotated.  All
 * other options and the masks are those of apex_attn_fwd_ex.
 * Supported: d_h = 128, d_r = 64 (else APEX_ERR_UNSUPPORTED); d_r must be
 * even and > 0 (else APEX_ERR_INVALID_ARG); H_q / H_kv as for apex_attn_fwd.
 * Runs on pairs of CTAs (a thread-block cluster of 2).
 */
apex_status apex_attn_mla_fwd(const void *q, const void *k, const void *v, void *out,
                              int B, int H_q, int H_kv, int S_q, int S_k, int d_h, int d_r,
                              const apex_attn_options *opt, apex_stream_t stream);

/*
 * Bytes of caller-provided device workspace apex_attn_mla_fwd_ws will use for
 * this call (same arguments): one copy of the key rows with the rope part
 * rotated, B * H_kv * S_k * (d_h + d_r) bf16 values, when the library's cost
 * model rotates the keys before the prefill; 0 when it would not, when
 * opt->keys_prerotated is set, and when the arguments are invalid or
 * unsupported.  Host-only, no CUDA call.
 */
size_t apex_attn_mla_fwd_workspace_bytes(int B, int H_q, int H_kv, int S_q, int S_k, int d_h, int d_r,
                                         const apex_attn_options *opt);

/*
 * Decoupled-RoPE prefill with a workspace: the same result as apex_attn_mla_fwd
 * (up to the order of fp32 sums), with the rope part of every key row rotated
 * once into the workspace beforehand (as apex_attn_mla_rope_keys computes it;
 * the content part copied) when the cost model says that is faster than
 * rotating it in every work item that visits the key tile.  workspace and
 * workspace_bytes as for apex_attn_fwd_ws, sized by
 * apex_attn_mla_fwd_workspace_bytes(...); NULL makes this apex_attn_mla_fwd.
 * Errors as for apex_attn_mla_fwd, plus APEX_ERR_INVALID_ARG for a smaller or
 * misaligned workspace (before any launch).
 */
apex_status apex_attn_mla_fwd_ws(const void *q, const void *k, const void *v, void *out,
                                 int B, int H_q, int H_kv, int S_q, int S_k, int d_h, int d_r,
                                 const apex_attn_options *opt, void *workspace, size_t workspace_bytes,
                                 apex_stream_t stream);

/*
 * Decode with options: as apex_attn_decode, with window, q_pos and rope_base
 * taken from *opt.  With a prefix and q_pos < P the query sees keys [0, P).
 * The workspace size is apex_attn_decode_workspace_bytes(...) as for
 * apex_attn_decode.
 */
apex_status apex_attn_decode_ex(const void *q, const void *k_cache, const void *v_cache, void *out,
                                int B, int H_q, int H_kv, int S_k, int d_h,
                                const apex_attn_options *opt, void *workspace,
                                size_t workspace_bytes, apex_stream_t stream);

/*
 * Diagnostic (the pages have no counterpart): launches one CTA whose bounded
 * mbarrier wait -- the wait every kernel of this library uses -- can never
 * complete.  After timeout_ms (1..5000, else APEX_ERR_INVALID_ARG) the wait
 * gives up, records its code in the per-device status word and the kernel
 * returns; apex_attn_device_status() then reports APEX_ERR_DEVICE_TIMEOUT
 * (and clears it) and the context stays usable.  Asynchronous on `stream`.
 */
apex_status apex_attn_selftest_wait_timeout(int timeout_ms, apex_stream_t stream);

/*
 * Decode of multi-head latent attention with decoupled RoPE (Part 2 §9.3):
 * one query per sequence against a cache of [content | rope part] keys.
 *
 *   q       [B, H_q,  1,   d_h + d_r] bf16, read   (the query sits at opt->q_pos)
 *   k_cache [B, H_kv, S_k, d_h + d_r] bf16, read   (key j at position j)
 *   v_cache [B, H_kv, S_k, d_h]       bf16, read
 *   out     [B, H_q,  1,   d_h]       bf16, written
 *   workspace: at least apex_attn_decode_workspace_bytes(B, H_q, H_kv, S_k, d_h)
 *           bytes (d_h: the value row length), 16-byte aligned.
 *
 * Rotation, scores and options as for apex_attn_mla_fwd; the result equals
 * apex_attn_mla_fwd with S_q = 1 and q_pos0 = q_pos (up to the order of fp32
 * sums).  Supported: d_h = 128, d_r = 64.
 */
apex_status apex_attn_mla_decode(const void *q, const void *k_cache, const void *v_cache, void *out,
                                 int B, int H_q, int H_kv, int S_k, int d_h, int d_r,
                                 const apex_attn_options *opt, void *workspace, size_t workspace_bytes,
                                 apex_stream_t stream);

/*
 * Rotate keys for a pre-rotated KV cache (Part 1 §4.2-§4.4, with the options'
 * rope_base / YaRN): for each of n_heads heads h and each s < n_pos,
 *   k_out[h * out_head_stride + s * d_h + :] = RoPE(k_in[h * in_head_stride + s * d_h + :], pos0 + s)
 * in bf16 (fp32 arithmetic).  Strides are in elements; with
 * out_head_stride = S_cache * d_h and k_out pointing at row pos0 of a cache,
 * this appends freshly projected keys to that cache.  k_out may equal k_in
 * (same strides) for an in-place rotation; otherwise the ranges must not
 * overlap.  Only window/prefix-independent fields of *opt are used.
 */
apex_status apex_attn_rope_keys(const void *k_in, void *k_out, int n_heads, int n_pos, int d_h, int pos0,
                                long long in_head_stride, long long out_head_stride,
                                const apex_attn_options *opt, apex_stream_t stream);

/*
 * The same for decoupled-RoPE key rows [content (d_h) | rope part (d_r)]
 * (Part 2 §9.3): for each head h and s < n_pos the row at
 * k_in[h * in_head_stride + s * (d_h + d_r)] goes to k_out with its content
 * part copied and its rope part rotated as a d_r-dimensional RoPE vector at
 * position pos0 + s (pairs numbered from the rope part's start,
 * theta_i = b^(-2i/d_r), the options' YaRN rule) -- the keys
 * apex_attn_mla_fwd / apex_attn_mla_decode take with opt->keys_prerotated.
 * Strides in elements (at least n_pos * (d_h + d_r), multiples of 8), overlap
 * rules as for apex_attn_rope_keys.  Supported: d_h = 128, d_r = 64 (else
 * APEX_ERR_UNSUPPORTED); d_r must be even and > 0 (else APEX_ERR_INVALID_ARG).
 */
apex_status apex_attn_mla_rope_keys(const void *k_in, void *k_out, int n_heads, int n_pos, int d_h, int d_r,
                                    int pos0, long long in_head_stride, long long out_head_stride,
                                    const apex_attn_options *opt, apex_stream_t stream);

/*
 * Bytes of caller-provided device workspace apex_attn_decode needs for these
 * sizes (the split-KV partial results).  Returns 0 when the sizes are invalid.
 * The same sizes with any window / q_pos never need more.
 */
size_t apex_attn_decode_workspace_bytes(int B, int H_q, int H_kv, int S_k, int d_h);

/*
 * Decode: one query per sequence against a bf16 KV cache.
 *
 *   q       [B, H_q,  1,   d_h] bf16, read   (the query sits at position q_pos)
 *   k_cache [B, H_kv, S_k, d_h] bf16, read   (raw keys, key j at position j)
 *   v_cache [B, H_kv, S_k, d_h] bf16, read
 *   out     [B, H_q,  1,   d_h] bf16, written
 *   q_pos   0 <= q_pos < S_k; keys j > q_pos are masked (causal)
 *   window  as for apex_attn_fwd
 *   workspace, workspace_bytes: device scratch of at least
 *           apex_attn_decode_workspace_bytes(B, H_q, H_kv, S_k, d_h) bytes,
 *           16-byte aligned, owned by the caller, not read before written.
 *
 * The result equals apex_attn_fwd with S_q = 1 and q_pos0 = q_pos (up to the
 * order of fp32 sums).  The KV range is split across CTAs; each split writes
 * a partial (max, sum, unnormalised output) and a log-sum-exp combine kernel
 * merges them (Part 2 §6.2: softmax is invariant to the shift by the max).
 * Cites: Part 2 §6.2, §7.4 (KV cache), §8.2, §10.2; Part 1 §4.
 */
apex_status apex_attn_decode(const void *q, const void *k_cache, const void *v_cache, void *out,
                             int B, int H_q, int H_kv, int S_k, int d_h, int window, int q_pos,
                             float rope_base, void *workspace, size_t workspace_bytes,
                             apex_stream_t stream);

/*
 * Decode that allocates nothing, for callers that cannot allocate device
 * memory when they call: an engine whose device memory is all handed out by
 * its own pool at start-up (a cudaMalloc would fail, fragment the pool or
 * synchronise the device), a plugin interface with a fixed signature and no
 * workspace slot, or a latency-critical loop that cannot afford an
 * allocation's synchronisation.  The APEX-1 pages have no counterpart of this
 * entry point; it computes exactly what apex_attn_decode computes.
 *
 *   Arguments, layouts and results: as apex_attn_decode, without workspace.
 *   Scratch: split-KV partials live in a 16 MiB file-scope device array and
 *     the RoPE table in a 16 MiB one (positions < 32768); every GPU that loads
 *     the library holds these 32 MiB until the process exits.  Nothing in them
 *     has to start at zero: each call writes every partial it reads.
 *   Limits (APEX_ERR_UNSUPPORTED beyond them): S_k <= 32768, d_h in {64, 128},
 *     G in {1, 2, 4, 8, 16}, and B * H_q * (4 * d_h + 8) <= 16 MiB (one split);
 *     larger B * H_q only lowers the number of KV splits the scratch allows.
 *   Set-up: the first call on a device (and the first call with a new
 *     (d_h, rope_base) pair) looks up the arrays' device addresses, builds the
 *     RoPE table on `stream` and synchronises that stream; make that call before
 *     capturing any CUDA graph.
 *   Concurrency: all calls on a device share the arrays, so calls that may
 *     overlap on the GPU (different streams without ordering between them) race
 *     and must not be issued.  Kernel waits are bounded as on the other entry
 *     points (APEX_ATTN_WAIT_TIMEOUT_MS, 2 s by default), but a wait that times
 *     out is not recorded (there is no status word without allocation); the
 *     output is then unspecified.  If the table build fails (APEX_ERR_CUDA),
 *     the next call rebuilds it.
 */
apex_status apex_attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, void *out,
                                     int B, int H_q, int H_kv, int S_k, int d_h, int window, int q_pos,
                                     float rope_base, apex_stream_t stream);

/*
 * Build (or grow) the RoPE cos/sin table of the current device so that
 * positions [0, max_pos) are covered for this (d_h, rope_base).  Synchronous.
 * Calling it before capturing a CUDA graph keeps the captured calls free of
 * allocations.  Part 1 §4.7 (cos/sin cache computed once, reused).
 */
apex_status apex_attn_rope_reserve(int max_pos, int d_h, float rope_base);

/*
 * Read and clear the current device's status word, after synchronising the
 * device.  APEX_OK when no kernel recorded a problem since the last call;
 * APEX_ERR_DEVICE_TIMEOUT when a bounded wait gave up; APEX_ERR_CUDA when the
 * synchronisation itself failed.
 */
apex_status apex_attn_device_status(void);

/* Static, human-readable name of a status code (never NULL). */
const char *apex_attn_status_string(apex_status s);

#ifdef __cplusplus
}
#endif

#endif /* APEX_ATTN_H */
