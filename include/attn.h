/*
 * attn.h — C ABI of the GB300 (sm_103a) attention library.
 *
 * Four operations, all from the pages' problem statement of LLM-serving attention:
 *   rope_apply          rotary position embedding on a [B,H,S,D] tensor
 *   attn_prefill        causal / non-causal grouped-query attention, RoPE optionally fused
 *   attn_prefill_chunk  a prompt chunk against a static cache (bottom-right causal)
 *   attn_decode         one query token per sequence against a static KV cache (split-KV)
 *   attn_decode_append  a decode step whose token joins the cache (growing decode)
 *   attn_decode_latent  absorbed latent (MLA-style) decode: 448 latent + 64 RoPE dims
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise.  The caller owns every
 *     buffer; the library never frees caller memory.
 *   - Tensors are dense, row-major, innermost dimension last, base addresses 16-byte aligned.
 *   - Storage types: ATTN_BF16 = bfloat16, ATTN_FP8_E5M2 = OCP float8 e5m2.  Outputs O are
 *     always bfloat16; optional LSE outputs are float32 natural-log log-sum-exp of the scaled
 *     scores.
 *   - Grouped-query mapping: query head hq reads KV head hq / (Hq / Hkv).
 *   - RoPE is the rotate-half pairing (x_i, x_{i+D/2}) rotated by pos * theta^(-2i/D).
 *   - softmax_scale <= 0 selects 1/sqrt(head dim used for scores).
 *   - Calls are asynchronous on `stream` and return after enqueueing.  Host-side validation
 *     happens before anything is enqueued; on any error nothing is launched and outputs are
 *     untouched.  Kernels never trap: a device-side problem (a cache_len out of range, a wait
 *     that timed out) sets a device status word read by attn_get_device_status().
 *   - Scratch memory comes from the caller: calls that need it take a workspace pointer and
 *     size (each with a *_workspace_size() query).  The library's own device memory is the
 *     cos/sin table used by RoPE, the 4-byte status word and attn_decode_noalloc's fixed array.
 *     The table is built on the host in float64, stored as float32 and cached per device and
 *     (D, theta).  The first call that needs a table (or more positions than the cached one
 *     holds) allocates it with cudaMalloc and copies it synchronously; call
 *     attn_rope_table_reserve() first to keep that out of timed regions and graph captures.
 *     Every other path allocates nothing.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t.  NULL selects the legacy default stream. */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, Hq % Hkv != 0 ... */
  ATTN_ERR_UNSUPPORTED = 2,   /* valid but not built: head dim, dtype or group size not covered */
  ATTN_ERR_WORKSPACE = 3,     /* workspace pointer null or smaller than the *_workspace_size() */
  ATTN_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  ATTN_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up (from attn_get_device_status) */
  ATTN_ERR_NO_DEVICE = 6,     /* no CUDA device, or not an sm_100-family device */
  ATTN_ERR_DEVICE_ARG = 7     /* a device-resident argument (cache_len) was out of range */
} attn_status_t;

typedef enum { ATTN_BF16 = 0, ATTN_FP8_E5M2 = 1 } attn_dtype_t;

/*
 * RoPE pairing convention.  Both rotate pair i by the angle pos * theta^(-2i/D) (the same
 * cos/sin table); they differ in which two dims form pair i:
 *   ATTN_ROPE_HALF_SPLIT   dims (i, i + D/2)  (the default everywhere)
 *   ATTN_ROPE_INTERLEAVED  dims (2i, 2i + 1)
 * The pages do not fix a convention; the interleaved one is the other common form.
 * The _INVERSE forms (rope_apply_style only) rotate by the opposite angles: the transpose of
 * the rotation, which maps gradients of rotated Q / K (attn_prefill_backward's dq, dk) back to
 * the un-rotated inputs.
 */
typedef enum {
  ATTN_ROPE_HALF_SPLIT = 0,
  ATTN_ROPE_INTERLEAVED = 1,
  ATTN_ROPE_HALF_SPLIT_INVERSE = 2,
  ATTN_ROPE_INTERLEAVED_INVERSE = 3
} attn_rope_style_t;

/* OR'd into the `rope` argument of the attention calls (with a nonzero mode) to select the
 * interleaved pairing; for the latent decode it applies to the 64 RoPE dims. */
#define ATTN_ROPE_FLAG_INTERLEAVED 16

/* Static English description of a status code.  Never NULL. */
ATTN_API const char* attn_status_string(attn_status_t status);

/* Library ABI version (major * 100 + minor). */
ATTN_API int attn_version(void);

/*
 * rope_apply — rotary position embedding, the unfused form.
 * Defines: the RoPE the pages fuse into attention or run as a separate pass (Lesson: shape
 * adaptive attention negative 20260722, rows "해본 것" and "실제 결과": fused versus unfused
 * RoPE + attention).
 *   x      [B,H,S,D] input, dtype `dtype`.
 *   y      [B,H,S,D] output, same dtype; y == x (in place) is allowed, partial overlap is not.
 *   pos0   position of row s = 0; row s is rotated at position pos0 + s (pos0 >= 0).
 *   theta  RoPE base (> 0), e.g. 10000.
 *   D      even, 2 <= D <= 256; B, H, S >= 1.  fp8 values are rotated in float32 and rounded
 *          back to e5m2.
 * Errors: INVALID_ARG for null/misaligned pointers or bad sizes; CUDA on launch failure.
 */
ATTN_API attn_status_t rope_apply(const void* x, void* y, attn_dtype_t dtype, int B, int H, int S, int D,
                         int pos0, float theta, attn_stream_t stream);

/*
 * rope_apply_style — rope_apply with the pairing convention given (rope_apply is this call with
 * ATTN_ROPE_HALF_SPLIT), or its inverse (the _INVERSE styles).  Arguments and errors as
 * rope_apply; `style` outside the enum is INVALID_ARG.
 */
ATTN_API attn_status_t rope_apply_style(const void* x, void* y, attn_dtype_t dtype, int B, int H,
                               int S, int D, int pos0, float theta, attn_rope_style_t style,
                               attn_stream_t stream);

/*
 * attn_prefill_workspace_size — bytes of device workspace attn_prefill needs for these
 * arguments (dtype and rope as passed to attn_prefill).  Nonzero only where RoPE runs as
 * rotation passes before the attention kernel: rope = 1 with bf16 inputs and S >= 1024, with
 * the interleaved flag, or at D = 256; then (B*Hq + B*Hkv)*S*D bf16 values (Q rounded up to
 * 256 bytes, then K).  0 for invalid arguments.  Needs no device.
 */
ATTN_API size_t attn_prefill_workspace_size(int B, int Hq, int Hkv, int S, int D,
                                            attn_dtype_t dtype, int rope);

/*
 * attn_prefill — grouped-query attention over a whole prompt, one GPU.
 * Defines: softmax(scale * Q K^T + causal mask) V for Hq query heads sharing Hkv KV heads,
 * the causal GQA prefill of Lesson: shape adaptive attention negative 20260722 ("당시 조건")
 * and the Z/H/D attention workloads of the persistent-attention refactor page
 * ("性能ベンチマーク").
 *   q        [B,Hq,S,D]   k, v  [B,Hkv,S,D]   (dtype `dtype`)
 *   o        [B,Hq,S,D] bfloat16 output.
 *   lse      NULL or [B,Hq,S] float32: natural-log log-sum-exp of each row of scaled scores.
 *   q_scale, k_scale, v_scale: dequantisation factors (stored value * scale = real value);
 *            pass 1 for bf16 and for the per-tensor-scale-1 fp8 workloads.
 *   causal   0 or 1; causal hides key j from query i when j > i (S_q == S_kv).
 *   rope     0 = Q and K used as given.  1 and 2 rotate Q and K at positions pos0 + s:
 *            1 = the library's choice: bf16 prompts of S >= 1024 rotate Q and K once per call
 *                (rope_apply passes into the caller's workspace), then run attention without
 *                RoPE; shorter prompts and fp8 rotate both inside the kernel;
 *            2 = both inside the kernel as they are loaded (K once per query block that reads
 *                it; the fully fused form, measured beside the other).
 *            | ATTN_ROPE_FLAG_INTERLEAVED: pairs (2i, 2i+1); bf16 with rope = 1 only (always
 *                the rope_apply passes); fp8 or rope = 2 with the flag is UNSUPPORTED.
 *   workspace  device buffer of at least attn_prefill_workspace_size(B,Hq,Hkv,S,D,dtype,rope)
 *            bytes, 16-byte aligned (may be NULL when that size is 0); contents need no
 *            initialisation.  Calls that run at the same time (e.g. on two streams) need
 *            workspaces of their own.
 *   D in {64, 128, 256} (256: bf16 with rope 0 or 1 through the rotation passes, or fp8 with
 *   rope 0); Hq % Hkv == 0;
 *   S >= 1.  fp8 e5m2 inputs: P is rounded to e4m3 for the PV
 *   product; with rope = 1 (D = 128 only) Q and K are rotated into bf16 tiles inside the
 *   kernel (QK^T then runs in bf16, PV stays fp8), because rotated values re-rounded to fp8
 *   would exceed the fp8 error budget.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
ATTN_API attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                           attn_dtype_t dtype, float q_scale, float k_scale, float v_scale,
                           int B, int Hq, int Hkv, int S, int D, int causal, float softmax_scale,
                           int rope, float rope_theta, int pos0, void* workspace,
                           size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_prefill_backward — gradients of attn_prefill's attention: dQ, dK, dV.
 * Defines: the gradient of the softmax attention the pages fuse into serving kernels (the
 * operation of attn_prefill, differentiated by the chain rule; the pages describe only its
 * forward use).  With P = softmax(scale Q K^T + causal mask): dV = P^T dO, dS = P * (dO V^T -
 * rowsum(dO * O)), dQ = scale dS K, dK = scale dS^T Q; a KV head's dK, dV sum over the G query
 * heads that read it.
 *   q, k, v  [B,Hq,S,D], [B,Hkv,S,D] bf16 as the forward used them (rotated when its RoPE was
 *            on: the rotation's gradient is the inverse rotation, applied by the caller).
 *   o        [B,Hq,S,D] bf16 forward output;  lse  [B,Hq,S] float32 forward LSE (natural log).
 *   dout     [B,Hq,S,D] bf16, dL/dO.
 *   dq       [B,Hq,S,D] bf16;  dk, dv  [B,Hkv,S,D] bf16 (written, not accumulated).
 *   causal   0 or 1; softmax_scale <= 0 means 1/sqrt(D).  dtype ATTN_BF16 only; D in {64, 128}.
 *   workspace  device buffer of attn_prefill_backward_workspace_size(B, Hq, S, D) bytes, 16-byte
 *            aligned; no initialisation needed (fp32 row sums Delta, then the fp32 dQ
 *            accumulator that only the mma.sync path of attn_set_backward_path uses).
 * Errors: INVALID_ARG, UNSUPPORTED (fp8, other D), WORKSPACE, CUDA, NO_DEVICE.
 */
ATTN_API size_t attn_prefill_backward_workspace_size(int B, int Hq, int S, int D);
ATTN_API attn_status_t attn_prefill_backward(const void* q, const void* k, const void* v,
                                    const void* o, const float* lse, const void* dout, void* dq,
                                    void* dk, void* dv, attn_dtype_t dtype, int B, int Hq,
                                    int Hkv, int S, int D, int causal, float softmax_scale,
                                    void* workspace, size_t workspace_bytes,
                                    attn_stream_t stream);

/*
 * attn_set_backward_path — which kernels attn_prefill_backward runs.  0: the default (2);
 * 1: warp-level mma.sync kernels (a dK/dV kernel that adds dQ into an fp32 accumulator with
 * atomics, then a conversion pass); 2: tcgen05 kernels with TMEM accumulators (a dK/dV kernel
 * over 128-key tiles and a dQ kernel over 128-row query tiles, no atomics; only the row-sum
 * part of the workspace is used).  Results agree up to rounding order.  Process-wide; set it
 * only while no other thread runs a backward.
 * Errors: INVALID_ARG (path outside 0..2).
 */
ATTN_API attn_status_t attn_set_backward_path(int path);

/*
 * attn_prefill_chunk_workspace_size — bytes of device workspace attn_prefill_chunk needs:
 * B*Hq*Sq*D bf16 values (rounded up to 256 bytes) for bf16 with rope = 1 (the chunk's queries
 * rotated once), else 0.  0 for invalid arguments.  Needs no device.
 */
ATTN_API size_t attn_prefill_chunk_workspace_size(int B, int Hq, int Sq, int D,
                                                  attn_dtype_t dtype, int rope);

/*
 * attn_prefill_chunk — one chunk of a prompt against a static cache (chunked prefill).
 * Defines: filling a static cache a chunk at a time before the decode steps (Fixed-budget
 * decode audit — 2026-09-11, "Setup and interpretation": chunked prefill with chunks of 32).
 * The chunk's Sq queries are the last Sq of Skv tokens: query row i sits at position
 * Skv - Sq + i and attends keys 0 .. Skv - Sq + i (causal, aligned at the bottom-right corner
 * of the Sq x Skv score matrix; Sq == Skv is the ordinary causal prefill).
 *   q        [B,Hq,Sq,D] (dtype `dtype`).
 *   k, v     the first Skv rows of [B,Hkv,kv_pitch,D]: a cache of kv_pitch >= Skv rows per
 *            head holding the keys before the chunk followed by the chunk's own.  Keys are used
 *            as stored (a cache holds them already rotated); rows >= Skv are never read.
 *   o        [B,Hq,Sq,D] bfloat16.   lse  NULL or [B,Hq,Sq] float32 (natural log).
 *   rope     1: q rotated at positions pos0 + Skv - Sq + i (bf16: a rope_apply pass into the
 *            caller's workspace; fp8: inside the kernel, into bf16 tiles); 0: q as given.
 *            1 | ATTN_ROPE_FLAG_INTERLEAVED: pairs (2i, 2i+1), bf16 only (fp8: UNSUPPORTED).
 *   workspace  device buffer of at least attn_prefill_chunk_workspace_size(B,Hq,Sq,D,dtype,
 *            rope) bytes, 16-byte aligned (NULL allowed when that size is 0); no initialisation.
 *   1 <= Sq <= Skv <= kv_pitch; D in {64, 128, 256} (fp8 with rope = 1: D = 128 only); the other
 *   arguments as attn_prefill.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
ATTN_API attn_status_t attn_prefill_chunk(const void* q, const void* k, const void* v, void* o,
                                          float* lse, attn_dtype_t dtype, float q_scale,
                                          float k_scale, float v_scale, int B, int Hq, int Hkv,
                                          int Sq, int Skv, int kv_pitch, int D,
                                          float softmax_scale, int rope, float rope_theta,
                                          int pos0, void* workspace, size_t workspace_bytes,
                                          attn_stream_t stream);

/*
 * attn_set_prefill_tiles — the prefill's tile configuration, for the "one global configuration
 * versus per-shape choice" comparison the Lesson page (shape adaptive attention negative
 * 20260722, 다음에 기억할 것) asks every path to report.  q_tiles = 2: a work item is 256 query
 * rows (two 128-row Q tiles whose softmaxes alternate with each other's matrix products; the
 * default); 1: a work item is 128 rows (twice as many items, no alternation); 0 restores the
 * default.  Applies to every later attn_prefill / attn_prefill_chunk at D <= 128 (D = 256
 * always runs one tile per item).  Process-wide; set it only while no other thread launches a
 * prefill.  Results are the same in either configuration up to rounding order.
 * Errors: INVALID_ARG (q_tiles outside 0..2).
 */
ATTN_API attn_status_t attn_set_prefill_tiles(int q_tiles);

/*
 * attn_set_prefill_events — a measurement hook: while set, every attn_prefill and
 * attn_prefill_chunk call records `begin_event` on its stream just before the attention kernel
 * is enqueued and `end_event` just after it (the RoPE rotation passes that may precede it stay
 * outside the pair), so cudaEventElapsedTime gives that kernel's own time inside a longer
 * sequence of work.  The two are cudaEvent_t handles created by the caller (with timing
 * enabled); NULL, NULL clears the hook.  Process-wide: set it only while no other thread runs
 * a prefill.  Not for use during stream capture.  No operation of the pages.
 * Errors: INVALID_ARG (exactly one of the two NULL).
 */
ATTN_API attn_status_t attn_set_prefill_events(void* begin_event, void* end_event);

/*
 * attn_decode_workspace_size — bytes of device workspace attn_decode needs for these sizes
 * (split-KV partial outputs and their log-sum-exp).  May be 0.  Needs no device memory; uses
 * the current device's SM count (152 when no device is visible).
 */
ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int D, int Lmax);

/*
 * attn_decode — single-token grouped-query decode against a static KV cache.
 * Defines: the grouped split-score decode of Fixed-budget decode audit — 2026-09-11 ("Which
 * implementation was tested": static append cache; "Optimized full-model results": split
 * size 128), with split partials merged by log-sum-exp weights ("A: group-entry queries ...").
 *   q          [B,Hq,D]      the new token's query (un-rotated; rotated here when rope = 1, or
 *                            1 | ATTN_ROPE_FLAG_INTERLEAVED for the pairs (2i, 2i+1))
 *   k_cache    [B,Hkv,Lmax,D], v_cache [B,Hkv,Lmax,D]  keys stored ALREADY rotated.
 *   cache_len  DEVICE int32 [B]; sequence b attends keys 0 .. cache_len[b]-1 and its query
 *              sits at position cache_len[b].  Needs 1 <= cache_len[b] <= Lmax; a row with an
 *              out-of-range length gets O = 0, LSE = -inf and the device status DEVICE_ARG.
 *   o          [B,Hq,D] bfloat16.  lse: NULL or [B,Hq] float32.
 *   workspace  device buffer of at least attn_decode_workspace_size(B,Hq,Hkv,D,Lmax) bytes
 *              (may be NULL when that size is 0).  Contents need no initialisation.
 *   dtype      storage type of the caches: ATTN_BF16, or ATTN_FP8_E5M2 (D = 128 only; values
 *              are widened exactly to f16 for the products).  q is always bfloat16.
 *   D in {64, 128, 256}; Hq % Hkv == 0; Hq / Hkv <= 16.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
ATTN_API attn_status_t attn_decode(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* cache_len, int Lmax, void* o, float* lse,
                          attn_dtype_t dtype, int B, int Hq, int Hkv, int D, float softmax_scale,
                          int rope, float rope_theta, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream);

/*
 * attn_decode_noalloc — attn_decode for callers that cannot allocate device memory at call
 * time: a host that forbids allocation in its enqueue path (inference-engine plugins), a
 * process whose device memory is entirely owned by another allocator, or a latency-bound
 * serving loop that cannot afford an allocation's cost or implicit synchronisation.  It takes
 * the same arguments as attn_decode minus the workspace, computes the same result, and calls
 * no cudaMalloc, cudaFree or other allocating routine.  Caches must be bfloat16 (dtype
 * ATTN_BF16, D in {64, 128, 256}); an fp8 e5m2 cache returns ATTN_ERR_UNSUPPORTED.  The pages have no counterpart; this is
 * an interface convenience around the same kernels.
 *   Scratch: the split partials live in one file-scope device array of 2 MiB (2097152 bytes)
 *   that every GPU loading this library holds until the process exits.  A call whose
 *   attn_decode_workspace_size(B,Hq,Hkv,D,Lmax) exceeds 2 MiB returns ATTN_ERR_WORKSPACE
 *   without launching.  All calls share the array and it keeps the last call's contents; every
 *   slot a call reads is written earlier in the same call, so nothing needs clearing.  Calls
 *   whose execution overlaps on the GPU (e.g. on two streams) race on the array: serialise them.
 *   Set-up: the first call on each device resolves the array's device address with
 *   cudaGetSymbolAddress (which may load the library's device code on that device); make that
 *   first call before any stream capture.
 *   RoPE: rope = 1 needs the cos/sin table for (D, rope_theta) covering position Lmax to exist
 *   already (attn_rope_table_reserve(D, rope_theta, Lmax) or an earlier attn_decode call);
 *   otherwise ATTN_ERR_WORKSPACE, because building it would allocate.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA, NO_DEVICE (as attn_decode otherwise).
 */
ATTN_API attn_status_t attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* cache_len, int Lmax, void* o, float* lse,
                                  attn_dtype_t dtype, int B, int Hq, int Hkv, int D,
                                  float softmax_scale, int rope, float rope_theta,
                                  attn_stream_t stream);

/*
 * attn_set_decode_splits — the "one global configuration versus per-shape choice" comparison
 * the Lesson page (shape adaptive attention negative 20260722, 다음에 기억할 것) asks every
 * path to report, for the split-KV decode.  nsplit > 0: every later attn_decode,
 * attn_decode_append and attn_decode_noalloc call (and their workspace sizes) splits each
 * sequence's keys into nsplit chunks (at most one per 64-key tile) instead of the per-shape
 * planner's choice; 0 restores the planner (the default).  Process-wide; set it only while no
 * other thread plans a decode.
 * Errors: INVALID_ARG (nsplit < 0 or > 1024).
 */
ATTN_API attn_status_t attn_set_decode_splits(int nsplit);

/*
 * attn_decode_append — one decode step whose token joins the cache (growing decode).
 * Defines: the decode steps of a static append cache that grows by one row per step, run as
 * growing CUDA graphs (Fixed-budget decode audit — 2026-09-11, "Which implementation was
 * tested" and "Setup and interpretation"), with the current token merged into the
 * cached-history result ("A: group-entry queries and one joint history scan": the current
 * token's weight is the logistic function of its score minus the history log-sum-exp).
 * Sequence b's query and new key sit at position L = cache_len[b] (read on the device):
 *   1. the history: attn_decode of q over cache rows 0 .. L-1;
 *   2. k_new rotated at L (when rope = 1, or 1 | ATTN_ROPE_FLAG_INTERLEAVED for the pairs
 *      (2i, 2i+1), the convention of the cached keys) and v_new are written to cache row L (bf16), and each
 *      query row merges that key into its history output;
 *   3. cache_len[b] becomes L + 1.
 * The result is attention over the L + 1 keys.  Because positions and lengths live on the
 * device, one captured CUDA graph of this call serves every later step.
 *   q        [B,Hq,D] bf16 (rotated at L inside when rope = 1).
 *   k_new, v_new [B,Hkv,D] bf16, the current token's key (unrotated) and value.
 *   k_cache, v_cache [B,Hkv,Lmax,D] bf16, written at row L.
 *   cache_len device int32 [B], 1 <= cache_len[b] <= Lmax - 1, incremented.
 *   o        [B,Hq,D] bf16.   lse  NULL or [B,Hq] float32 (natural log, over the L + 1 keys).
 *   workspace  device buffer of attn_decode_append_workspace_size() bytes (never zero).
 *   dtype    ATTN_BF16 only; D in {64, 128, 256}; Hq / Hkv <= 16.
 * Device errors: a cache_len outside [1, Lmax - 1] sets DEVICE_ARG; that sequence's row is not
 * written, its length not changed, and its output is the history result (zero when L < 1).
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
ATTN_API size_t attn_decode_append_workspace_size(int B, int Hq, int Hkv, int D, int Lmax);
ATTN_API attn_status_t attn_decode_append(const void* q, const void* k_new, const void* v_new,
                                          void* k_cache, void* v_cache, int32_t* cache_len,
                                          int Lmax, void* o, float* lse, attn_dtype_t dtype,
                                          int B, int Hq, int Hkv, int D, float softmax_scale,
                                          int rope, float rope_theta, void* workspace,
                                          size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_latent_workspace_size — bytes of workspace attn_decode_latent needs.
 */
ATTN_API size_t attn_decode_latent_workspace_size(int B, int H, int Lmax);

/*
 * attn_decode_latent — absorbed latent (MLA-style) single-token decode.
 * Defines: the MLA decode of Fixed-budget decode audit — 2026-09-11 ("Which implementation was
 * tested": 448-dimensional latent + 64-dimensional RoPE), with W_UK already absorbed into q and
 * W_UV applied by the caller to the latent output.
 *   q          [B,H,512] bfloat16: 448 absorbed-latent dims then 64 RoPE dims (the RoPE dims
 *              are rotated at position cache_len[b] when rope = 1; pairs (i, i + 32) of those
 *              64 dims, or (2i, 2i+1) with rope = 1 | ATTN_ROPE_FLAG_INTERLEAVED).
 *   c_cache    [B,Lmax,512] of `dtype` (ATTN_BF16, or ATTN_FP8_E5M2 at half the bytes; every
 *              e5m2 value is an exact f16, so the kernel runs f16 MMAs on the widened cache and
 *              the query in f16): per token the 448-dim latent then the 64-dim rotated key.
 *              Scores use all 512 dims; values are the first 448 dims.
 *   cache_len  DEVICE int32 [B], as in attn_decode.
 *   o          [B,H,448] bfloat16.  lse: NULL or [B,H] float32.
 *   H <= 16 (all heads of a sequence share one MMA tile); B <= 2048.  softmax_scale <= 0 means
 *   1/sqrt(512).  The key tiles of all sequences are split evenly over the SMs, so a sequence
 *   may be computed in pieces that a second kernel merges; the workspace holds those pieces.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
ATTN_API attn_status_t attn_decode_latent(const void* q, const void* c_cache,
                                          const int32_t* cache_len, int Lmax, void* o, float* lse,
                                          attn_dtype_t dtype, int B, int H, float softmax_scale,
                                          int rope, float rope_theta, void* workspace,
                                          size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_rope_table_reserve — build (if needed) the cos/sin table for head dim D and base theta
 * covering positions 0 .. max_pos on the current device.  Allocates and copies synchronously.
 * Call before timing or stream capture.  Errors: INVALID_ARG, CUDA, NO_DEVICE.
 */
ATTN_API attn_status_t attn_rope_table_reserve(int D, float theta, int max_pos);

/*
 * attn_get_device_status — synchronise `stream`, then return (in *status_out) the device status
 * word the kernels set since the last call (ATTN_OK, ATTN_ERR_TIMEOUT or ATTN_ERR_DEVICE_ARG)
 * and clear it.  The return value reports failures of this call itself.
 */
ATTN_API attn_status_t attn_get_device_status(attn_stream_t stream, int* status_out);

/*
 * attn_selftest_wait_timeout — a self-test of the kernels' bounded waits: one warp waits on a
 * shared-memory mbarrier that nothing ever arrives at, through the same bounded-wait routine
 * every attention kernel uses, with a limit of `timeout_us` microseconds instead of the
 * kernels' 2 s.  The wait gives up, the kernel sets ATTN_ERR_TIMEOUT in the device status word
 * (attn_get_device_status then reports it once) and returns; the CUDA context stays usable.
 * No operation of the pages; it lets a caller or a test check the failure path without
 * faulting or hanging the GPU.
 *   timeout_us  1 .. 2000000.
 * Errors: INVALID_ARG, NO_DEVICE, CUDA.
 */
ATTN_API attn_status_t attn_selftest_wait_timeout(unsigned int timeout_us, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
