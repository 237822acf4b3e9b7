/*
 * ps.h -- C ABI of libps.so: Prefix-Sliding attention for NVIDIA B300 (sm_103a).
 *
 * Prefix-Sliding attention: the query at absolute position p attends to key j
 * iff  j <= p  and  (j < P  or  j > p - W): a fixed task prefix of P tokens
 * plus the last W positions, the current token included.  Keys in between are
 * evicted, so at most P + W keys are ever cached, and positions keep counting
 * up ("Continue PE") so RoPE'd keys stay valid after eviction.
 *   Sources: njhaofan.com article, section "PrefixSliding如何丢掉中间Token？";
 *   "Prefix Sliding：面向高效 test-time scaling 的前缀滑动方法"
 *   (papers.ananclaw.com), sections "核心方法" and "伪代码";
 *   "Prefix Sliding for efficient test-time scaling" (agihunt.info), the
 *   paragraphs on the 4,196-token cap, on Continue PE and on the two-level
 *   tile filter of the FlashAttention kernel.
 *
 * Conventions for every call
 *   - Pointers marked "device" are CUDA device pointers owned by the caller
 *     (e.g. torch tensors).  The library never allocates or frees them; only
 *     a decode-graph handle (ps_decode_graph_create) keeps them, until its
 *     destroy call.
 *   - "bf16" is IEEE bfloat16 (__nv_bfloat16), stored row-major as documented.
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and never synchronises, except
 *     ps_decode_graph_step when asked to.  The library keeps no state between
 *     calls and is thread-safe, with two exceptions: ps_decode_noalloc uses a
 *     scratch array inside the library that all its calls share, and a
 *     decode-graph handle is caller-owned state that one caller steps at a
 *     time (see their comments).
 *   - Host-side checks run before any launch and return a ps_status_t.
 *     Checks that need device data (per-sequence prefix lengths, positions,
 *     pool bases) run inside the kernels: a failing sequence is skipped and
 *     PS_DEV_* bits are OR-ed into the optional device status word, which
 *     ps_check_device_status() reads back.  Kernels never trap.
 *   - RoPE: half-split ("NeoX") rotation, element i with element i + D/2, by
 *     the angle pos * theta^(-2i/D), at the absolute position.  The angle is
 *     reduced modulo one turn in 64-bit fixed point, so positions up to 2^31
 *     keep full precision.  Rotated Q and K are rounded to bf16.
 *   - Softmax scale is the `scale` argument (normally 1/sqrt(D)); LSE is the
 *     natural log of sum_j exp(scale * q.k_j).  Query head h reads KV head
 *     h / (Hq / Hkv).
 */
#ifndef PS_H_
#define PS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ps_status_t {
  PS_OK = 0,
  PS_ERR_INVALID_ARGUMENT = 1, /* null pointer, W < 1, P < 0, Hq % Hkv != 0, sizes */
  PS_ERR_UNSUPPORTED = 2,      /* head_dim not in {64, 128}, group size, tile size */
  PS_ERR_ALIGNMENT = 3,        /* a tensor pointer is not 16-byte aligned          */
  PS_ERR_WORKSPACE = 4,        /* workspace missing or too small                   */
  PS_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed             */
  PS_ERR_DEVICE = 6            /* ps_check_device_status found flags set           */
} ps_status_t;

/* Bits a kernel ORs into the device status word. */
#define PS_DEV_BAD_PREFIX 0x1  /* prefix_len < 0 or > prefix_max                  */
#define PS_DEV_BAD_POS    0x2  /* a position < 0                                   */
#define PS_DEV_BAD_SLOT   0x4  /* slot_base/capacity outside the pool              */
#define PS_DEV_TIMEOUT    0x8  /* a bounded wait on an mbarrier gave up            */
#define PS_DEV_BAD_RUN    0x10 /* cu_tokens not increasing / outside [0, n_tokens] */
#define PS_DEV_BAD_SEQ    0x20 /* a sequence index outside [0, nseq)               */

/* Human-readable name of a status code (static string). */
const char* ps_status_string(ps_status_t status);

/*
 * The bounded KV cache ("伪代码" section: total cache size is the constant
 * prefix_len + W).  Position pos of sequence s lives in its logical slot
 *     slot(pos) = pos                       if pos < P_s
 *               = P_s + (pos - P_s) mod W   otherwise,
 * so prefix slots never move and each window slot is overwritten exactly
 * when its previous occupant leaves the window.  After positions 0..p are
 * appended, slots [0, min(p+1, P_s+W)) hold exactly the keys query p may see.
 * Logical slot -> pool row:
 *   block_table == NULL: contiguous, row = slot_base[s] + slot; sequence s
 *     owns rows [slot_base[s], slot_base[s] + capacity).
 *   block_table != NULL: paged, as in paged-attention serving engines (the
 *     papers.ananclaw.com explainer, section "对工程落地的启发", calls the
 *     method orthogonal to paged KV memory management); row =
 *     block_table[s * blocks_per_seq + slot / block_size] * block_size
 *     + slot % block_size.  slot_base is not read and may be NULL.  Only the
 *     blocks covering slots [0, P_s + W) are read or written.  A block id
 *     outside the pool sets PS_DEV_BAD_SLOT; the access goes to block 0 or is
 *     skipped, never outside the pool.
 */
typedef struct ps_cache_desc {
  void* k_pool;              /* device bf16 [total_slots, n_kv_heads, head_dim], RoPE'd K */
  void* v_pool;              /* device bf16 [total_slots, n_kv_heads, head_dim], V        */
  const int64_t* slot_base;  /* device [nseq]: first pool row of each sequence (contiguous) */
  const int32_t* prefix_len; /* device [nseq]: P of each sequence, 0 <= P <= prefix_max   */
  int32_t* status;           /* device int32 status word, or NULL                         */
  int64_t total_slots;       /* rows in each pool                                          */
  int32_t nseq;              /* sequences described                                        */
  int32_t n_kv_heads;        /* Hkv >= 1                                                   */
  int32_t head_dim;          /* D: 64 or 128                                               */
  int32_t window;            /* W >= 1                                                     */
  int32_t capacity;          /* rows reserved per sequence, >= prefix_max + window         */
  int32_t prefix_max;        /* host bound on every prefix_len                             */
  double rope_theta;         /* RoPE base, > 0                                             */
  const int32_t* block_table; /* device int32 [nseq, blocks_per_seq], or NULL (contiguous) */
  int32_t block_size;        /* paged: slots per block, a multiple of 16                   */
  int32_t blocks_per_seq;    /* paged: >= ceil(capacity / block_size)                      */
  int32_t pe_mode;           /* PS_PE_CONTINUE (0) or PS_PE_RESET (1); see below           */
} ps_cache_desc;

/*
 * Position encoding of the cached keys (agihunt.info paragraph on position
 * encodings; njhaofan.com section "PrefixSliding如何丢掉中间Token？").
 *   PS_PE_CONTINUE: positions keep climbing; a query at p sees every cached
 *     key at its absolute position (the pages' default).
 *   PS_PE_RESET: the cache is renumbered in order for each query: prefix keys
 *     0..P-1, then the window keys, oldest first, and the query as the newest
 *     entry (L - 1, with L the keys it sees).  The pages do not give the rule;
 *     this is the plainest one.  Keys stay stored rotated at their absolute
 *     positions; window keys keep their distance to the query, so only the
 *     prefix keys see a different query rotation: at L - 1 = min(p, P + W - 1).
 *     ps_decode (from the cache's pe_mode) and ps_prefill (its pe_mode
 *     argument) honour it; ps_kv_append stores keys the same way in both
 *     modes; ps_prefill_backward differentiates Continue PE only.
 */
#define PS_PE_CONTINUE 0
#define PS_PE_RESET 1

/*
 * ps_ring_slots: slot(pos) of the formula above for n independent entries.
 *   pos, prefix_len : device int32 [n]; window >= 1; slot : device int32 [n].
 * Entries with pos < 0 or prefix_len < 0 get slot -1.
 */
ps_status_t ps_ring_slots(const int32_t* pos, const int32_t* prefix_len, int32_t window,
                          int32_t* slot, int64_t n, void* stream);

/*
 * ps_kv_append: rotate new keys at their absolute positions (Continue PE:
 * agihunt.info paragraph on position encodings) and store K and V into the
 * ring ("PrefixSliding如何丢掉中间Token？": older middle tokens leave the cache).
 *   k, v      : device bf16 [n_tokens, n_kv_heads, head_dim], raw (un-rotated) K, V.
 *   Tokens come in runs: run r covers tokens [cu_tokens[r], cu_tokens[r+1]) of
 *   sequence seq_idx[r], at consecutive positions pos0[r], pos0[r]+1, ...
 *   seq_idx, pos0 : device int32 [nrun]; cu_tokens : device int32 [nrun+1],
 *   cu_tokens[0] = 0, non-decreasing, cu_tokens[nrun] = n_tokens.
 *   A run longer than W writes only its survivors (prefix positions and the
 *   last W positions), so the result equals appending one token at a time.
 *   Two runs of one sequence in one call: undefined.
 * Decode appends one token per sequence: nrun = nseq, cu_tokens = 0..nseq.
 */
ps_status_t ps_kv_append(const ps_cache_desc* cache, const int32_t* seq_idx,
                         const int32_t* pos0, const int32_t* cu_tokens, int32_t nrun,
                         const void* k, const void* v, int64_t n_tokens, void* stream);

/*
 * ps_decode_workspace_size: bytes of device workspace ps_decode needs for
 * nseq sequences on the current device (split-KV partial results).
 */
ps_status_t ps_decode_workspace_size(int32_t nseq, int32_t n_q_heads, int32_t n_kv_heads,
                                     int32_t head_dim, size_t* bytes);

/*
 * ps_decode: one query token per sequence against the prefix and window keys
 * in the cache (the generation step of the "伪代码" section).
 *   q   : device bf16 [nseq, n_q_heads, head_dim], raw (rotated here at pos[s]).
 *   pos : device int32 [nseq], absolute position of each query; its own K/V
 *         must already be appended.  Sequence s reads slots
 *         [0, min(pos[s]+1, P_s+W)).
 *   out : device bf16 [nseq, n_q_heads, head_dim]; lse : device fp32 [nseq, n_q_heads].
 *   workspace : device, >= ps_decode_workspace_size bytes, 256-byte aligned.
 * Work is split evenly over all SMs in 16-slot tiles regardless of per-sequence
 * length (no host synchronisation), then a second kernel merges the partial
 * softmax results by their log-sum-exp.  n_q_heads / n_kv_heads in {1,2,4,8}.
 */
ps_status_t ps_decode(const ps_cache_desc* cache, const void* q, const int32_t* pos,
                      int32_t n_q_heads, float scale, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * The two launches of ps_decode, callable on their own (same arguments and
 * workspace): ps_decode_partial streams the K/V tiles and writes the partial
 * softmax records into the workspace; ps_decode_combine merges them into out
 * and lse.  Between the two calls the workspace must not be reused.
 */
ps_status_t ps_decode_partial(const ps_cache_desc* cache, const void* q, const int32_t* pos,
                              int32_t n_q_heads, float scale, void* workspace,
                              size_t workspace_bytes, void* stream);
ps_status_t ps_decode_combine(const ps_cache_desc* cache, int32_t n_q_heads, void* out, float* lse,
                              const void* workspace, size_t workspace_bytes, void* stream);

/*
 * ps_decode_append: one whole decode step in one call, the equivalent of
 * ps_kv_append of one token per sequence (run s: sequence s, position pos[s])
 * followed by ps_decode with the same positions, without the separate append
 * launch.  The warp whose tile holds a sequence's new slot finds the slot's
 * previous occupant there; it puts the new token's K, rotated at pos[s] with
 * the same arithmetic as ps_kv_append, and its V in its place, in the tile it
 * reads and in the pool, so the cache afterwards holds the same bits as after
 * the two separate calls, and out / lse are the same bits too.
 *   k, v : device bf16 [nseq, n_kv_heads, head_dim], raw (un-rotated) K and V of
 *          the new tokens, 16-byte aligned.
 *   Other arguments, workspace and errors: as ps_decode.  A sequence the device
 *   checks refuse is neither appended nor attended (out 0, lse -inf).
 */
ps_status_t ps_decode_append(const ps_cache_desc* cache, const void* q, const void* k,
                             const void* v, const int32_t* pos, int32_t n_q_heads, float scale,
                             void* out, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * ps_decode_noalloc: ps_decode without a caller-supplied workspace, for
 * callers that cannot allocate device memory when they decode -- a host that
 * has no allocator of its own (plain C linking this library), code that runs
 * while a caching allocator is locked or shutting down, or a server that
 * reserves all its memory at start-up and forbids allocation during
 * generation.  The pages have no counterpart to this call; it is a packaging
 * choice.
 *   Arguments, outputs and numerics are those of ps_decode.  The scratch is a
 *   fixed 4 MiB device array inside this library (every GPU that loads the
 *   library holds it until the process exits); the call allocates and frees
 *   nothing.  It returns PS_ERR_WORKSPACE when ps_decode_workspace_size for
 *   these shapes exceeds 4 MiB; 4 MiB holds, on a 148-SM B300, 256 sequences
 *   at Hkv = 8, head_dim 128 and two query heads per KV head.
 *   The first call on each device looks up the array's device address with
 *   that device current (and again if the device's context has been
 *   destroyed and re-created since); make that first call before any stream
 *   capture.  All calls share the one array and nothing in it needs to start
 *   at zero: every call rewrites the per-sequence tile counts, segment
 *   bounds and partial records it later reads.  Calls whose kernels overlap
 *   on the GPU (several streams, or threads on one device) race on the
 *   array, so serialise them.
 */
ps_status_t ps_decode_noalloc(const ps_cache_desc* cache, const void* q, const int32_t* pos,
                              int32_t n_q_heads, float scale, void* out, float* lse,
                              void* stream);

/*
 * Decode-step executor: the generation loop of the "伪代码" section (one step
 * per new token: append its K/V, attend, hand the output on) for a caller whose
 * new tokens arrive from and whose outputs go back to host memory.  A step's
 * inputs travel as one packed input block and its results as one packed result
 * block, and ps_decode_graph_step moves the block in, runs ps_decode_append
 * from a CUDA graph built once, and moves the results out, in one call.  The
 * pages have no counterpart; it is a packaging of ps_decode_append.
 *
 * ps_decode_step_layout_get: byte offsets of the views in the two blocks for
 * nseq sequences; each view starts on a 256-byte boundary:
 *   input block  = q [nseq, n_q_heads, D] bf16 raw | k [nseq, Hkv, D] bf16 raw
 *                | v [nseq, Hkv, D] bf16 | pos [nseq] int32
 *   result block = out [nseq, n_q_heads, D] bf16 | lse [nseq, n_q_heads] fp32
 * in_bytes / res_bytes: the blocks' sizes (each view's size rounded up to 256).
 * Errors: null layout, nseq or heads < 1, Hq % Hkv != 0 -> PS_ERR_INVALID_ARGUMENT;
 * head_dim not 64 or 128 -> PS_ERR_UNSUPPORTED.
 */
typedef struct ps_decode_step_layout {
  size_t q_off, k_off, v_off, pos_off, in_bytes;
  size_t out_off, lse_off, res_bytes;
} ps_decode_step_layout;

ps_status_t ps_decode_step_layout_get(int32_t nseq, int32_t n_q_heads, int32_t n_kv_heads,
                                      int32_t head_dim, ps_decode_step_layout* layout);

/* Opaque handle of one captured decode step. */
typedef struct ps_decode_graph ps_decode_graph;

/*
 * ps_decode_graph_create: capture one ps_decode_append on `cache` into a CUDA
 * graph and instantiate it, on the current device.
 *   cache : the ring the step appends to and reads; the descriptor's values
 *     (pools, tables, prefix lengths pointer, W, P bound, pe_mode ...) are
 *     copied at capture, so later steps use them as they were here.
 *   inp, res : device blocks laid out by ps_decode_step_layout_get for
 *     (cache->nseq, n_q_heads, cache->n_kv_heads, cache->head_dim), 256-byte
 *     aligned, owned by the caller and kept alive (with cache's buffers and
 *     the workspace) until ps_decode_graph_destroy.
 *   workspace : as for ps_decode_append (ps_decode_workspace_size bytes).
 *   graph : receives the handle.
 * The capture runs on a private stream and launches nothing: the cache is not
 * touched until the first step.  The handle owns the graph and its
 * instantiation (driver resources, no caller memory).  Errors: as
 * ps_decode_append's host checks, a null or misaligned block or a null
 * `graph` -> PS_ERR_INVALID_ARGUMENT / PS_ERR_ALIGNMENT, a failed capture or
 * instantiation -> PS_ERR_CUDA; on error *graph is NULL.
 */
ps_status_t ps_decode_graph_create(const ps_cache_desc* cache, int32_t n_q_heads, float scale,
                                   void* inp, void* res, void* workspace, size_t workspace_bytes,
                                   ps_decode_graph** graph);

/*
 * ps_decode_graph_step: one decode step, in order on `stream` (which must
 * belong to the graph's device; NULL = that device's legacy default stream):
 *   1. host_in != NULL: copy in_bytes from host_in into the input block;
 *      NULL: the caller has filled the input block on the device;
 *   2. launch the graph (ps_decode_append);
 *   3. host_res != NULL: copy res_bytes of the result block into host_res.
 * sync != 0: wait for the stream before returning, so host_res holds the
 * step's results.  Host buffers should be page-locked (pinned) for the copies
 * to run asynchronously; with pageable memory they still complete, staged by
 * the driver.  A handle is stepped by one caller at a time (steps on
 * different streams would race on the blocks).  Errors: null graph or
 * another device current -> PS_ERR_INVALID_ARGUMENT; a failed copy, launch or
 * synchronisation -> PS_ERR_CUDA.  Device-side refusals are reported through
 * the cache's status word, as for ps_decode_append.
 */
ps_status_t ps_decode_graph_step(ps_decode_graph* graph, const void* host_in, void* host_res,
                                 int32_t sync, void* stream);

/* ps_decode_graph_destroy: release the handle (NULL is a no-op).  Steps in
 * flight must have completed. */
ps_status_t ps_decode_graph_destroy(ps_decode_graph* graph);

/*
 * ps_prefill_workspace_size: device workspace for ps_prefill (rotated Q and K,
 * with a ring the gathered cached keys and values, and under Reset PE the
 * query rotated at its renumbered position).
 *   ring_rows_max : 0 without a ring, else the ring's prefix_max + window.
 *   pe_mode : PS_PE_CONTINUE or PS_PE_RESET, as passed to ps_prefill.
 */
ps_status_t ps_prefill_workspace_size(int32_t batch, int32_t seqlen, int32_t n_q_heads,
                                      int32_t n_kv_heads, int32_t head_dim,
                                      int32_t ring_rows_max, int32_t pe_mode, size_t* bytes);

/*
 * ps_prefill: tiled forward of Prefix-Sliding attention for a chunk of
 * `seqlen` tokens per batch row (prompt prefill, chunked extend, and the
 * truncated-backprop training forward of the agihunt.info paragraph on RL).
 * Tiles that hold no admitted (query, key) pair are skipped; tiles that hold
 * some but not all are masked element by element; the rest run unmasked
 * (agihunt.info paragraph on the two-level filter; njhaofan.com section
 * "PrefixSliding如何丢掉中间Token？").
 *   q : device bf16 [batch, seqlen, n_q_heads, head_dim]; k, v : device bf16
 *       [batch, seqlen, n_kv_heads, head_dim]; raw, rotated here.
 *   q_start : device int32 [batch]: absolute position of the chunk's first token;
 *       0 <= q_start and q_start + seqlen <= 2^31 - 1 (a negative value sets
 *       PS_DEV_BAD_POS; that row's outputs are then undefined).
 *   prefix_len : device int32 [batch]: P of each row.
 *   pe_mode : PS_PE_CONTINUE, or PS_PE_RESET: prefix keys are scored with the
 *       query rotated at min(p, P + W - 1) instead of p (see PS_PE_RESET); must
 *       equal ring->pe_mode when a ring is given.
 *   ring == NULL: the keys are the chunk's own tokens.
 *   ring != NULL: the keys are the ring's live entries of sequence ring_seq[b]
 *       (positions < q_start[b], as left by ps_kv_append) followed by the
 *       chunk; ring_seq : device int32 [batch] (NULL = identity), and
 *       prefix_len must equal the ring's prefix_len of that sequence.
 *   out : device bf16 [batch, seqlen, n_q_heads, head_dim];
 *   lse : device fp32 [batch, n_q_heads, seqlen] (natural log).
 *   status : device int32 word or NULL.
 * Uses tcgen05 tensor cores with TMEM accumulators.  head_dim 64 or 128.
 */
ps_status_t ps_prefill(const void* q, const void* k, const void* v, int32_t batch,
                       int32_t seqlen, const int32_t* q_start, const int32_t* prefix_len,
                       int32_t window, int32_t n_q_heads, int32_t n_kv_heads,
                       int32_t head_dim, float scale, double rope_theta, int32_t pe_mode,
                       const ps_cache_desc* ring, const int32_t* ring_seq, void* out,
                       float* lse, void* workspace, size_t workspace_bytes,
                       int32_t* status, void* stream);

/*
 * ps_prefill_backward_workspace_size: device workspace for ps_prefill_backward:
 * rotated Q and K (bf16), and per (batch row, query head, row rounded up to 128)
 * the pair {LSE * log2(e), D = rowsum(dO * O)} (fp32).  Errors: null `bytes`,
 * batch / seqlen / heads < 1 or Hq % Hkv != 0 -> PS_ERR_INVALID_ARGUMENT;
 * head_dim not 64 or 128 -> PS_ERR_UNSUPPORTED.
 */
ps_status_t ps_prefill_backward_workspace_size(int32_t batch, int32_t seqlen, int32_t n_q_heads,
                                               int32_t n_kv_heads, int32_t head_dim,
                                               size_t* bytes);

/*
 * ps_prefill_backward: gradients of ps_prefill without a ring (the
 * truncated-backprop training step: "Prefix Sliding for efficient test-time
 * scaling", agihunt.info, paragraph on RL, back-propagates through the last
 * 4W tokens under the same mask).
 *   q, k, v, q_start, prefix_len, window, heads, scale, rope_theta: as given
 *     to ps_prefill (without a ring; q_start within [0, 2^31 - 1 - seqlen], not
 *     checked here); out (bf16 [batch, seqlen, n_q_heads, head_dim]) and lse
 *     (fp32 [batch, n_q_heads, seqlen]) are its results; d_out: bf16 like out.
 *   fwd_workspace : NULL, or the workspace of that ps_prefill call (Continue
 *     PE, no ring, same arguments), still holding the rotated Q and K it wrote
 *     at its start; the backward then reads them from there instead of
 *     rotating Q and K again (256-byte aligned; only read).
 *   dq : device fp32 [batch, seqlen, n_q_heads, head_dim], gradient of raw q;
 *   dk, dv : device fp32 [batch, seqlen, n_kv_heads, head_dim] (summed over the
 *     query heads of each group).  The rotation is differentiated exactly; the
 *     bf16 rounding of the rotated q and k passes gradients straight through.
 *   Probabilities and dS enter the tensor-core products as bf16.
 *   workspace : device, 256-byte aligned, at least the size above; the caller
 *     owns it and may reuse it once the call's stream work has completed.
 *   status : device int32 word or NULL; PS_DEV_TIMEOUT if a bounded wait gave up.
 * Errors (host, before any launch): a null pointer, batch / seqlen / window /
 * heads < 1, Hq % Hkv != 0, scale <= 0 or rope_theta <= 0 -> PS_ERR_INVALID_ARGUMENT;
 * head_dim not 64 or 128 -> PS_ERR_UNSUPPORTED; a tensor not 16-byte aligned ->
 * PS_ERR_ALIGNMENT; workspace missing, misaligned or too small -> PS_ERR_WORKSPACE;
 * a failed launch -> PS_ERR_CUDA.  Two launches on `stream` (a pre-pass, then one
 * grid of dK/dV and dQ CTAs using 230,656 bytes of shared memory and all 512 TMEM
 * columns per CTA); asynchronous, no synchronisation.
 */
ps_status_t ps_prefill_backward(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* d_out, int32_t batch,
                                int32_t seqlen, const int32_t* q_start, const int32_t* prefix_len,
                                int32_t window, int32_t n_q_heads, int32_t n_kv_heads,
                                int32_t head_dim, float scale, double rope_theta,
                                const void* fwd_workspace, float* dq, float* dk, float* dv,
                                void* workspace, size_t workspace_bytes, int32_t* status,
                                void* stream);

/*
 * Tile geometry used by ps_prefill for one batch row: nq x nk tiles of
 * bm x bn.  with_ring != 0 counts the ring rows a chunk starting at q_start
 * would gather ((min(P, q_start) prefix keys plus the window keys before q_start).
 */
ps_status_t ps_prefill_tile_grid(int32_t seqlen, int32_t q_start, int32_t prefix_len,
                                 int32_t window, int32_t with_ring, int32_t bm, int32_t bn,
                                 int32_t* nq, int32_t* nk);

/*
 * ps_prefill_tile_classes: the class ps_prefill assigns to each (query tile,
 * key tile) of one batch row: 0 = skip, 1 = partial (masked), 2 = full.
 *   out : device uint8 [nq * nk] (row-major by query tile), sizes from
 *   ps_prefill_tile_grid with the same arguments.  Any bm, bn >= 1.
 */
ps_status_t ps_prefill_tile_classes(int32_t seqlen, int32_t q_start, int32_t prefix_len,
                                    int32_t window, int32_t with_ring, int32_t bm, int32_t bn,
                                    uint8_t* out, void* stream);

/*
 * ps_device_code_version: the compute capability the library's kernels were
 * compiled for, as the CUDA runtime reports it for a loaded kernel on the
 * current device (major * 10 + minor: 103 for sm_103a).  Needs a device;
 * PS_ERR_CUDA if none can be used, PS_ERR_INVALID_ARGUMENT for a null pointer.
 */
ps_status_t ps_device_code_version(int32_t* version);

/*
 * ps_test_force_wait_timeout: test hook for the kernels' bounded waits.  Every
 * wait of a kernel on a copy, a tensor-core product or another role gives up
 * after a time limit (2 s), sets PS_DEV_TIMEOUT in the status word, lets the
 * copies and products it has already issued finish (each wait for them again
 * bounded) and returns, so the context stays usable.  With enable = 1, the
 * decode partial kernel, the prefill tile kernels and the backward kernel
 * launched afterwards use wait_limit_ns (1e3 .. 2e9) as that limit, and CTA 0
 * of each skips its first streamed copy, so one wait is sure to run out: the
 * call sets PS_DEV_TIMEOUT and its results are undefined.  enable = 0 restores the defaults.  Process-wide
 * and not synchronised with calls in flight: for tests only.
 */
ps_status_t ps_test_force_wait_timeout(int32_t enable, int64_t wait_limit_ns);

/*
 * ps_check_device_status: synchronously copy the device status word to
 * *host_flags.  Returns PS_ERR_DEVICE if any flag is set, PS_OK otherwise.
 * Test and debugging use; it synchronises the device.
 */
ps_status_t ps_check_device_status(const int32_t* status, int32_t* host_flags);

#ifdef __cplusplus
}
#endif
#endif /* PS_H_ */
