/*
 * hikv — importance-aware, budgeted KV-cache decode step on one GPU (sm_103a).
 *
 * C ABI.  Every tensor argument is a plain pointer plus sizes; no C++ or torch
 * types cross this boundary.  All tensor pointers are DEVICE pointers owned
 * by the caller (contiguous, row-major, 16-byte aligned), unless a comment
 * says "host".  The cache owns its page pool and metadata and frees them in
 * hikv_destroy_cache.
 *
 * Method (citations name the page and its section):
 *   - decode attention o_h = softmax(q_h K^T * scale) V over the retained
 *     tokens of each (layer, batch, KV head) "unit"; query head h uses KV head
 *     h / G (HiKV paper, sec. II-A; Kelle summary, sec. 2.2 eq. 1-2);
 *   - each retained token's importance accumulates the softmax mass it
 *     receives, summed over the G query heads of its KV group (KV cache
 *     compression blog, sec. 3 "H2O" and sec. 5.2 on GQA; Kelle summary,
 *     sec. 4.1 eq. 3);
 *   - when a unit holds more than its budget B_u, it keeps the S sink tokens,
 *     the W most recent tokens and the B_u - S - W most important others
 *     (ties: lowest position kept), and compacts the survivors into its first
 *     pages (blog sec. 3 "H2O" and "StreamingLLM"; per-head budgets, HeadKV
 *     summary sec. 3.2; compaction, blog sec. 5.1).
 *
 * Streams and ordering: every call enqueues work on `stream` and returns
 * without waiting for the GPU (create/destroy excepted).  Calls on one cache
 * must be ordered on one stream (or ordered by the caller); overlapping calls
 * on one cache race.  Argument and capacity errors are detected on the host,
 * before anything is enqueued, from an exact host mirror of every unit's
 * length; they leave the cache unchanged.  Launch failures return
 * HIKV_ERR_CUDA.  hikv_last_error() gives a message for the calling thread.
 *
 * Units are numbered u = (layer * batch + b) * num_kv_heads + g.  A call on
 * layers [layer0, layer0 + nlayers) touches exactly those units.
 */
#ifndef HIKV_H_
#define HIKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                    /* same type as cudaStream_t */
typedef struct CUstream_st* hikv_stream_t;

typedef struct hikv_cache hikv_cache;  /* opaque, library-owned */

typedef enum {
    HIKV_OK = 0,
    HIKV_ERR_INVALID_ARG = 1,     /* bad pointer, size, range or config */
    HIKV_ERR_OUT_OF_MEMORY = 2,   /* device allocation failed at create */
    HIKV_ERR_CAPACITY = 3,        /* append past max_tokens or past the page pool */
    HIKV_ERR_CUDA = 4,            /* a CUDA call or kernel launch failed */
    HIKV_ERR_TIMEOUT = 5,         /* a bounded device-side wait gave up */
    HIKV_ERR_STATE = 6,           /* call not valid in the cache's state (e.g. decode on an empty unit) */
    HIKV_ERR_UNSUPPORTED = 7      /* shape outside the compiled kernel set */
} hikv_status;

typedef enum { HIKV_F32 = 0, HIKV_BF16 = 1 } hikv_dtype;

typedef struct {
    int32_t num_layers;     /* > 0 */
    int32_t batch;          /* > 0 */
    int32_t num_q_heads;    /* Hq, multiple of num_kv_heads */
    int32_t num_kv_heads;   /* Hkv; group size G = Hq / Hkv in {1, 2, 4, 8} */
    int32_t head_dim;       /* d in {64, 128} */
    int32_t dtype;          /* hikv_dtype of K, V, q and out; accumulation is fp32 */
    int32_t num_sink;       /* S >= 0: positions < S are never evicted */
    int32_t recent_window;  /* W >= 0: the W newest positions are never evicted */
    const int32_t* budgets; /* HOST [num_layers * num_kv_heads], B_u per (layer, KV
                               head), shared by all batch rows; each >= S + W and >= 1.
                               Copied at create. */
    int32_t max_tokens;     /* slots per unit: a unit never holds more tokens */
    int32_t page_tokens;    /* tokens per KV page: power of two, multiple of 16 (0 => 64) */
    int64_t pool_pages;     /* pages in the shared pool (0 => every unit can reach
                               max_tokens at once) */
    int32_t max_window_queries; /* largest nq for hikv_score_window (0 => 32) */
    float scale;            /* logit scale; 0 => 1/sqrt(head_dim) */
    int32_t pool_kernel;    /* SnapKV prefill selection (KV cache compression blog,
                               sec. 3 "SnapKV"): with k = pool_kernel > 1,
                               hikv_score_window replaces each prompt token's score
                               by the largest window score of positions [p, p + k)
                               (positions past the prompt contribute nothing), and
                               the cut then keeps the top pooled scores.  0 or 1 =>
                               plain window scores.  At most 64. */
    int32_t importance_mode; /* 0: H2O -- every decode step adds each retained token's
                               attention mass, summed over the group, to its score
                               (blog sec. 3 "H2O").  1: HiKV Stage I -- only tokens
                               of the recent bank (the recent_window newest
                               positions and the one leaving it this step,
                               pos >= t - W) accumulate; older scores are frozen
                               (HiKV sec. III-B, Algorithm 1).  With budget 2W and
                               no sinks this is HiKV's dual bank: the eviction of
                               the lowest score outside the window is its "promote
                               the ejected token only if it beats the important
                               bank's minimum". */
    int32_t element_budget; /* HiKV Stage II (HiKV sec. III-C, Algorithm 1): with
                               0 < B2 = element_budget < head_dim, decode steps
                               approximate attention at element level -- per query
                               head only the B2 dimensions of q with the largest
                               magnitude enter the logits; the softmax P of those
                               logits over every retained token updates the
                               importance; P is cut into chunks of head_dim
                               entries in position order and only each chunk's B2
                               largest entries (ties: the lower position)
                               contribute p_j v_j to the output, which is not
                               renormalised.  Units must then hold at most 16384
                               tokens when a decode step runs.  0 or head_dim =>
                               exact attention. */
    int32_t band_scoring;   /* 1: allow hikv_score_band (HiKV's banded prefill
                               scores); create then also allocates its per-query
                               softmax statistics, batch * Hkv * G * max_tokens *
                               8 bytes.  0: off. */
} hikv_config;

/* Create a cache: allocates the page pool, page tables, per-slot importance
 * (fp32) and position (int32) arrays, and the work buffers, with cudaMalloc
 * on the current device.  The work buffers include the decode kernel's
 * logits for chunks too long for shared memory, G fp32 per slot of every
 * unit (max_tokens x G x 4 bytes a unit: 3 % of the K/V pool at G = 4, 6 %
 * at G = 8, with d = 128 in bf16), so that no call allocates.  Synchronous.
 * On success *out owns all of it.
 * Errors: INVALID_ARG (config), UNSUPPORTED (G or d or dtype), OUT_OF_MEMORY. */
hikv_status hikv_create_cache(const hikv_config* cfg, hikv_cache** out);

/* Free everything the cache owns (synchronises the device first).  NULL is a no-op. */
hikv_status hikv_destroy_cache(hikv_cache* cache);

/* Append ntok tokens to every unit of the layer range (HiKV Algorithm 1,
 * last step: the new token's (k, v) enter the cache; Kelle summary sec. 8.4:
 * a new token may reuse any free slot).  k, v: [nlayers][batch][Hkv][ntok][d]
 * in the cache dtype.  New tokens get importance 0 and the next positions of
 * their unit (positions count every token ever appended, from 0).
 * Errors: INVALID_ARG, CAPACITY (a unit would exceed max_tokens, or the pool
 * would run out of pages). */
hikv_status hikv_append(hikv_cache* cache, int32_t layer0, int32_t nlayers, int32_t ntok,
                        const void* k, const void* v, hikv_stream_t stream);

/* Prefill importance: score the cached tokens with the queries of the last
 * nq appended positions, causally (query i, at position t - nq + 1 + i, sees
 * tokens at positions <= its own), adding each query's softmax mass summed
 * over the group's heads to the tokens' importance, queries in position
 * order (HiKV sec. III-D; SnapKV observation window, blog sec. 3).  No
 * attention output.  q: [nlayers][batch][Hq][nq][d], 1 <= nq <=
 * max_window_queries.  Errors: INVALID_ARG, STATE (a unit holds fewer than
 * nq positions). */
hikv_status hikv_score_window(hikv_cache* cache, int32_t layer0, int32_t nlayers, int32_t nq,
                              const void* q, hikv_stream_t stream);

/* HiKV prefill initialisation (HiKV sec. III-D, with the importance score
 * IS of sec. III-B): every prompt token l of a unit gets
 *     imp_l += sum_{h in group} sum_{i = l}^{min(l + band, n) - 1} P_hi[l],
 * P_hi being query head h's softmax at position i over the tokens at
 * positions <= i (causal) -- the attention column the token receives from
 * the band of queries starting at its own position.  With band = B_I / 2 =
 * the recent window, importance_mode = 1, no sinks and a budget of 2W, the
 * following hikv_evict fills HiKV's two banks as the paper describes (the
 * last W prompt tokens, then the W best-scored of the rest), and decoding
 * continues its Stage I rule.
 * q: [nlayers][batch][Hq][n][d] in the cache dtype, the queries of every
 * held position 0..n-1.  Every unit of the range must hold exactly n tokens,
 * appended and never cut (so slot = position).  No pooling is applied.
 * The cache must have been created with band_scoring = 1.  Cost: O(n^2 d G)
 * per unit (it forms every prompt query's softmax statistics).
 * Errors: INVALID_ARG (band < 1, null q), STATE (band_scoring off, units of
 * unequal length, a cut or empty unit). */
hikv_status hikv_score_band(hikv_cache* cache, int32_t layer0, int32_t nlayers, int32_t band,
                            const void* q, hikv_stream_t stream);

/* One decode step of attention over every retained token (including any
 * appended since the last step), plus the importance update.  q and out:
 * [nlayers][batch][Hq][d] in the cache dtype; out may not alias q.
 * Also records, for each unit holding more than its budget, its single
 * least-important evictable token, which a following hikv_evict uses when it
 * needs to drop exactly one token.  With an element_budget set the step is
 * HiKV Stage II's element-level approximation (see hikv_config).
 * Errors: INVALID_ARG, STATE (an empty unit), CAPACITY (Stage II and a unit
 * holding more than 16384 tokens). */
hikv_status hikv_decode_step(hikv_cache* cache, int32_t layer0, int32_t nlayers,
                             const void* q, void* out, hikv_stream_t stream);

/* One whole decode step in one call: exactly hikv_append (one token per unit,
 * k, v: [nlayers][batch][Hkv][1][d]) + hikv_decode_step (q, out as there)
 * and, with evict != 0, hikv_evict -- same results.  When every unit's new
 * slot already has its page and no unit needs more than one eviction (the
 * steady state once a unit reached its budget) the appended rows enter the
 * cache inside the attention kernel and the evicted slot is refilled with
 * the new token there: one kernel launch (two when the call's equal units
 * need more rounds of clusters than one and the last round would be at most
 * half busy, or when ragged units split between the cluster and the
 * warp-per-unit kernels; with an element_budget, the element-level
 * kernels).  Otherwise it runs the three calls.  k and v must be 16-byte aligned (HIKV_ERR_INVALID_ARG
 * otherwise).  Errors: as the three calls. */
hikv_status hikv_decode_step_fused(hikv_cache* cache, int32_t layer0, int32_t nlayers,
                                   const void* k, const void* v, const void* q, void* out,
                                   int32_t evict, hikv_stream_t stream);

/* Cut every unit of the range holding n > B_u tokens to exactly B_u:
 * keep sinks, recent window and the B_u - S - W highest-importance others
 * (ties keep the lower position), compact the survivors into slots
 * [0, B_u) and return to the pool the whole pages beyond room for B_u + 16
 * tokens (so up to 16 more steps append without allocating).
 * Survivors keep their importance.  No-op for units with n <= B_u.  The
 * caller picks the interval: after every step, every E steps, or once after
 * prefill.  Errors: INVALID_ARG. */
hikv_status hikv_evict(hikv_cache* cache, int32_t layer0, int32_t nlayers, hikv_stream_t stream);

/* Export the retained state of every unit of the range, positions
 * ascending.  lengths: [units]; positions (int32), importance (fp32):
 * [units][cap]; k_out, v_out: [units][cap][d] in the cache dtype, or NULL to
 * skip.  Rows past a unit's length hold position -1, importance 0 and zero
 * K/V.  cap must be >= every unit's length.  lengths is written on the
 * stream (read it after the stream synchronises).  Errors: INVALID_ARG. */
hikv_status hikv_gather_retained(hikv_cache* cache, int32_t layer0, int32_t nlayers, int32_t cap,
                                 int32_t* lengths, int32_t* positions, float* importance,
                                 void* k_out, void* v_out, hikv_stream_t stream);

/* Diagnostic: the cluster-kernel launches of the latest decode call of this
 * cache, as the host's cost model configured them (a call of equal units
 * whose last round of clusters would be at most half busy runs as two
 * launches).  out_host[8]: per launch (up to two, zeros past the last)
 * units, cluster size (CTAs per unit), clusters, and 1 if the logits stayed
 * in shared memory (0: the global buffer).  Host only.  Errors: INVALID_ARG. */
hikv_status hikv_last_decode_config(const hikv_cache* cache, int32_t* out_host);

/* Diagnostic: the number of V rows the element-level (HiKV Stage II) decode
 * steps of this cache have read since it was created -- rows that at least
 * one query head of the unit's group kept (HiKV sec. III-C: V is loaded only
 * at the selected entries of P).  0 when element_budget is off.  Synchronous
 * (a device-to-host copy after the work queued before it on the legacy
 * stream).  Errors: INVALID_ARG, CUDA. */
hikv_status hikv_element_rows(const hikv_cache* cache, int64_t* rows_host);

/* Diagnostic: the raw contents of slot `slot` of unit `unit` -- K row and V
 * row (d elements of the cache dtype each), importance, position -- copied
 * to HOST buffers (any may be NULL), whether the slot is live or not.
 * Synchronises the device.  With the environment variable HIKV_DEBUG=1 set
 * when the cache is created, slots that no token holds read as NaN rows,
 * NaN importance and position -1: the pool starts that way, and every slot
 * an eviction vacates and every page returned to a shared pool is
 * overwritten so, so a kernel reading a dead slot turns its outputs into
 * NaN; slot indices taken from data are also range-checked and reported as
 * HIKV_ERR_STATE by hikv_device_status.
 * Errors: INVALID_ARG, STATE (no page mapped for the slot), CUDA. */
hikv_status hikv_read_slot(const hikv_cache* cache, int32_t unit, int32_t slot, void* k_host, void* v_host,
                           float* imp_host, int32_t* pos_host);

/* HOST copy of the host mirror of each unit's length (no device access):
 * lengths_host: [nlayers * batch * Hkv].  Errors: INVALID_ARG. */
hikv_status hikv_get_lengths(const hikv_cache* cache, int32_t layer0, int32_t nlayers,
                             int32_t* lengths_host);

/* Budget schedules: host-only helpers that fill a budgets table for
 * hikv_config (no device, no cache).  out_host: [num_layers * num_kv_heads].
 *
 * PyramidKV (KV cache compression blog, sec. 3 "PyramidKV"): layer l =
 * 1..num_layers gets C_l = C_max - (l - 1)(C_max - C_min)/(num_layers - 1)
 * with C_min = min_budget and C_max = 2 * avg - min_budget, so that the
 * mean is avg; each C_l is rounded half up and raised to at least
 * floor_budget (pass max(1, S + W)); one layer gets avg.  Every KV head of
 * a layer shares the layer's budget.  HIKV_ERR_INVALID_ARG unless
 * num_layers, num_kv_heads >= 1, 0 <= min_budget <= avg, floor_budget >= 0
 * and out_host is non-null. */
hikv_status hikv_budgets_pyramid(int32_t num_layers, int32_t num_kv_heads, int32_t avg, int32_t min_budget,
                                 int32_t floor_budget, int32_t* out_host);

/* DuoAttention (blog sec. 3 "DuoAttention"): heads flagged in retrieval_host
 * ([num_layers * num_kv_heads], nonzero = retrieval head) keep the full
 * cache (full_budget, e.g. max_tokens); the others, streaming heads, keep
 * num_sink + recent_window tokens.  HIKV_ERR_INVALID_ARG on null pointers,
 * sizes < 1 or full_budget < num_sink + recent_window. */
hikv_status hikv_budgets_duo(int32_t num_layers, int32_t num_kv_heads, const uint8_t* retrieval_host,
                             int32_t full_budget, int32_t num_sink, int32_t recent_window, int32_t* out_host);

/* Failure-detection self-test: enqueues one kernel whose bounded device wait
 * (on a barrier nothing arrives on) gives up after limit_us microseconds
 * (1 .. 2e6) and records the timeout in the cache's device error word, as a
 * real stalled wait would; the kernel then returns and the context stays
 * usable.  The next hikv_device_status reports HIKV_ERR_TIMEOUT (site
 * "self-test") and clears it.  HIKV_ERR_INVALID_ARG on a null cache or a
 * limit out of range. */
hikv_status hikv_selftest_timeout(hikv_cache* cache, int32_t limit_us, hikv_stream_t stream);

/* Number of kernels launched on the caller's streams through this cache
 * since it was created (every entry point counts what it enqueued; a call
 * that returned an error before launching counts nothing).  Host-only, no
 * synchronisation.  Returns -1 for a null cache. */
int64_t hikv_kernel_launches(const hikv_cache* cache);

/* Synchronise the device and report device-side errors recorded by the
 * kernels (a bounded wait that gave up, a page id out of range); clears them.
 * Returns TIMEOUT or STATE for a recorded error, CUDA for a sticky CUDA
 * error, else OK. */
hikv_status hikv_device_status(hikv_cache* cache);

/* Prompt importance for callers that cannot allocate device memory.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that may not call cudaMalloc: a plugin inside an inference engine that owns
 * every device allocation and forbids allocating while it runs, or a
 * real-time path where an allocation, and the synchronisation it can cause,
 * is not allowed.  Such a caller cannot create a cache (hikv_create_cache
 * allocates), so this call is stateless: it computes, for a prompt of ntok
 * tokens (positions 0..ntok-1) per unit, what hikv_append + hikv_score_window
 * would leave as importance in a fresh cache, from buffers the caller owns.
 *
 * k: [nlayers][batch][Hkv][ntok][d], q: [nlayers][batch][Hq][nq][d] (queries
 * of positions ntok-nq..ntok-1), both in `dtype`; importance:
 * [nlayers][batch][Hkv][ntok] fp32, overwritten.  Device pointers, 16-byte
 * aligned.  scale 0 => 1/sqrt(head_dim).
 *
 * It allocates nothing.  Its scratch is a file-scope static device array of
 * 2^20 floats (4 MiB) that every GPU loading the library holds until the
 * process exits; calls needing more -- nlayers*batch*Hkv * ceil(ntok/1024) *
 * G*nq * 2 floats -- are rejected with HIKV_ERR_INVALID_ARG and a message.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process; make that
 * first call before any stream capture.  A cudaDeviceReset unloads the
 * module and may move the array, so a process that resets a device must not
 * call this entry point on that device afterwards.
 * Every call shares the one array: calls that overlap on the GPU (other
 * streams, other threads) race and must be serialised by the caller.
 * Errors: INVALID_ARG, UNSUPPORTED (head_dim, dtype or too many query
 * vectors for shared memory), CUDA (launch). */
hikv_status hikv_score_window_noalloc(int32_t nlayers, int32_t batch, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                                      int32_t ntok, int32_t nq, float scale, const void* k,
                                      const void* q, float* importance, hikv_stream_t stream);

/* Measurement aid, no part of the method: the plainest streaming read of
 * `bytes` bytes at `buf` (DEVICE, 16-byte aligned, bytes a positive multiple
 * of 16) -- eight independent 16-byte loads per thread and round over a
 * grid of ctas_per_sm (1..4) CTAs of 512 threads per SM, nothing stored
 * except, almost never, one word to `sink` (DEVICE, 4 bytes) to keep the
 * loads alive.  Timed around a cold buffer, it is the floor for any kernel
 * that reads that many bytes once in one launch.
 * Errors: INVALID_ARG, CUDA (launch). */
hikv_status hikv_read_floor(const void* buf, int64_t bytes, int32_t ctas_per_sm, uint32_t* sink,
                            hikv_stream_t stream);

/* Message for the last failing call on this thread ("" if none). */
const char* hikv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* HIKV_H_ */
