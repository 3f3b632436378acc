/*
 * dkv.h — C ABI of libdkv: differentiated KV compaction and mixed-precision
 * paged decode attention for one NVIDIA GB300 (sm_103a).
 *
 * The operations follow "DiffKV: Differentiated Memory Management for Large
 * Language Models with Parallel KV Compaction" (SOSP'25, arXiv 2412.03131).
 * Section names below refer to that page:
 *   [Bkg-Q]    Background — per-vector quantization Q = round((X - z)/s),
 *              X^ = s*Q + z, applied to every key and value vector.
 *   [Bkg-Attn] Background — the attention equation (softmax(q.k/sqrt(d)) v).
 *   [Pol-P]    Compaction policy — prompt-phase logic (importance = mean
 *              attention a token receives; GQA heads combined with max;
 *              recent window W always high precision; thresholds a_h/N, a_l/N).
 *   [Pol-G]    Compaction policy — generation-phase logic and algorithm flow
 *              (candidate t_c, victim t_v, demote or prune).
 *   [Mem-PC]   Memory management — parallel KV compaction (plan / coordinate,
 *              parallel prefix sum).
 *   [Mem-UP]   Memory management — unified pages (six segments).
 *   [Mem-FL]   Memory management — circular free page list (start pointer
 *              allocates, end pointer reclaims, both wrap).
 *   [Mem-BT]   Memory management — bidirectional page table (high-precision
 *              pages grow from the left, low-precision from the right).
 *   [Mem-Fig6] Memory management — prompt-phase workflow, Figure 6.
 *   [Mem-Gen]  Memory management — generation-phase workflow.
 *   [Impl-Kern] System implementation — custom attention kernel (hi pages
 *              first, then lo pages; key / value layouts; sequence split).
 *   [Pol-Ext]  Compaction policy — extensibility (more precision levels;
 *              thresholds adjusted for each head individually).
 *   [Impl-Arch] System implementation — architecture overview (the KV
 *              compactor is invoked once the layer's keys and values exist,
 *              next to the model's own attention over the prompt).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Return 0 on success, a negative DKV_ERR_* code otherwise.
 *  - "host" pointers are read before the call returns and may be reused at
 *    once. "device" pointers must stay valid until the work queued on
 *    `stream` (a cudaStream_t passed as void*, NULL = legacy default stream)
 *    completes. The caller owns every input and output buffer. Device
 *    buffers of fp16/fp32 vectors (k, v, q_obs, q, out) must start on a
 *    16-byte boundary, score arrays on a 4-byte boundary (DKV_ERR_ARG
 *    otherwise).
 *  - All calls on one pool must be ordered on one stream (or synchronised by
 *    the caller). compact_step, decode_attention and free_request never
 *    synchronise the host; argument and request-state errors are detected on
 *    the host and returned at once with nothing queued.
 *  - Data-dependent failures (free list exhausted, page table full) are
 *    detected on the device before anything is written: the whole call
 *    becomes a no-op and the code latches in the pool's sticky status word.
 *    While the sticky status is non-zero every later call is a device no-op;
 *    dkv_pool_status reads it and dkv_pool_clear_error resets it. A bounded
 *    device wait that gives up (DKV_ERR_TIMEOUT) latches the same way; the
 *    call that raised it leaves its own outputs (attention out, the scores
 *    it updates) undefined.
 *
 * Unified page format  [Mem-UP]
 * -----------------------------
 * Two tiers, fixed bit widths: hi = K8V4 (8-bit key codes, 4-bit value
 * codes), lo = K4V2 [Pol-P]; optionally a third, mid = K8V2, between them
 * [Pol-Ext] (config.mid_enabled). head_dim d = 128. A page holds T tokens of
 * one tier; T is the largest multiple of g = 8/vbits (tokens sharing a value
 * byte: 2 for hi, 4 for lo and mid) whose six segments fit in page_bytes.
 * For page_bytes = 4096: T_hi = 18, T_lo = 36, T_mid = 20. Segments, in
 * order, each starting on a 16-byte boundary, slot t in [0, T):
 *   1. K codes  T rows of d*kbits/8 bytes (128 B hi, 64 B lo).
 *               8-bit: byte i = code of feature i.
 *               4-bit: byte i bits 0-3 = feature 2i, bits 4-7 = feature 2i+1.
 *   2. V codes  T/g rows of 128 bytes; row u holds slots u*g .. u*g+g-1.
 *               A row is 32 little-endian 32-bit words; word w covers
 *               features 4w..4w+3. For feature 4w+i, slot u*g+e:
 *               4-bit (g=2): bits [16e + 4i, +4)
 *               2-bit (g=4): bits [16(e&1) + 4i + 2(e>>1), +2)
 *   3. K meta   T x {fp16 scale, fp16 zero} (4 bytes per slot).
 *   4. V meta   same for values.
 *   5. score    T x fp32 accumulated attention score S.
 *   6. position T x int32 token position in the request.
 * Codes [Bkg-Q], per token vector x (128 values, fp16 inputs widened to
 * fp32), L = 2^bits - 1, all fp32 arithmetic correctly rounded, no fused
 * contraction unless stated:
 *   mn = min x, mx = max x; s = half(fdiv(fsub(mx, mn), L)); z = half(mn)
 *   s == 0 -> every code 0; else inv = fdiv(1, s) and
 *   code_i = clamp(rint_even(fmul(fsub(x_i, z), inv)), 0, L)
 *   dequantised value = fma(s, code, z) (one rounding).
 *   half() is IEEE binary16 round-to-nearest-even. Re-quantising a hi token to
 *   lo applies the same steps to its dequantised hi values.
 *
 * Free list and page table  [Mem-FL] [Mem-BT]
 * -------------------------------------------
 * The free list is an int32 array of n_pages page IDs with two monotone
 * 64-bit counters start and end; free = end - start, entry = list[c mod P].
 * Initially list[i] = i, start = 0, end = n_pages. Allocation consumes from
 * start, reclaim appends at end. One table row per (layer, request slot, KV
 * head) of L_e = ceil(max_seq_len / T_hi) + 1 int32 entries: hi page k at
 * entry k, lo page k at entry L_e-1-k, unused entries -1. Hi slot s lives on
 * hi page s / T_hi at slot s % T_hi; lo slot s on lo page s / T_lo.
 * With the mid tier each row composes that two-way table with a one-way
 * table of L_m = ceil(max_seq_len / T_mid) + 1 entries after it [Mem-Gen:
 * further precision levels by combining one-way or two-way page tables]:
 * mid page k at entry L_e + k; the row then has L_e + L_m entries.
 *
 * Three tiers [Pol-Ext]: a token is hi if I > alpha_h/N, else mid if
 * I >= alpha_m/N, else lo if I >= alpha_l/N, else pruned. The prompt grant
 * stays ceil(N0/T_hi)+slack pages (slack 2 covers the three partial pages);
 * mid pages take the grant pages right after the hi ones. In a generation
 * step the victim is the least important token of the tier t_c ended in (hi:
 * outside the window; mid and lo: t_c included); it stays if it classifies
 * at its tier or above, else moves to the end of the tier it classifies at
 * (re-quantised from its dequantised values) or is pruned. New pages of a
 * head are taken hi, lo, then mid; request completion returns hi, lo, then
 * mid pages.
 */
#ifndef DKV_H
#define DKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes ---------------------------------------------------- */
#define DKV_OK               0
#define DKV_ERR_ARG         -1  /* bad argument (NULL, out of range, bad config) */
#define DKV_ERR_CUDA        -2  /* a CUDA runtime call failed */
#define DKV_ERR_STATE       -3  /* request slot in the wrong state for the call */
#define DKV_ERR_NO_PAGES    -4  /* free list holds fewer pages than the call needs */
#define DKV_ERR_TABLE_FULL  -5  /* a head needs more pages than its grant / row */
#define DKV_ERR_TIMEOUT     -6  /* a bounded device wait gave up */
#define DKV_ERR_CHECK       -7  /* a device-side consistency check failed */
#define DKV_ERR_UNSUPPORTED -8  /* configuration outside what the kernels support */
#define DKV_ERR_SCRATCH     -9  /* call needs more than the fixed scratch array holds */

/* ---- modes ------------------------------------------------------------ */
#define DKV_PROMPT 0  /* compact a whole prompt            [Pol-P] [Mem-Fig6] */
#define DKV_DECODE 1  /* append one token, compact one      [Pol-G] [Mem-Gen]  */

/* ---- configuration ------------------------------------------------------ */
typedef struct dkv_config {
  int32_t n_layers;            /* layers sharing the page pool                 */
  int32_t n_kv_heads;          /* Hkv                                          */
  int32_t group_size;          /* G = query heads per KV head, 1..8            */
  int32_t head_dim;            /* must be 128                                  */
  int32_t page_bytes;          /* unified page size, multiple of 16, e.g. 4096 */
  int32_t n_pages;             /* P, pages in the pool                         */
  int32_t max_requests;        /* request slots 0..max_requests-1              */
  int32_t max_seq_len;         /* longest request (prompt + generated)         */
  int32_t tokens_per_hi_page;  /* 0 = largest that fits; else a multiple of 2  */
  int32_t tokens_per_lo_page;  /* 0 = largest that fits; else a multiple of 4  */
  int32_t lo_enabled;          /* 0: no K4V2 tier; survivors are stored hi     */
  float   alpha_h;             /* hi threshold alpha_h / N                     */
  float   alpha_l;             /* lo threshold alpha_l / N                     */
  int32_t recent_window;       /* W: the last W tokens are always hi, >= 0     */
  int32_t obs_window;          /* observation queries per prompt; must be 32   */
  int32_t prompt_grant_slack;  /* extra pages in each head's all-hi grant, >=0 */
  int32_t reclaim_in_decode;   /* 1: free a tier's emptied tail page in DECODE */
  int32_t mid_enabled;         /* 1: a third tier mid = K8V2 (needs lo_enabled;
                                  every tier's T a multiple of 16)            */
  float   alpha_m;             /* mid threshold alpha_m / N (mid_enabled)      */
  int32_t tokens_per_mid_page; /* 0 = largest that fits; else a multiple of 4  */
} dkv_config;

typedef struct dkv_pool dkv_pool;   /* opaque; owns every device structure */

/* Pool geometry derived from the config (valid after dkv_pool_create). */
typedef struct dkv_geometry {
  int32_t t_hi, t_lo;              /* tokens per hi / lo page              */
  int32_t table_len;               /* L_e                                  */
  int32_t hi_off[6];               /* segment byte offsets, hi page        */
  int32_t lo_off[6];               /* segment byte offsets, lo page        */
  int32_t hi_used, lo_used;        /* bytes used by the six segments       */
  int32_t t_mid;                   /* tokens per mid page (0 without mid)  */
  int32_t mid_table_len;           /* L_m (0 without mid)                  */
  int32_t row_len;                 /* table entries per head: L_e + L_m    */
  int32_t count_stride;            /* head counter ints: 4, or 8 with mid  */
  int32_t mid_off[6];              /* segment byte offsets, mid page       */
  int32_t mid_used;                /* bytes used by a mid page's segments  */
} dkv_geometry;

/* Sticky status and pool-wide counters (host struct). */
typedef struct dkv_status {
  int32_t error;        /* first data-dependent error since the last clear, 0 if none */
  int32_t error_info;   /* head or layer index associated with the error, -1 if none  */
  int64_t list_start;   /* free-list allocation counter                                */
  int64_t list_end;     /* free-list reclaim counter                                   */
  int64_t free_pages;   /* list_end - list_start                                       */
  int64_t hi_tokens;    /* stored hi tokens over all layers, requests and heads        */
  int64_t lo_tokens;    /* stored lo tokens                                            */
  int64_t hi_pages;     /* pages held as hi                                            */
  int64_t lo_pages;     /* pages held as lo                                            */
  int64_t mid_tokens;   /* stored mid tokens (0 without mid)                           */
  int64_t mid_pages;    /* pages held as mid                                           */
} dkv_status;

/* Host snapshot of the device state; every pointer may be NULL to skip it.
 * Sizes: pages  n_pages*page_bytes bytes; free_list n_pages int32;
 *        table  n_layers*max_requests*n_kv_heads*row_len int32;
 *        head_counts n_layers*max_requests*n_kv_heads*count_stride int32
 *                    {hi tokens, lo tokens, hi pages, lo pages
 *                     [, mid tokens, mid pages, 0, 0 with the mid tier]};
 *        req_state   n_layers*max_requests*4 int32 {active, N0, N, updates};
 *        pointers    2 int64 {start, end}. */
typedef struct dkv_snapshot {
  uint8_t* pages;
  int32_t* free_list;
  int32_t* table;
  int32_t* head_counts;
  int32_t* req_state;
  int64_t* pointers;
} dkv_snapshot;

/* Create a pool on `cuda_device`: allocates the pages, the free list, page
 * tables, counters, scratch and the status word, all on the device. The
 * pool's memory is fixed for its lifetime. Errors: DKV_ERR_ARG for an invalid
 * config (mid_enabled without lo_enabled included), DKV_ERR_UNSUPPORTED
 * (head_dim != 128, G outside 1..8, obs_window != 32, mid_enabled with a
 * tier whose T is not a multiple of 16), DKV_ERR_CUDA if an allocation fails
 * (nothing leaks). */
int dkv_pool_create(const dkv_config* cfg, int cuda_device, dkv_pool** out);

/* Synchronise the device, free everything the pool owns. NULL is a no-op. */
int dkv_pool_destroy(dkv_pool* pool);

/* Geometry of a created pool (host struct). */
int dkv_pool_geometry(const dkv_pool* pool, dkv_geometry* out);

/* One compaction step of one layer for n_req requests.
 *
 * PROMPT [Pol-P] [Mem-PC] [Mem-Fig6]: req_slots[i] (host, distinct, inactive
 * in `layer`) gets a prompt of seq_lens[i] (host, 1..max_seq_len) tokens.
 *   k, v    device fp16 [sum(seq_lens)][n_kv_heads][128], requests back to
 *           back in call order.
 *   q_obs   device fp16 [n_req][32][n_kv_heads*G][128]: the queries of the
 *           last 32 prompt positions (row o is position seq_len-32+o; rows
 *           with a negative position are ignored). Query head h belongs to KV
 *           head h / G.
 *   scores_in  NULL: the kernels score every token from q_obs (importance =
 *           sum over observation queries at or after the token of the max
 *           over the group's heads of softmax(q.k/sqrt(128)); divided by the
 *           number of such queries). Non-NULL: device fp32
 *           [sum(seq_lens)][n_kv_heads] scores given by the caller (q_obs is
 *           then ignored and may be NULL).
 *   scores_out NULL or device fp32 [sum(seq_lens)][n_kv_heads]: receives
 *           the score S of every token (given or computed).
 *   Each head is granted ceil(N0/T_hi)+slack pages by one prefix sum over
 *   the heads (call order, then KV head) at the list start; hi tokens fill
 *   the grant from the left (mid tokens the pages after them), lo tokens
 *   from the right, the unused middle pages are reclaimed at the list end by
 *   a second prefix sum.
 *
 * DECODE [Pol-G] [Mem-Gen]: every req_slots[i] must be active in `layer`.
 *   k, v    device fp16 [n_req][n_kv_heads][128]: the new token of each
 *           request (position N, N = the request's current length).
 *   seq_lens, q_obs, scores_in, scores_out must be NULL.
 *   Per head: append the new token hi; classify the window's oldest token
 *   t_c; demote or prune one victim; new pages come from one prefix sum at
 *   the list start, emptied tail pages (if reclaim_in_decode) go to the end.
 *
 * Errors: DKV_ERR_ARG, DKV_ERR_STATE (host, nothing queued); DKV_ERR_NO_PAGES,
 * DKV_ERR_TABLE_FULL latch in the sticky status (device, call is a no-op). */
int dkv_compact_step(dkv_pool* pool, int32_t layer, int32_t mode, int32_t n_req,
                     const int32_t* req_slots, const int32_t* seq_lens,
                     const void* k, const void* v, const void* q_obs,
                     const float* scores_in, float* scores_out, void* stream);

/* Causal attention over whole prompts [Bkg-Attn] [Impl-Arch], the model's
 * own prompt attention, computed by the same library so that its
 * observation rows' log-sum-exps can feed the compactor (the prompt's
 * scores then need one pass over the keys instead of two). For request i
 * (seq_lens[i] tokens, host, 1..max_seq_len; requests back to back in call
 * order) and query head h (KV head h / G):
 *   out[t][h] = sum_{j<=p} softmax_j(q[t][h] . k_j / sqrt(128)) v_j
 * for the token t at position p, over the request's keys j = 0..p.
 *   q       device fp16 [sum(seq_lens)][n_kv_heads*G][128]
 *   k, v    device fp16 [sum(seq_lens)][n_kv_heads][128]
 *   out     device fp32 [sum(seq_lens)][n_kv_heads*G][128]
 *   lse_obs NULL or device fp32 [n_req][n_kv_heads*G][32]: row o receives
 *           log2 sum_{j<=p} 2^(q.k_j log2(e)/sqrt(128)) for position
 *           p = seq_len-32+o (the base-2 log-sum-exp of the observation
 *           query at p), -inf where p < 0.
 * The pool supplies the geometry and the stream order; no pool state is
 * read or written (a latched sticky error makes it a device no-op like
 * every other call). fp16 products accumulate in fp32; the probabilities
 * enter the value product as an fp16 pair of about 22 significant bits.
 * Errors: DKV_ERR_ARG (host, nothing queued); DKV_ERR_CUDA. */
int dkv_prefill_attention(dkv_pool* pool, int32_t n_req, const int32_t* seq_lens, const void* q,
                          const void* k, const void* v, float* out, float* lse_obs, void* stream);

/* PROMPT compaction [Pol-P] [Mem-PC] [Mem-Fig6] [Impl-Arch] with the
 * observation rows' log-sum-exps already known (lse_obs of
 * dkv_prefill_attention over the same requests, in the same order): the
 * score pass reads the keys once instead of twice. Arguments, results and
 * errors are those of dkv_compact_step in PROMPT mode with scores_in = NULL;
 * q_obs holds the last 32 query rows of each prompt, the rows lse_obs was
 * computed for. lse_obs: device fp32 [n_req][n_kv_heads*G][32]. */
int dkv_compact_step_prefilled(dkv_pool* pool, int32_t layer, int32_t n_req, const int32_t* req_slots,
                               const int32_t* seq_lens, const void* k, const void* v, const void* q_obs,
                               const float* lse_obs, float* scores_out, void* stream);

/* Decode attention of one layer over the mixed-precision pages [Impl-Kern]
 * [Bkg-Attn]: for each request i and query head h,
 *   out[i][h] = sum_j softmax_j(q[i][h] . k^_j / sqrt(128)) v^_j
 * over every stored token j of KV head h / G (hi pages, then mid pages, then
 * lo pages), with
 * k^, v^ the dequantised codes. q: device fp16 [n_req][n_kv_heads*G][128];
 * out: device fp32 [n_req][n_kv_heads*G][128]. If update_scores != 0, each
 * stored token's score gains max over the group's heads of its softmax
 * probability, and the request's update counter (used for the importance
 * denominator in DECODE compaction) increases by one.
 * Errors: DKV_ERR_ARG, DKV_ERR_STATE (slot inactive in `layer`). */
int dkv_decode_attention(dkv_pool* pool, int32_t layer, int32_t n_req,
                         const int32_t* req_slots, const void* q, float* out,
                         int32_t update_scores, void* stream);

/* Size of the fixed device array that dkv_decode_attention_static works in. */
#define DKV_ATTN_STATIC_SCRATCH_BYTES (64u << 20)

/* dkv_decode_attention without the pool's scratch, for callers that cannot
 * allocate device memory. The paper has no counterpart: it is an interface
 * addition of this library. Arguments, layouts, results and the other
 * errors are those of dkv_decode_attention, and it runs the same kernels.
 *
 * Who needs it: a host runtime whose own allocator already holds the device's
 * free memory (a serving engine hands nearly all HBM to its KV page pool at
 * start-up, so a later cudaMalloc fails or fragments that memory), or code
 * that must not call cudaMalloc/cudaFree at all because those calls
 * synchronise the device. Neither attention entry point allocates per call;
 * this one also needs no scratch sized for the pool's maximum batch and
 * length: it works in one static array of DKV_ATTN_STATIC_SCRATCH_BYTES
 * (64 MiB) in the library's device image, reserved by the CUDA driver when
 * the library's module is loaded. No cudaMalloc, cudaFree or other
 * allocating routine is called.
 *
 * Size limit: with U = n_req * n_kv_heads, C = ceil(max_n / 16) + 1, or + 2
 * in a pool with the mid tier (max_n = the largest current length N among
 * the call's requests: prompt length plus generated tokens, pruned tokens
 * included, not the stored count) and
 * r(x) = x rounded up to 256, the call needs r(4UG) + r(4U(C/8 + 2)(128G + 16))
 * bytes, plus 64GUC if update_scores != 0. A larger call returns
 * DKV_ERR_SCRATCH and queues nothing.
 *
 * Set-up: dkv_pool_create looks up the array's address on the pool's device
 * (cudaGetSymbolAddress, with that device current) and keeps it in the pool,
 * so a call does no set-up of its own. A pool created after the device's
 * context was reset (cudaDeviceReset) holds the address in the new context;
 * pools from before a reset are unusable anyway. Every call on a device
 * shares the array and it keeps the last call's contents; nothing in it has
 * to start at zero, because every value a call reads from the array
 * (partials and the per-chunk rows of logits) is written earlier in the
 * same call.
 * This entry point leaves no victim keys for the next generation step, which
 * then searches the heads itself (same result, more work).
 * Calls that overlap on the GPU (on different streams, or from different
 * pools of one device) race on the array and give wrong results: order them
 * on one stream or synchronise between them.
 * Errors: DKV_ERR_ARG, DKV_ERR_STATE, DKV_ERR_SCRATCH (host, nothing queued);
 * DKV_ERR_CUDA if a launch fails. */
int dkv_decode_attention_static(dkv_pool* pool, int32_t layer, int32_t n_req,
                                const int32_t* req_slots, const void* q, float* out,
                                int32_t update_scores, void* stream);

/* Thresholds for each KV head of one layer [Pol-Ext]: from the next
 * compaction step of `layer` on (stream order), head h's tokens are compared
 * with alpha_h[h]/N and alpha_l[h]/N instead of the configuration's pair
 * (prompt classification and the generation step's t_c and victims).
 * alpha_h, alpha_l: host arrays of n_kv_heads floats, copied before the call
 * returns (the copy from pageable memory may wait for work already queued on
 * `stream`). Until set, every head of every layer uses config.alpha_h and
 * config.alpha_l. Decode attention does not use thresholds.
 * Errors: DKV_ERR_ARG (NULL, layer out of range, NaN); DKV_ERR_CUDA. */
int dkv_pool_set_thresholds(dkv_pool* pool, int32_t layer, const float* alpha_h, const float* alpha_l,
                            void* stream);

/* The mid tier's threshold for each KV head of one layer [Pol-Ext]: from the
 * next compaction step of `layer` on (stream order), head h's tokens are mid
 * when I >= alpha_m[h]/N and not hi. alpha_m: host array of n_kv_heads
 * floats, copied before the call returns. Until set, every head uses
 * config.alpha_m. Errors: DKV_ERR_ARG (NULL, layer out of range, NaN, pool
 * without the mid tier); DKV_ERR_CUDA. */
int dkv_pool_set_mid_thresholds(dkv_pool* pool, int32_t layer, const float* alpha_m, void* stream);

/* Return every page of request `req_slot` in every layer to the list end
 * (one prefix sum over (layer, KV head); within a head hi pages left to
 * right, then lo pages from the outermost inward, then mid pages left to
 * right) and clear its rows [Mem-Gen]. Errors: DKV_ERR_ARG, DKV_ERR_STATE
 * (slot active in no layer). */
int dkv_free_request(dkv_pool* pool, int32_t req_slot, void* stream);

/* Synchronise the pool's device work and read the sticky status and counters. */
int dkv_pool_status(dkv_pool* pool, dkv_status* out);

/* Synchronise, clear the sticky status and re-read the host's copy of the
 * request state from the device. */
int dkv_pool_clear_error(dkv_pool* pool);

/* Synchronise and copy the device state into host buffers (see dkv_snapshot). */
int dkv_pool_export(dkv_pool* pool, dkv_snapshot* out);

/* Static description of an error code. */
const char* dkv_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* DKV_H */
