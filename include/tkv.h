/*
 * tkv.h — C ABI of a tiered KV-cache decode step for GB300 (sm_103a).
 *
 * The method is the semantic-aware four-tier KV hierarchy of "Not All Thoughts
 * Need HBM" (summary of arXiv 2605.09490):
 *   T0  tokens resident in GPU HBM (protected prompt, attention sinks, recent
 *       window, and the most important reasoning tokens)  — Methodology 1;
 *   T1  medium-importance tokens in pinned host DDR at full precision,
 *       prefetched to the GPU before each attention step   — Methodology 1, 4;
 *   T2  low-importance tokens in host memory as 8-bit codes — Methodology 1;
 *   T3  the absolute tail, deleted for good                — Methodology 1.
 * Importance is the cumulative attention score of Methodology 2,
 *   s_i(t) = s_i(t-1) + (1/|L|) sum_l (1/H) sum_h alpha_{l,h}(t)[i],
 * accumulated inside the decode step; tiers are reassigned every Delta decode
 * steps (Methodology 4) and only tokens whose tier changed are moved.
 * Proposition 1 (Methodology 3): T1 is read at full precision, so splitting
 * the retained set between T0 and T1 changes no attention output.
 *
 * Ownership: the caller owns every buffer — the device workspace, the pinned
 * host workspace and both CUDA streams — and passes raw pointers. The library
 * owns only host-side bookkeeping, kernels and CUDA events. Pointers passed to
 * a call are borrowed for that call; work is enqueued on the compute stream
 * (prefetches on the copy stream) and is complete once tkv_synchronize
 * returns. A handle is not thread-safe.
 *
 * Errors: every call returns a tkv_status; tkv_last_error() gives the message.
 * No C++ exception crosses this interface. A call that fails argument or
 * capacity checks leaves the state unchanged. A CUDA failure in the middle of
 * a call marks the handle broken (later calls return TKV_ERR_STATE). A device
 * wait that runs out of its iteration budget sets a flag that the next
 * synchronising call reports as TKV_ERR_TIMEOUT; no kernel traps.
 *
 * Layouts (all row-major, element type = the configured KV dtype unless noted):
 *   decode-step query     q     [B][L][Hq][d]
 *   decode-step new K/V   k, v  [B][L][Hkv][d]
 *   decode-step output    out   [B][L][Hq][d]
 *   prefill K/V           k, v  [L][n][Hkv][d]
 * B is the number of sequences created so far (see tkv_append).
 */
#ifndef TKV_H_
#define TKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TKV_API __attribute__((visibility("default")))
#else
#define TKV_API
#endif

typedef struct tkv_ctx* tkv_handle;
typedef void* tkv_stream; /* a cudaStream_t passed as an opaque pointer; NULL = legacy stream */

typedef enum {
  TKV_OK = 0,
  TKV_ERR_INVALID_ARG = 1, /* bad pointer, size, shape or value (e.g. a NaN score) */
  TKV_ERR_CAPACITY = 2,    /* a pool, the workspace or a per-sequence limit is too small */
  TKV_ERR_STATE = 3,       /* call not valid now (e.g. no sequence yet, broken handle) */
  TKV_ERR_CUDA = 4,        /* a CUDA runtime call failed; the message names it */
  TKV_ERR_TIMEOUT = 5,     /* a bounded device wait gave up */
  TKV_ERR_INTERNAL = 6     /* an internal consistency check failed */
} tkv_status;

enum { TKV_DTYPE_F32 = 0, TKV_DTYPE_BF16 = 1 };
enum { TKV_BUDGET_PERCENT = 0, TKV_BUDGET_COUNT = 1 };
enum { TKV_SCALE_PER_TOKEN = 0, TKV_SCALE_PER_TOKEN_HEAD = 1 };
enum { TKV_SCALE_F32 = 0, TKV_SCALE_F16 = 1 };
enum { TKV_T2_ATTEND = 0, TKV_T2_MASK = 1 };
enum { TKV_T0 = 0, TKV_T1 = 1, TKV_T2 = 2, TKV_T3 = 3 };
enum { TKV_FLAG_TIMING = 1 }; /* record CUDA events around attention, prefetch, reclassify */
/* Where attention finds the host tiers T1 and T2 (Methodology 1 and 4):
 *   STREAM   every step copies each layer group's used T1 / T2 range from the pinned host
 *            pools into a two-slot device staging ring on the copy stream, overlapped with
 *            the previous group's attention (T1 is prefetched before each attention step);
 *   MIRROR   device-resident copies of the T1 / T2 pools are kept in step with the host
 *            pools: only tokens whose tier changes cross the host link, at reassignment
 *            (the differential transfer of newly promoted tokens); no per-step copies;
 *   ZEROCOPY attention reads T1 / T2 pages in place from the pinned host pools through
 *            device-mapped pointers (no staging copy, no HBM write of staged pages).
 * The three give bitwise identical attention outputs (the same pages in the same order). */
enum { TKV_HOST_TIERS_STREAM = 0, TKV_HOST_TIERS_MIRROR = 1, TKV_HOST_TIERS_ZEROCOPY = 2 };

/* Configuration. Budgets (Methodology 1): in PERCENT mode budget[k] are the
 * integer percentages of T0..T3 (n_k = floor(budget[k] * N / 100) for k = 1..3,
 * n0 = N - n1 - n2 - n3); in COUNT mode budget[0..2] are token counts of
 * T0..T2 and T3 takes the rest. The protected set of a sequence is
 * [0, max(prompt_len, n_sink)) plus its last recent_window positions. */
typedef struct {
  int32_t n_layers, n_q_heads, n_kv_heads, head_dim; /* Hq % Hkv == 0; d in {64, 128} */
  int32_t kv_dtype;                                   /* TKV_DTYPE_* */
  int32_t max_batch;                                  /* 1 .. 64 sequences */
  int64_t max_tokens;                                 /* positions per sequence, <= 262080 */
  int32_t page_size;                                  /* must be 16 */
  int32_t n_sink, recent_window;
  int32_t budget_mode;                                /* TKV_BUDGET_* */
  int64_t budget[4];
  int32_t reclassify_interval;                        /* Delta (Methodology 4: 64) */
  int32_t t2_scale_gran;                              /* TKV_SCALE_PER_TOKEN[_HEAD] */
  int32_t t2_scale_dtype;                             /* TKV_SCALE_F32 | TKV_SCALE_F16 */
  int32_t t2_mode;                                    /* TKV_T2_ATTEND | TKV_T2_MASK */
  int64_t t0_pages, t1_pages, t2_pages;               /* pool capacities; 0 = derived */
  int64_t max_staged_movers;                          /* staging rows (one layer each) for moves into
                                                         slots vacated in the same reassignment;
                                                         0 = one per position (always enough) */
  int32_t split_pages;                                /* pages per attention CTA; 0 = auto */
  int32_t flags;                                      /* TKV_FLAG_* */
  int32_t host_tiers;                                 /* TKV_HOST_TIERS_* */
  int32_t layers_per_launch;                          /* layers one attention launch covers (and one
                                                         prefetch copies in STREAM mode), at most 32;
                                                         0 = auto: the largest divisor of n_layers
                                                         up to 7 (up to 14 when one layer's K and V
                                                         at full capacity are under 64 MB) */
} tkv_config;

typedef struct {
  int64_t steps, reclassifies, movers;
  int64_t attn_launches;       /* attention kernel launches (one per layer group per step) */
  int64_t attn_bytes;          /* algorithmic KV bytes the attention kernels read */
  int64_t prefetch_bytes;      /* T1 + T2 bytes copied host -> device by prefetch */
  int64_t h2d_move_bytes;      /* bytes moved host -> device at reclassify */
  int64_t d2h_move_bytes;      /* bytes moved device -> host at reclassify */
  int64_t tier_counts[4];      /* current tokens per tier over all sequences */
  double attn_ms;              /* summed attention kernel time; each launch also finishes the
                                  previous launch's output merge and score epilogue (TKV_FLAG_TIMING) */
  double combine_ms;           /* summed time of the epilogue kernel of each step's last launch
                                  (TKV_FLAG_TIMING) */
  double prefetch_ms;          /* summed prefetch copy time      (TKV_FLAG_TIMING) */
  double reclassify_ms;        /* summed reclassify wall time    (TKV_FLAG_TIMING) */
  int64_t kernel_launches;     /* kernels this handle launched (steps, reclassify, prefill) */
  double attn_span_ms;         /* summed device span of the attention launches: first CTA start to
                                  last CTA end, %globaltimer (TKV_FLAG_TIMING; last 4096 launches) */
  int64_t attn_layers;         /* layers attended (attn_launches x layers per launch) */
  double classify_ms;          /* reassignment phases, host wall time (TKV_FLAG_TIMING): classifier */
  double allocate_ms;          /*   host slot allocator                                           */
  double move_ms;              /*   data movement kernels and metadata upload                     */
} tkv_stats;

/* Device and pinned-host bytes tkv_create needs for this configuration: the
 * HBM tier and staging (T0 pool, two T1/T2 staging slots, metadata) on the
 * device, the T1 and T2 pools in pinned host memory (Methodology 1; the
 * Problem statement's ~800 MB per 2,000-token chain is what the tiers split).
 * Errors: TKV_ERR_INVALID_ARG for an invalid configuration (message says why). */
TKV_API tkv_status tkv_workspace_size(const tkv_config* cfg, size_t* dev_bytes, size_t* pinned_bytes);

/* Build a handle over caller-owned memory (no allocation inside the library
 * beyond host bookkeeping). dev_ws: device memory of at least
 * dev_bytes (256-byte aligned); pinned_ws: page-locked host memory of at
 * least pinned_bytes (from cudaHostAlloc / pin_memory). The current CUDA
 * device must be the one that owns dev_ws. */
TKV_API tkv_status tkv_create(const tkv_config* cfg, void* dev_ws, size_t dev_bytes, void* pinned_ws,
                      size_t pinned_bytes, tkv_stream compute, tkv_stream copy, tkv_handle* out);
/* Release the handle's events and bookkeeping (the caller frees the memory). */
TKV_API tkv_status tkv_destroy(tkv_handle h);

/* Prefill: append n_tokens positions (device k, v [L][n][Hkv][d]) to sequence
 * seq, all into T0 with score 0. seq == current count starts a new sequence;
 * prompt tokens (is_prompt != 0) must precede generated ones and are
 * protected (Methodology 1). */
TKV_API tkv_status tkv_append(tkv_handle h, int32_t seq, const void* k, const void* v, int64_t n_tokens,
                      int32_t is_prompt);

/* One decode step for every sequence (device pointers, layouts above):
 * append each new token to T0 (Methodology 1: the recent window is in T0),
 * prefetch T1 and T2 of each layer on the copy stream (Methodology 1, 4),
 * attend over T0 + T1 + T2 with T3 absent (Methodology 3) with the score
 * update of Methodology 2 fused in, fold the step's score increments into s,
 * and reassign tiers when the step count reaches a multiple of Delta
 * (Methodology 4). In STREAM mode a step that ends without a reassignment
 * also enqueues the next step's first layer-group prefetch (T1 and T2 change
 * only at a reassignment), so the host link stays busy between calls.
 * Errors: TKV_ERR_CAPACITY when a sequence or pool is full (state unchanged);
 * TKV_ERR_CUDA marks the handle broken. */
TKV_API tkv_status tkv_decode_step(tkv_handle h, const void* q, const void* k_new, const void* v_new,
                           void* out);

/* The same step (as tkv_decode_step) with HOST buffers: copies q, k_new, v_new
 * in and out back inside the call; returns once out holds the result. Pinned
 * host buffers make the copies asynchronous. */
TKV_API tkv_status tkv_decode_step_host(tkv_handle h, const void* q, const void* k_new, const void* v_new,
                                void* out);

/* Reassign tiers now (Methodology 1, 4) and move the tokens whose tier
 * changed; synchronises the compute stream. */
TKV_API tkv_status tkv_reclassify(tkv_handle h);

/* Enqueue the copy of layer `layer`'s T1 pages and T2 codes into staging slot
 * `slot` (0 or 1) on the copy stream: T1 is prefetched to the GPU before each
 * attention step (Methodology 1), asynchronously (Methodology 4).
 * decode_step calls this itself. Errors: TKV_ERR_INVALID_ARG for a bad layer
 * or slot. */
TKV_API tkv_status tkv_prefetch(tkv_handle h, int32_t layer, int32_t slot);

/* Wait for all enqueued work; reports a device-side timeout flag
 * (TKV_ERR_TIMEOUT). Library plumbing: the paper has no counterpart. */
TKV_API tkv_status tkv_synchronize(tkv_handle h);

/* Test hook for the bounded device waits (the paper has no counterpart): the
 * next attention launch of h withholds the first page copy of one CTA, and from
 * now on h's device waits give up after wait_limit_ns (1 ms .. 2 s) instead of
 * 2 s. The waiting warp gives up, the CTA lands every copy still in flight and
 * publishes an empty partial, and the next synchronising call returns
 * TKV_ERR_TIMEOUT and marks h broken. No kernel traps or hangs. */
TKV_API tkv_status tkv_test_stall_next_attention(tkv_handle h, uint64_t wait_limit_ns);

/* Host-side fault injection (library plumbing for failure tests; the paper has
 * none). Each site is a host call the library makes; when an armed site fires,
 * the library reports that call as failed instead of making it. No device code
 * is involved and nothing faults, traps or hangs on the GPU. */
typedef enum {
  TKV_FAULT_NONE = 0,
  /* the workspace set-up inside tkv_create (event creation, clearing and
   * initialising the device workspace): tkv_create returns TKV_ERR_CUDA,
   * *out stays NULL and nothing the attempt created is left behind */
  TKV_FAULT_ALLOC = 1,
  /* a copy of caller host data to the device: the three input copies of
   * tkv_decode_step_host and the copy of tkv_set_scores. Both run before
   * anything changes: TKV_ERR_CUDA, state unchanged, handle usable */
  TKV_FAULT_H2D = 2,
  /* a copy of device data to a caller host buffer: tkv_get_scores,
   * tkv_get_kv_row of a T0 row and the output of tkv_decode_step_host.
   * TKV_ERR_CUDA, buffer not written, handle usable; for
   * tkv_decode_step_host the step itself has taken effect */
  TKV_FAULT_D2H = 3,
  /* the enqueue of one layer group's T1/T2 prefetch (STREAM mode; a decode
   * step makes one per layer group, tkv_prefetch one): a decode step stops
   * half done, so TKV_ERR_CUDA marks the handle broken; the work already
   * enqueued drains and tkv_destroy returns */
  TKV_FAULT_PREFETCH = 4,
  /* the allocator of the next reassignment finds a pool full: TKV_ERR_CAPACITY
   * with tiers, page tables and scores unchanged, handle usable */
  TKV_FAULT_CLASSIFY_OVERFLOW = 5
} tkv_fault_site;

/* Arms `site` so that the countdown-th time it is reached from now on
 * (1 = the next time) it fails; one site per handle is armed at a time and
 * firing disarms it; TKV_FAULT_NONE disarms. TKV_FAULT_ALLOC takes h = NULL
 * and counts the set-up calls of the next tkv_create only (a countdown beyond
 * them is dropped). The environment variable TKV_FAULT="<site>[:<countdown>]"
 * with site alloc | h2d | d2h | prefetch | classify_overflow arms the same
 * faults at each tkv_create (alloc: that create; others: the new handle).
 * Errors: TKV_ERR_INVALID_ARG for an unknown site, a countdown < 1, or a
 * handle given with TKV_FAULT_ALLOC / missing for the others. */
TKV_API tkv_status tkv_test_inject_fault(tkv_handle h, int32_t site, int32_t countdown);

/* Test hook, host only (no device work; the paper has no counterpart): the
 * attention work plan a decode step uses. Sequence b has full_pages[b] T0 + T1
 * pages and i8_pages[b] T2 pages (a T2 page costs 1.5 full pages). Writes
 * chunk_first[0..B] (prefix sums of the chunks each sequence's page list is
 * split into, equal in cost; one work unit per chunk, KV head and layer),
 * order[0..B) (the sequences by decreasing chunk cost, ties by index: the
 * order in which units are handed out), order_chunk_first[0..B] (prefix sums
 * of the chunk counts in that order) and *page_bound (pages of the largest
 * chunk, an upper bound). resident_ctas: attention CTAs resident at once;
 * split_pages: pages per chunk, 0 = automatic (whole waves of resident CTAs).
 * Errors: TKV_ERR_INVALID_ARG for batch outside 1..64, a page count outside
 * 0..16384, n_kv_heads < 1, resident_ctas < 1, split_pages < 0 or a null
 * pointer. */
TKV_API tkv_status tkv_test_plan_attention(int32_t batch, const int64_t* full_pages, const int64_t* i8_pages,
                                           int32_t n_kv_heads, int32_t split_pages, int32_t resident_ctas,
                                           int32_t* chunk_first, int32_t* order, int32_t* order_chunk_first,
                                           int32_t* page_bound);

/* 1 when this library is the debug build (compiled with TKV_DEBUG), else 0.
 * The debug build checks on the device every page id, page-list index, score
 * position and staging row a kernel derives from the bookkeeping against the
 * area it indexes; a failed check records the check, the index and its bound
 * and skips the access it guards (no trap), and the next synchronising call
 * returns TKV_ERR_INTERNAL with those details and marks the handle broken.
 * Release builds compile the checks away. */
TKV_API int32_t tkv_debug_build(void);

/* Test hook of the debug build (the paper has no counterpart): overwrites
 * entry `index` of sequence seq's tier-`tier` page list (tier 0..2) in the
 * device page table with that tier pool's capacity, the first page id past
 * the pool's end, and returns it in *planted. Every address such an id can
 * form lies inside the workspace that holds the pool (later regions of it
 * follow each pool), so even an unchecked use would read allocated memory. The host
 * bookkeeping keeps the true entry and the next metadata upload (an append or
 * a reassignment) restores it; until then the index checks catch the id at
 * the next decode step. Errors: TKV_ERR_STATE in a release build (nothing is
 * written); TKV_ERR_INVALID_ARG for a bad sequence, tier or index. */
TKV_API tkv_status tkv_test_plant_bad_page(tkv_handle h, int32_t seq, int32_t tier, int64_t index, int32_t* planted);

/* Introspection and test hooks (host buffers; each synchronises). The scores
 * are the s_i of Methodology 2, the tiers those of Methodology 1; page tables
 * follow this library's slot rule (the paper fixes none). Errors:
 * TKV_ERR_INVALID_ARG for a bad sequence, position or tier. */
TKV_API tkv_status tkv_num_sequences(tkv_handle h, int32_t* n);
TKV_API tkv_status tkv_seq_len(tkv_handle h, int32_t seq, int64_t* n_tokens);
TKV_API tkv_status tkv_get_scores(tkv_handle h, int32_t seq, double* host_out, int64_t n);
/* Replace the scores of positions [0, n); NaN is rejected, -0 becomes +0. */
TKV_API tkv_status tkv_set_scores(tkv_handle h, int32_t seq, const double* host_in, int64_t n);
TKV_API tkv_status tkv_get_tiers(tkv_handle h, int32_t seq, uint8_t* host_out, int64_t n);
/* Pages of one tier of one sequence in page order: pages[i] its pool id,
 * valid_mask[i] the 16-bit slot mask, positions[16 i + j] the position in
 * slot j or -1. Writes min(cap, count) entries and the count to *n_out. */
TKV_API tkv_status tkv_get_page_table(tkv_handle h, int32_t seq, int32_t tier, int32_t* pages,
                              uint16_t* valid_mask, int32_t* positions, int64_t cap,
                              int64_t* n_out);
/* 8-bit codes of a T2 position: codes [L][2][Hkv][d] (K then V), scales
 * [L][2] float32 (per token) or [L][2][Hkv] float16 (per token and head). */
TKV_API tkv_status tkv_get_t2_row(tkv_handle h, int32_t seq, int64_t pos, int8_t* codes, void* scales);
/* Values held by a T0 or T1 position: k, v [L][Hkv][d] in the KV dtype, the
 * full-precision values Proposition 1 relies on (Methodology 3). */
TKV_API tkv_status tkv_get_kv_row(tkv_handle h, int32_t seq, int64_t pos, void* k, void* v);
TKV_API tkv_status tkv_get_stats(tkv_handle h, tkv_stats* out);
TKV_API tkv_status tkv_reset_stats(tkv_handle h);
/* Message of the last failed call on h (or of the last failed handle-less
 * call when h is NULL); never NULL. */
TKV_API const char* tkv_last_error(tkv_handle h);

/* ---- stateless kernels -------------------------------------------------- */

/* Split-K paged decode attention over one full-precision page pool, with the
 * score increment of Methodology 2 fused into the softmax epilogue.
 *   q        device [B][Hq][d]           (KV dtype)
 *   pool     device [n_pages][Hkv][2][16][d]  page p, head h: K rows then V rows
 *   page_table device int32 [B][max_pages]  pool ids of each sequence's pages
 *   slot_mask  device uint32 [n_pages]      bit j set = slot j holds a token
 *   page_counts HOST int32 [B]              pages used by each sequence (max_pages <= 16384)
 *   out      device [B][Hq][d]           (KV dtype)
 *   alpha_sum device float [B][Hkv][max_pages * 16] (16-byte aligned) or NULL: adds, for each slot,
 *            the softmax weight summed over the G query heads of KV head h (slot order = page
 *            table order); multiply by 1/(L * Hq) and sum over layers for s.
 *   scratch  device, tkv_paged_attention_scratch_size bytes (256-aligned); its
 *            first int32 is 0 after the call, or 1 if a bounded wait gave up.
 * Returns after enqueueing on `stream`. */
TKV_API tkv_status tkv_paged_attention_scratch_size(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                                            int32_t head_dim, int32_t max_pages,
                                            size_t* scratch_bytes);
TKV_API tkv_status tkv_paged_attention(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                               int32_t head_dim, int32_t kv_dtype, const void* q, const void* pool,
                               const int32_t* page_table, const uint32_t* slot_mask,
                               const int32_t* page_counts, int32_t max_pages, void* out,
                               float* alpha_sum, void* scratch, size_t scratch_bytes,
                               tkv_stream stream);

/* Allocation-free form of tkv_paged_attention. The paper has no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc — for
 * example an inference-engine plugin whose per-step hook must not allocate, or
 * a process whose framework has already reserved all device memory for its own
 * pool — and so cannot provide the scratch buffer tkv_paged_attention needs.
 * Arguments are those of tkv_paged_attention without scratch and
 * scratch_bytes; the caller still passes every input and output.
 *   Scratch: a fixed 16 MiB array in the library's device code, which every
 *   GPU that loads the library holds until the process exits. Shapes whose
 *   scratch (tkv_paged_attention_scratch_size) exceeds 16 MiB are rejected
 *   with TKV_ERR_CAPACITY and nothing is launched.
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 *   The cached address is valid for the device's current context only: after
 *   cudaDeviceReset the library must be reloaded.
 *   Sharing: every call on a device uses the same array and the array keeps
 *   the last call's contents; each call clears the parts that must start at
 *   zero. Calls that overlap on the GPU (other streams, other threads) race on
 *   it: serialise them.
 *   Status: the kernels' error word sits in that array, out of the caller's
 *   reach; read it with tkv_paged_attention_noalloc_status. */
TKV_API tkv_status tkv_paged_attention_noalloc(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                                               int32_t head_dim, int32_t kv_dtype, const void* q,
                                               const void* pool, const int32_t* page_table,
                                               const uint32_t* slot_mask, const int32_t* page_counts,
                                               int32_t max_pages, void* out, float* alpha_sum,
                                               tkv_stream stream);
/* Device status word of the last allocation-free call on the current device:
 * after the work enqueued on `stream` so far, *host_out = 0 (no error), 1 (a
 * bounded device wait gave up; that call's output is not valid) or 2 (an
 * internal index check failed). Copies 4 bytes to the host and synchronises
 * `stream`; allocates nothing. TKV_ERR_STATE if no allocation-free call has
 * run on this device. The paper has no counterpart. */
TKV_API tkv_status tkv_paged_attention_noalloc_status(int32_t* host_out, tkv_stream stream);

/* Tier reassignment of Methodology 1 for B sequences (device buffers):
 *   scores   double [B][stride], old_tier uint8 [B][stride], new_tier uint8 [B][stride]
 *   params   HOST int64 [B][5] = {N, prompt_len, n0, n1, n2} per sequence
 * Candidates (not protected, not already T3) are ranked by score descending,
 * ties by lower position; the first max(n0 - |P|, 0) go to T0, the next n1 to
 * T1, the next n2 to T2, the rest to T3; protected positions go to T0. */
TKV_API tkv_status tkv_classify_scratch_size(int32_t batch, int64_t stride, size_t* scratch_bytes);
TKV_API tkv_status tkv_classify(int32_t batch, const double* scores, const uint8_t* old_tier,
                        uint8_t* new_tier, int64_t stride, const int64_t* params, int32_t n_sink,
                        int32_t recent_window, void* scratch, size_t scratch_bytes,
                        tkv_stream stream);

/* Symmetric absmax 8-bit quantisation of `rows` rows of `row_len` values
 * (device x in kv_dtype): scale = absmax/127 in float32 (then float16 if
 * scale_dtype is F16), code = clamp(rint(x / scale), -127, 127); an all-zero
 * row gives scale 0 and codes 0. codes int8 [rows][row_len], scales [rows]. */
TKV_API tkv_status tkv_quantize_rows(const void* x, int32_t kv_dtype, int64_t rows, int32_t row_len,
                             int8_t* codes, void* scales, int32_t scale_dtype, tkv_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* TKV_H_ */
