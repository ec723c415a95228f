// Host runtime of libtkv: the C ABI of include/tkv.h.
//
// It owns the bookkeeping of the four-tier cache of "Not All Thoughts Need
// HBM" — which tier and which (page, slot) every position occupies, the page
// lists of each sequence, the pools' page counters — and orchestrates one
// decode step: append (Methodology 1: the recent window is in T0), per-layer
// prefetch of T1 and T2 on the copy stream overlapped with the previous
// layer's attention (Methodology 4), split-K attention with the fused score
// epilogue (Methodology 2, 3), the float64 score fold, and every Delta steps
// the reassignment (classifier kernel) and the differential data movement
// (only tokens whose tier changed move; Methodology 4).
//
// Slot rule (the page fixes none; this is the reading used throughout): a
// token that keeps its tier keeps its slot; arrivals, in ascending position,
// fill the sequence's holes in ascending (page id, slot) order, then take a new
// page (the pool's lowest freed id, else the next never-used id); a sequence's
// pages are kept in ascending id. After each reassignment the T0 pages of a
// sequence are compacted into its first ceil(n / 16) pages (moves inside HBM
// only) and the emptied pages are freed. Sequences are served in ascending order.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>
#include <queue>
#include <string>
#include <vector>

#include "tkv.h"
#include "tkv_internal.h"

using namespace tkv;

namespace {

thread_local std::string g_last_error = "no error";

constexpr size_t kAlign = 256;
constexpr size_t kStartedWordOffset = 32;  // byte offset of the started word in the error region
constexpr size_t kEpOffset = 64;           // byte offset of the epilogue counter sets in the error region
constexpr size_t kErrRegion = 2048;        // bytes of the error region
static_assert(kEpOffset + 4 * sizeof(EpCounters) <= kErrRegion, "error region too small");
size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
#ifndef TKV_EP_FIRST_DIV
#define TKV_EP_FIRST_DIV 3
#endif
// One in kEpFirstDiv attention CTAs starts on the previous launch's epilogue
// items (0: none), while the rest stream pages, when the epilogue's bytes are at
// least kEpFirstShare of the attention bytes. Measured per 7-layer launch at
// batch 32 (share 7 %): 1.519 ms per step against 1.583 with items only in the
// tail; 4 x 131k (share 4.7 %, 128 items of 3 MB): 0.93 of the HBM peak against
// 0.85; MHA 8 x 16k (share 2.3 %): 0.95 against 0.97, so there the tail keeps them.
constexpr int kEpFirstDiv = TKV_EP_FIRST_DIV;
constexpr double kEpFirstShare = 0.035;
// a pool capacity as the int32 page bound of the device index checks
int32_t cap32(int64_t pages) { return static_cast<int32_t>(std::min<int64_t>(pages, INT32_MAX)); }

using MinHeap = std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>>;

struct Seq {
  int64_t N = 0, prompt_len = 0;
  std::vector<uint8_t> tier;
  std::vector<int32_t> loc;      // page * 16 + slot in the pool of its tier; -1 when T3
  std::vector<int32_t> pages[3]; // page ids per tier, in acquisition (= ascending) order
  MinHeap holes[3];              // page * 16 + slot of free slots in those pages
};

// Sizes derived from a configuration; shared by tkv_workspace_size and tkv_create.
struct Layout {
  int L, Hq, Hkv, D, G, esz, maxb;
  int Lg;                // layers per attention launch (and per prefetch in STREAM mode)
  int mode;              // TKV_HOST_TIERS_*
  int64_t maxtok, maxp;
  int64_t cap[3];
  int64_t total_pages;   // pages of all three pools: bounds the pages of all sequences together
  int64_t plb[3];        // bytes of one page record per layer (T2: int8 codes)
  int64_t scale_rec;     // bytes of one T2 scale record per page per layer
  int64_t max_chunks, spill_stride, temp_rows;
  // device offsets
  size_t o_pool0, o_stage1, o_stage2c, o_stage2s, o_mirror1, o_mirror2c, o_mirror2s, o_table, o_mask, o_posmap, o_tier, o_tier_new,
      o_s, o_acc, o_part_o, o_part_m, o_part_z, o_spill, o_keys, o_cls_state, o_cls_ties, o_err, o_span, o_movers,
      o_temp, o_locs, o_io, dev_bytes;
  size_t io_q, io_k, io_out;
  // pinned offsets
  size_t p_pool1, p_pool2c, p_pool2s, p_arena, arena_bytes, pinned_bytes;
};

bool budget_pages(const tkv_config& c, int tier, int64_t maxtok, int64_t* pages) {
  int64_t count;
  if (c.budget_mode == TKV_BUDGET_PERCENT)
    count = c.budget[tier] * maxtok / 100;
  else
    count = tier < 3 ? c.budget[tier] : maxtok;
  count = std::min(count, maxtok);
  *pages = ceil_div(std::max<int64_t>(count, 0), kPage) + 1;
  return true;
}

std::string validate(const tkv_config& c) {
  char buf[256];
  auto bad = [&](const char* what) { std::snprintf(buf, sizeof buf, "invalid config: %s", what); return std::string(buf); };
  if (c.n_layers < 1 || c.n_layers > 4096) return bad("n_layers out of range");
  if (c.n_q_heads < 1 || c.n_kv_heads < 1 || c.n_q_heads % c.n_kv_heads) return bad("n_q_heads must be a multiple of n_kv_heads");
  if (!attention_supported(c.kv_dtype, c.n_q_heads / c.n_kv_heads, c.head_dim))
    return bad("unsupported (Hq/Hkv, head_dim): group size must be 1, 2, 4, 7 or 8 and head_dim 64 or 128");
  if (c.kv_dtype != TKV_DTYPE_F32 && c.kv_dtype != TKV_DTYPE_BF16) return bad("kv_dtype");
  if (c.max_batch < 1 || c.max_batch > kMaxBatch) return bad("max_batch must be 1..64");
  if (c.max_tokens < 1 || c.max_tokens > int64_t(kMaxSeqPages) * kPage - 4 * kPage)
    return bad("max_tokens out of range (1 .. 262080)");
  if (c.page_size != kPage) return bad("page_size must be 16");
  if (c.n_sink < 0 || c.recent_window < 0) return bad("n_sink / recent_window negative");
  if (c.budget_mode == TKV_BUDGET_PERCENT) {
    int64_t s = 0;
    for (int i = 0; i < 4; ++i) {
      if (c.budget[i] < 0 || c.budget[i] > 100) return bad("percent budgets must be 0..100");
      s += c.budget[i];
    }
    if (s != 100) return bad("percent budgets must sum to 100");
  } else if (c.budget_mode == TKV_BUDGET_COUNT) {
    for (int i = 0; i < 3; ++i)
      if (c.budget[i] < 0) return bad("count budgets must be >= 0");
  } else {
    return bad("budget_mode");
  }
  if (c.reclassify_interval < 1) return bad("reclassify_interval must be >= 1");
  const bool combo_ok = (c.t2_scale_gran == TKV_SCALE_PER_TOKEN && c.t2_scale_dtype == TKV_SCALE_F32) ||
                        (c.t2_scale_gran == TKV_SCALE_PER_TOKEN_HEAD && c.t2_scale_dtype == TKV_SCALE_F16);
  if (!combo_ok) return bad("T2 scales: per-token scales are float32, per-token-head scales float16");
  if (c.t2_mode != TKV_T2_ATTEND && c.t2_mode != TKV_T2_MASK) return bad("t2_mode");
  if (c.t0_pages < 0 || c.t1_pages < 0 || c.t2_pages < 0 || c.max_staged_movers < 0) return bad("negative capacity");
  if (c.split_pages < 0 || c.split_pages > kMaxChunkPages) return bad("split_pages must be 0..256");
  if (c.host_tiers != TKV_HOST_TIERS_STREAM && c.host_tiers != TKV_HOST_TIERS_MIRROR &&
      c.host_tiers != TKV_HOST_TIERS_ZEROCOPY)
    return bad("host_tiers");
  if (c.layers_per_launch < 0) return bad("layers_per_launch must be >= 0");
  return std::string();
}

// Layers per attention launch: the configured count (at most L), else the
// largest divisor of L up to 7, or up to 14 when one layer's K and V at full
// capacity are under 64 MB. Each launch pays a fixed start-up, tail and launch
// cost; on the batch-32 workload one layer per launch ran the kernel at 60 % of
// the measured HBM peak, 4 layers at 67 % and 7 at 72 %; a single 2k-token
// request, where a launch is ~20 us of fixed cost, took 142 us per 28-layer step
// with 7 layers per launch, 111 us with 14 and 117 us with 28. In STREAM mode
// the staging ring holds two groups, so the grouping costs 2 x 7 layers of the
// used T1 / T2 range in HBM.
int layers_per_launch(const tkv_config& c) {
  if (c.layers_per_launch > 0) return std::min({c.layers_per_launch, c.n_layers, kMaxLaunchLayers});
  const int64_t esz = c.kv_dtype == TKV_DTYPE_BF16 ? 2 : 4;
  const int64_t layer_bytes = int64_t(c.max_batch) * c.max_tokens * 2 * c.n_kv_heads * c.head_dim * esz;
  const int cap = layer_bytes < (int64_t(64) << 20) ? 14 : 7;
  int best = 1;
  for (int g = 1; g <= std::min(cap, c.n_layers); ++g)
    if (c.n_layers % g == 0) best = g;
  return best;
}

Layout make_layout(const tkv_config& c) {
  Layout y{};
  y.L = c.n_layers; y.Hq = c.n_q_heads; y.Hkv = c.n_kv_heads; y.D = c.head_dim;
  y.Lg = layers_per_launch(c);
  y.mode = c.host_tiers;
  y.G = y.Hq / y.Hkv; y.esz = c.kv_dtype == TKV_DTYPE_BF16 ? 2 : 4; y.maxb = c.max_batch;
  y.maxtok = c.max_tokens;
  y.maxp = ceil_div(y.maxtok, kPage) + 1;
  int64_t per[3];
  per[0] = y.maxp;
  budget_pages(c, 1, y.maxtok, &per[1]);
  budget_pages(c, 2, y.maxtok, &per[2]);
  y.cap[0] = c.t0_pages ? c.t0_pages : y.maxb * per[0];
  y.cap[1] = c.t1_pages ? c.t1_pages : y.maxb * per[1];
  y.cap[2] = c.t2_pages ? c.t2_pages : y.maxb * per[2];
  y.plb[0] = y.plb[1] = int64_t(y.Hkv) * 2 * kPage * y.D * y.esz;
  y.plb[2] = int64_t(y.Hkv) * 2 * kPage * y.D;
  y.scale_rec = c.t2_scale_gran == TKV_SCALE_PER_TOKEN ? 2 * kPage * 4 : int64_t(y.Hkv) * 2 * kPage * 2;
  y.total_pages = y.cap[0] + y.cap[1] + y.cap[2];
  // a sequence of n pages gets at most min(128, ceil(n / 8)) chunks (plan_chunks)
  y.max_chunks = std::min<int64_t>(int64_t(y.maxb) * kMaxChunksPerSeq, ceil_div(y.total_pages, 8) + y.maxb);
  y.spill_stride = y.total_pages * y.G * kPage;   // floats per (layer slice, KV head)
  // staging rows hold one layer (phase-2 moves run layer by layer); by default
  // one per position, so any reassignment fits
  y.temp_rows = c.max_staged_movers ? c.max_staged_movers : int64_t(y.maxb) * y.maxtok;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  y.o_pool0 = take(size_t(y.L) * y.cap[0] * y.plb[0]);
  // STREAM: a two-slot staging ring, each slot one layer group of the T1 / T2
  // pools; MIRROR: device copies of all layers of those pools; ZEROCOPY: neither
  const size_t stage_layers = y.mode == TKV_HOST_TIERS_STREAM ? 2 * size_t(y.Lg) : 0;
  const size_t mirror_layers = y.mode == TKV_HOST_TIERS_MIRROR ? size_t(y.L) : 0;
  y.o_stage1 = take(stage_layers * y.cap[1] * y.plb[1]);
  y.o_stage2c = take(stage_layers * y.cap[2] * y.plb[2]);
  y.o_stage2s = take(stage_layers * y.cap[2] * y.scale_rec);
  y.o_mirror1 = take(mirror_layers * y.cap[1] * y.plb[1]);
  y.o_mirror2c = take(mirror_layers * y.cap[2] * y.plb[2]);
  y.o_mirror2s = take(mirror_layers * y.cap[2] * y.scale_rec);
  y.o_table = take(3 * size_t(y.maxb) * y.maxp * 4);
  y.o_mask = take(size_t(y.cap[0] + y.cap[1] + y.cap[2]) * 4);
  y.o_posmap = take(size_t(y.cap[0] + y.cap[1] + y.cap[2]) * kPage * 4);
  y.o_tier = take(size_t(y.maxb) * y.maxtok);
  y.o_tier_new = take(size_t(y.maxb) * y.maxtok);
  y.o_s = take(size_t(y.maxb) * y.maxtok * 8);
  // slot-indexed score increments, one slice per layer of a launch: [Lg][Hkv][total_pages][16]
  y.o_acc = take(size_t(y.Lg) * y.Hkv * y.total_pages * kPage * 4);
  // partials and spilled logits: two launches' worth, since each launch's
  // epilogue runs inside the next attention launch
  y.o_part_o = take(2 * size_t(y.Lg) * y.max_chunks * y.Hkv * y.G * y.D * 4);
  y.o_part_m = take(2 * size_t(y.Lg) * y.max_chunks * y.Hkv * y.G * 4);
  y.o_part_z = take(2 * size_t(y.Lg) * y.max_chunks * y.Hkv * y.G * 4);
  y.o_spill = take(2 * size_t(y.Lg) * y.Hkv * y.spill_stride * 4);
  y.o_keys = take(size_t(y.maxb) * y.maxtok * 8);
  y.o_cls_state = take(size_t(y.maxb) * sizeof(ClassifyState));
  y.o_cls_ties = take(size_t(y.maxb) * classify_slices(y.maxtok) * 3 * 8);
  y.o_err = take(kErrRegion);   // int32 [0]: device error word; from byte 64: four sets of epilogue counters;
                        // [8]: sequence number of the last attention launch that started
  y.o_span = take(size_t(kSpanSlots) * 16);  // device span (start, end) of attention launches, by sequence number
  y.o_movers = take(2 * size_t(y.maxb) * y.maxtok * sizeof(Mover));
  y.o_temp = take(size_t(y.temp_rows) * 2 * y.Hkv * y.D * y.esz);
  y.o_locs = take(size_t(y.maxtok) * 4);
  const size_t q_bytes = size_t(y.maxb) * y.L * y.Hq * y.D * y.esz;
  const size_t kv_bytes = size_t(y.maxb) * y.L * y.Hkv * y.D * y.esz;
  y.io_q = 0;
  y.io_k = align_up(q_bytes);
  y.io_out = y.io_k + 2 * align_up(kv_bytes);
  y.o_io = take(y.io_out + q_bytes);
  y.dev_bytes = o;
  o = 0;
  y.p_pool1 = take(size_t(y.L) * y.cap[1] * y.plb[1]);
  y.p_pool2c = take(size_t(y.L) * y.cap[2] * y.plb[2]);
  y.p_pool2s = take(size_t(y.L) * y.cap[2] * y.scale_rec);
  const size_t arena = align_up(size_t(y.maxb) * y.maxtok) +                       // tier read-back
                       align_up(2 * size_t(y.maxb) * y.maxtok * sizeof(Mover)) +   // movers
                       align_up(3 * size_t(y.maxb) * y.maxp * 4) +                 // page tables
                       align_up(size_t(y.cap[0] + y.cap[1] + y.cap[2]) * 4) +      // masks
                       align_up(size_t(y.cap[0] + y.cap[1] + y.cap[2]) * kPage * 4) +  // posmaps
                       align_up(size_t(y.maxtok) * 4);                              // prefill slots
  y.arena_bytes = arena;
  y.p_arena = take(arena);
  y.pinned_bytes = o;
  return y;
}

// The driver's stream memory wait (cuStreamWaitValue32, "wait until
// (int32_t)(*addr - value) >= 0"), obtained at run time so that the library
// links against the runtime alone.
typedef int (*WaitValue32Fn)(void* stream, unsigned long long addr, unsigned int value, unsigned int flags);
constexpr unsigned int kWaitGeq = 0;

struct TimedPair {
  cudaEvent_t a, b;
  int kind;  // 0 attention stream kernel, 1 prefetch, 2 combine / score kernel
};

}  // namespace

struct tkv_ctx {
  tkv_config cfg;
  Layout y;
  int device = 0;
  char* dev = nullptr;
  char* pin = nullptr;       // host address of the pinned workspace
  char* pin_dev = nullptr;   // the same memory as seen by kernels
  cudaStream_t cs = nullptr, xs = nullptr;
  cudaEvent_t ev_ready[2] = {nullptr, nullptr}, ev_free[2] = {nullptr, nullptr};
  int slot_rr = 0;
  int64_t steps = 0;
  int64_t attn_launch_seq = 0;    // attention launches so far: their parity picks buffers and counters
  int64_t last_launch_seq = 0;    // number of the last attention launch actually enqueued (0: none)
  bool stall_next = false;        // test hook: the next attention launch withholds one page
  unsigned long long wait_limit_ns = 2000000000ull;  // bounded device waits give up after this long
  bool ahead_valid = false;       // the next step's first layer group is staged in ahead_slot
  int ahead_slot = 0;
  int32_t fault_site = TKV_FAULT_NONE;  // test hook: host call reported as failed when its countdown ends
  int32_t fault_countdown = 0;
  int64_t span_from = 0;          // first attention launch counted in attn_span_ms
  // Copy-stream gate: a prefetch waits (stream memory wait) until the previous
  // attention launch has started, so that launch is not made behind a host
  // link that the next prefetch already saturates. Null where unsupported.
  WaitValue32Fn wait_value = nullptr;
  int64_t next_page[3] = {0, 0, 0};
  MinHeap free_pages[3];          // freed page ids per tier pool
  std::vector<Seq> seqs;
  std::vector<uint32_t> mask[3];
  std::vector<int32_t> posmap[3];
  std::vector<int32_t> table[3];  // [maxb][maxp]
  bool broken = false;
  std::string err = "no error";
  tkv_stats stats{};
  std::vector<TimedPair> pending, spare;
  uint8_t* d_tier = nullptr;
  uint8_t* d_tier_new = nullptr;
  int resident_ctas = 304;  // attention CTAs resident on the whole GPU at once

  char* D(size_t off) const { return dev + off; }
  char* P(size_t off) const { return pin + off; }
  char* PD(size_t off) const { return pin_dev + off; }
};

namespace {

tkv_status fail(tkv_ctx* h, tkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  if (h) h->err = buf;
  return st;
}

tkv_status fail_cuda(tkv_ctx* h, const char* what, cudaError_t e) {
  if (h) h->broken = true;
  return fail(h, TKV_ERR_CUDA, "%s failed: %s", what, cudaGetErrorString(e));
}

// ---- host-side fault injection (tkv_test_inject_fault, TKV_FAULT)

// Set-up calls of the next tkv_create until one is reported as failed (0: off).
std::atomic<int32_t> g_create_fault{0};

// True when `site` is armed on h and its countdown ends with this visit.
bool fault_fires(tkv_ctx* h, int32_t site) {
  if (!h || site == TKV_FAULT_NONE || h->fault_site != site) return false;
  if (--h->fault_countdown > 0) return false;
  h->fault_site = TKV_FAULT_NONE;
  return true;
}

tkv_status injected(tkv_ctx* h, const char* what) {
  return fail(h, TKV_ERR_CUDA, "%s failed: injected host-side fault", what);
}

// TKV_FAULT="<site>[:<countdown>]"; false when unset or malformed.
bool fault_from_env(int32_t* site, int32_t* countdown) {
  const char* v = std::getenv("TKV_FAULT");
  if (!v || !*v) return false;
  static const struct { const char* name; int32_t site; } names[] = {
      {"alloc", TKV_FAULT_ALLOC}, {"h2d", TKV_FAULT_H2D}, {"d2h", TKV_FAULT_D2H},
      {"prefetch", TKV_FAULT_PREFETCH}, {"classify_overflow", TKV_FAULT_CLASSIFY_OVERFLOW}};
  const char* colon = std::strchr(v, ':');
  const size_t n = colon ? size_t(colon - v) : std::strlen(v);
  long cd = 1;
  if (colon) {
    char* end = nullptr;
    cd = std::strtol(colon + 1, &end, 10);
    if (end == colon + 1 || *end != '\0' || cd < 1 || cd > INT32_MAX) return false;
  }
  for (const auto& e : names)
    if (std::strlen(e.name) == n && std::strncmp(v, e.name, n) == 0) {
      *site = e.site;
      *countdown = static_cast<int32_t>(cd);
      return true;
    }
  return false;
}

// A copy between caller memory and the device made before anything changes or
// after everything has: its failure leaves the handle usable (a failure that
// took the context down shows again at the next synchronising call).
#define CK_SOFT(h, what, call)                                                              \
  do {                                                                                      \
    cudaError_t e_ = (call);                                                                \
    if (e_ != cudaSuccess) {                                                                \
      (void)cudaGetLastError();                                                             \
      return fail((h), TKV_ERR_CUDA, "%s failed: %s", (what), cudaGetErrorString(e_));      \
    }                                                                                       \
  } while (0)

#define CK(h, call)                                            \
  do {                                                         \
    cudaError_t e_ = (call);                                   \
    if (e_ != cudaSuccess) return fail_cuda((h), #call, e_);   \
  } while (0)

// A kernel launch that took place when `launched` holds (launchers return
// early without a launch on empty work); counted in the handle's statistics.
#define LK(h, call, launched)                                  \
  do {                                                         \
    CK(h, call);                                               \
    if (launched) (h)->stats.kernel_launches += 1;             \
  } while (0)

tkv_status check_usable(tkv_ctx* h) {
  if (!h) return fail(nullptr, TKV_ERR_INVALID_ARG, "null handle");
  if (h->broken) return fail(h, TKV_ERR_STATE, "handle is broken by an earlier CUDA failure: %s", h->err.c_str());
  return TKV_OK;
}

// Harvest finished timing events into the stats.
void harvest(tkv_ctx* h) {
  for (auto& tp : h->pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, tp.a, tp.b) == cudaSuccess) {
      if (tp.kind == 0)
        h->stats.attn_ms += ms;
      else if (tp.kind == 1)
        h->stats.prefetch_ms += ms;
      else
        h->stats.combine_ms += ms;
    }
    h->spare.push_back(tp);
  }
  h->pending.clear();
  (void)cudaGetLastError();
}

tkv_status timed_pair(tkv_ctx* h, int kind, TimedPair* out) {
  if (h->spare.empty()) {
    TimedPair tp{};
    CK(h, cudaEventCreate(&tp.a));
    CK(h, cudaEventCreate(&tp.b));
    h->spare.push_back(tp);
  }
  *out = h->spare.back();
  h->spare.pop_back();
  out->kind = kind;
  return TKV_OK;
}

tkv_status sync_all(tkv_ctx* h) {
  CK(h, cudaStreamSynchronize(h->cs));
  if (h->xs != h->cs) CK(h, cudaStreamSynchronize(h->xs));
  // error word, site, index, bound (the last three written by the debug build's index checks)
  int32_t rec[6] = {0, 0, 0, 0, 0, 0};
  CK(h, cudaMemcpy(rec, h->D(h->y.o_err), sizeof rec, cudaMemcpyDeviceToHost));
  const int32_t e = rec[0];
  harvest(h);
  if (e == DEV_TIMEOUT) {
    h->broken = true;
    return fail(h, TKV_ERR_TIMEOUT, "a bounded device wait gave up (copy never landed)");
  }
  if (e == DEV_BAD_INDEX) {
    h->broken = true;
    static const char* const kSite[kDebugSites] = {
        "attention chunk larger than the page limit", "attention page-list index", "attention page id",
        "score fold page id", "score fold position", "append page id", "append page-list length",
        "prefill page id", "mover source page", "mover destination page", "mover staging row"};
    const int site = rec[1];
    long long idx = 0, bound = 0;
    std::memcpy(&idx, rec + 2, 8);
    std::memcpy(&bound, rec + 4, 8);
    if (site <= DBG_NONE || site >= kDebugSites)
      return fail(h, TKV_ERR_INTERNAL, "device index check failed: %s", kSite[0]);
    return fail(h, TKV_ERR_INTERNAL, "device index check failed: %s %lld outside [0, %lld)", kSite[site], idx, bound);
  }
  if (e != 0) {
    h->broken = true;
    return fail(h, TKV_ERR_INTERNAL, "device reported error code %d", e);
  }
  return TKV_OK;
}

// Places `positions` (ascending) of sequence b in tier t: holes first, then new
// pages (lowest freed id, else the next never-used id), kept in ascending id.
// Returns false on capacity. *inserted_at receives the list index of the last
// page added (or is left untouched).
bool place(tkv_ctx* h, Seq& sq, int b, int t, const std::vector<int64_t>& positions,
           std::vector<int32_t>* locs_out, int* inserted_at = nullptr) {
  for (int64_t pos : positions) {
    if (sq.holes[t].empty()) {
      if (int64_t(sq.pages[t].size()) >= h->y.maxp) return false;
      int64_t page;
      if (!h->free_pages[t].empty()) {
        page = h->free_pages[t].top();
        h->free_pages[t].pop();
      } else {
        if (h->next_page[t] >= h->y.cap[t]) return false;
        page = h->next_page[t]++;
      }
      std::vector<int32_t>& pl = sq.pages[t];
      auto it = std::lower_bound(pl.begin(), pl.end(), static_cast<int32_t>(page));
      const size_t at = size_t(it - pl.begin());
      pl.insert(it, static_cast<int32_t>(page));
      for (size_t i = at; i < pl.size(); ++i) h->table[t][size_t(b) * h->y.maxp + i] = pl[i];
      if (inserted_at) *inserted_at = static_cast<int>(at);
      for (int s = 0; s < kPage; ++s) sq.holes[t].push(page * kPage + s);
    }
    const int64_t code = sq.holes[t].top();
    sq.holes[t].pop();
    const int64_t page = code / kPage, slot = code % kPage;
    h->mask[t][page] |= 1u << slot;
    h->posmap[t][page * kPage + slot] = static_cast<int32_t>(pos);
    sq.loc[pos] = static_cast<int32_t>(code);
    sq.tier[pos] = static_cast<uint8_t>(t);
    if (locs_out) locs_out->push_back(static_cast<int32_t>(code));
  }
  return true;
}

// Packs sequence b's T0 tokens into its first ceil(n / 16) pages; appends the
// T0 -> T0 moves to `out` and frees the emptied pages.
void compact_t0(tkv_ctx* h, Seq& sq, int b, std::vector<Mover>& out) {
  std::vector<int32_t>& pl = sq.pages[0];
  int64_t n = 0;
  for (int32_t pg : pl) n += __builtin_popcount(h->mask[0][pg]);
  const size_t keep = size_t(ceil_div(n, kPage));
  if (keep >= pl.size()) return;
  std::vector<std::pair<int64_t, int32_t>> movers;  // (position, old code)
  for (size_t i = keep; i < pl.size(); ++i)
    for (int s = 0; s < kPage; ++s) {
      const int32_t pos = h->posmap[0][size_t(pl[i]) * kPage + s];
      if (pos >= 0) movers.emplace_back(pos, pl[i] * kPage + s);
    }
  std::sort(movers.begin(), movers.end());
  std::vector<int32_t> holes;
  for (size_t i = 0; i < keep; ++i)
    for (int s = 0; s < kPage; ++s)
      if (!((h->mask[0][pl[i]] >> s) & 1u)) holes.push_back(pl[i] * kPage + s);
  for (size_t k = 0; k < movers.size(); ++k) {
    const int64_t pos = movers[k].first;
    const int32_t from = movers[k].second, to = holes[k];
    h->mask[0][from / kPage] &= ~(1u << (from % kPage));
    h->posmap[0][from] = -1;
    h->mask[0][to / kPage] |= 1u << (to % kPage);
    h->posmap[0][to] = static_cast<int32_t>(pos);
    sq.loc[pos] = to;
    out.push_back(Mover{b, 0, from, 0, to, -1});
  }
  for (size_t i = keep; i < pl.size(); ++i) {
    h->free_pages[0].push(pl[i]);
    h->table[0][size_t(b) * h->y.maxp + i] = 0;
  }
  pl.resize(keep);
  MinHeap fresh;
  for (size_t k = movers.size(); k < holes.size(); ++k) fresh.push(holes[k]);
  sq.holes[0].swap(fresh);
}

void vacate(tkv_ctx* h, Seq& sq, int t, int64_t pos) {
  const int64_t code = sq.loc[pos];
  const int64_t page = code / kPage, slot = code % kPage;
  h->mask[t][page] &= ~(1u << slot);
  h->posmap[t][page * kPage + slot] = -1;
  sq.holes[t].push(code);
  sq.loc[pos] = -1;
}

tkv_status upload_metadata(tkv_ctx* h) {
  const Layout& y = h->y;
  char* arena = h->P(y.p_arena);
  size_t off = align_up(size_t(y.maxb) * y.maxtok) + align_up(2 * size_t(y.maxb) * y.maxtok * sizeof(Mover));
  const size_t tbytes = size_t(y.maxb) * y.maxp * 4;
  for (int t = 0; t < 3; ++t) {
    std::memcpy(arena + off + t * tbytes, h->table[t].data(), tbytes);
    CK(h, cudaMemcpyAsync(h->D(y.o_table) + t * tbytes, arena + off + t * tbytes, tbytes,
                          cudaMemcpyHostToDevice, h->cs));
  }
  off += align_up(3 * tbytes);
  size_t moff = off, poff = off + align_up(size_t(y.cap[0] + y.cap[1] + y.cap[2]) * 4);
  int64_t base = 0;
  for (int t = 0; t < 3; ++t) {
    const size_t n = size_t(h->next_page[t]);
    if (n) {
      std::memcpy(arena + moff + base * 4, h->mask[t].data(), n * 4);
      CK(h, cudaMemcpyAsync(h->D(y.o_mask) + base * 4, arena + moff + base * 4, n * 4,
                            cudaMemcpyHostToDevice, h->cs));
      std::memcpy(arena + poff + base * kPage * 4, h->posmap[t].data(), n * kPage * 4);
      CK(h, cudaMemcpyAsync(h->D(y.o_posmap) + base * kPage * 4, arena + poff + base * kPage * 4,
                            n * kPage * 4, cudaMemcpyHostToDevice, h->cs));
    }
    base += y.cap[t];
  }
  return TKV_OK;
}

uint32_t* d_mask(tkv_ctx* h, int t) {
  int64_t base = 0;
  for (int i = 0; i < t; ++i) base += h->y.cap[i];
  return reinterpret_cast<uint32_t*>(h->D(h->y.o_mask)) + base;
}
int32_t* d_posmap(tkv_ctx* h, int t) {
  int64_t base = 0;
  for (int i = 0; i < t; ++i) base += h->y.cap[i];
  return reinterpret_cast<int32_t*>(h->D(h->y.o_posmap)) + base * kPage;
}
int32_t* d_table(tkv_ctx* h, int t) {
  return reinterpret_cast<int32_t*>(h->D(h->y.o_table)) + size_t(t) * h->y.maxb * h->y.maxp;
}

// Splits every sequence's page list into chunks, one attention CTA per
// (chunk, KV head). Chunks are balanced by cost (page_at_cost): the kernel
// splits each sequence into equal-cost chunks, and the number of chunks per
// sequence is chosen greedily to minimise the costliest chunk, so that the
// grid's last CTAs finish close to the typical one; the total fills whole
// waves of resident CTAs. Writes chunk_first[0..B] and returns the page bound.
int plan_chunks(const std::vector<int64_t>& ntot, const std::vector<int64_t>& cost, int Hkv, int split_pages,
                int resident_ctas, int32_t* chunk_first) {
  const int B = static_cast<int>(ntot.size());
  std::vector<int64_t> nch(B, 1), cap(B, 1);
  int64_t sum = 0;
  for (int64_t n : ntot) sum += n;
  for (int b = 0; b < B; ++b) {
    // at most kMaxChunkPages pages per chunk, at least ~8 pages per chunk
    const int64_t floor_b = std::max<int64_t>(1, ceil_div(cost[b], kMaxChunkCost));
    nch[b] = floor_b;
    cap[b] = std::max<int64_t>(floor_b, std::min<int64_t>(kMaxChunksPerSeq, std::max<int64_t>(ceil_div(ntot[b], 8), 1)));
  }
  if (split_pages > 0) {
    for (int b = 0; b < B; ++b)
      nch[b] = std::min(cap[b], std::max(nch[b], ceil_div(std::max<int64_t>(ntot[b], 1), split_pages)));
  } else {
    // whole waves of resident CTAs with up to ~240 pages per chunk: each CTA pays
    // a fixed start-up, partial write and finish spread, so long contexts run
    // best in few waves of large chunks (measured: 4 x 131k tokens went from 8
    // waves of ~68 pages at 55 % of HBM peak to 3 waves of ~182 pages at 78 %)
    int64_t waves = std::max<int64_t>(1, ceil_div(sum * Hkv, int64_t(resident_ctas) * 240));
    waves = std::min<int64_t>(waves, 8);
    const int64_t target = std::max<int64_t>(B, waves * resident_ctas / Hkv);
    int64_t given = 0;
    for (int b = 0; b < B; ++b) given += nch[b];
    // greedy min-max: the next chunk goes to the sequence whose chunks are costliest
    auto worse = [&](int x, int y) { return cost[x] * nch[y] < cost[y] * nch[x]; };
    std::priority_queue<int, std::vector<int>, decltype(worse)> heap(worse);
    for (int b = 0; b < B; ++b)
      if (nch[b] < cap[b]) heap.push(b);
    while (given < target && !heap.empty()) {
      const int b = heap.top();
      heap.pop();
      ++nch[b];
      ++given;
      if (nch[b] < cap[b]) heap.push(b);
    }
  }
  int bound = 1;
  chunk_first[0] = 0;
  for (int b = 0; b < B; ++b) {
    chunk_first[b + 1] = chunk_first[b] + static_cast<int32_t>(nch[b]);
    bound = std::max<int>(bound, static_cast<int>(std::min<int64_t>(ntot[b], ceil_div(cost[b], nch[b] * kCostFull) + 1)));
  }
  return bound;
}

// Hand-out order of a launch's units: the sequences by decreasing chunk cost
// (cost / chunks; ties by sequence id), and the prefix sums of their chunk
// counts in that order. The CTAs take units largest first, so their finishing
// times end up within about one small unit of each other.
void plan_unit_order(const std::vector<int64_t>& cost, const int32_t* chunk_first, int32_t* order,
                     int32_t* order_chunk_first) {
  const int B = static_cast<int>(cost.size());
  std::vector<int> idx(B);
  for (int b = 0; b < B; ++b) idx[b] = b;
  auto nch = [&](int b) { return int64_t(chunk_first[b + 1] - chunk_first[b]); };
  std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) { return cost[x] * nch(y) > cost[y] * nch(x); });
  order_chunk_first[0] = 0;
  for (int r = 0; r < B; ++r) {
    order[r] = idx[r];
    order_chunk_first[r + 1] = order_chunk_first[r] + static_cast<int32_t>(nch(idx[r]));
  }
}

// STREAM mode: copy the used T1 / T2 range of layers [l0, l0 + nl) into
// staging slot `slot` on the copy stream (one copy per pool and layer).
// gate_seq != 0: first wait until the attention launch with that sequence
// number has started (its first CTA writes the number to the started word).
// Invariant behind that wait (a stream memory wait has no time limit): gate_seq
// is always the number of an attention launch that was already enqueued on the
// compute stream (h->last_launch_seq), and every enqueued attention launch
// writes its number at entry, so the wait ends once that launch starts.
tkv_status enqueue_prefetch(tkv_ctx* h, int l0, int nl, int slot, uint32_t gate_seq = 0) {
  const Layout& y = h->y;
  if (y.mode != TKV_HOST_TIERS_STREAM) return TKV_OK;
  if (fault_fires(h, TKV_FAULT_PREFETCH)) {
    h->broken = true;  // a decode step stops half done
    return injected(h, "T1/T2 prefetch enqueue");
  }
  const bool timing = h->cfg.flags & TKV_FLAG_TIMING;
  TimedPair tp{};
  if (h->xs != h->cs) CK(h, cudaStreamWaitEvent(h->xs, h->ev_free[slot], 0));
  if (gate_seq != 0 && h->wait_value && h->xs != h->cs) {
    if (gate_seq > h->last_launch_seq)
      return fail(h, TKV_ERR_INTERNAL, "prefetch gated on attention launch %u, which was never enqueued", gate_seq);
    const unsigned long long addr = reinterpret_cast<unsigned long long>(h->D(y.o_err)) + kStartedWordOffset;
    if (h->wait_value(h->xs, addr, gate_seq, kWaitGeq) != 0) h->wait_value = nullptr;  // unsupported: ungated from now on
  }
  if (timing) {
    tkv_status st = timed_pair(h, 1, &tp);
    if (st) return st;
    CK(h, cudaEventRecord(tp.a, h->xs));
  }
  const int64_t n1 = h->next_page[1], n2 = h->next_page[2];
  const bool t2_read = h->cfg.t2_mode == TKV_T2_ATTEND;
  for (int j = 0; j < nl; ++j) {
    const size_t sl = size_t(slot) * y.Lg + j;  // staging layer index
    const int l = l0 + j;
    if (n1 > 0) {
      CK(h, cudaMemcpyAsync(h->D(y.o_stage1) + sl * y.cap[1] * y.plb[1],
                            h->P(y.p_pool1) + size_t(l) * y.cap[1] * y.plb[1], size_t(n1) * y.plb[1],
                            cudaMemcpyHostToDevice, h->xs));
      h->stats.prefetch_bytes += n1 * y.plb[1];
    }
    if (n2 > 0 && t2_read) {
      CK(h, cudaMemcpyAsync(h->D(y.o_stage2c) + sl * y.cap[2] * y.plb[2],
                            h->P(y.p_pool2c) + size_t(l) * y.cap[2] * y.plb[2], size_t(n2) * y.plb[2],
                            cudaMemcpyHostToDevice, h->xs));
      CK(h, cudaMemcpyAsync(h->D(y.o_stage2s) + sl * y.cap[2] * y.scale_rec,
                            h->P(y.p_pool2s) + size_t(l) * y.cap[2] * y.scale_rec,
                            size_t(n2) * y.scale_rec, cudaMemcpyHostToDevice, h->xs));
      h->stats.prefetch_bytes += n2 * (y.plb[2] + y.scale_rec);
    }
  }
  if (timing) {
    CK(h, cudaEventRecord(tp.b, h->xs));
    h->pending.push_back(tp);
  }
  CK(h, cudaEventRecord(h->ev_ready[slot], h->xs));
  return TKV_OK;
}

// Page sources of the launch covering layers from l0: T0 from the HBM pool;
// T1 / T2 from the staging slot (STREAM), the device mirror (MIRROR) or the
// pinned host pools in place (ZEROCOPY).
void fill_sources(tkv_ctx* h, int l0, int slot, AttnParams& p) {
  const Layout& y = h->y;
  const int64_t head_full = int64_t(2) * kPage * y.D * y.esz;
  const int64_t lb0 = y.cap[0] * y.plb[0], lb1 = y.cap[1] * y.plb[1], lb2 = y.cap[2] * y.plb[2];
  const int64_t lbs = y.cap[2] * y.scale_rec;
  const char *b1, *b2, *b2s;
  int host = 0;
  if (y.mode == TKV_HOST_TIERS_STREAM) {
    b1 = h->D(y.o_stage1) + size_t(slot) * y.Lg * lb1;
    b2 = h->D(y.o_stage2c) + size_t(slot) * y.Lg * lb2;
    b2s = h->D(y.o_stage2s) + size_t(slot) * y.Lg * lbs;
  } else if (y.mode == TKV_HOST_TIERS_MIRROR) {
    b1 = h->D(y.o_mirror1) + size_t(l0) * lb1;
    b2 = h->D(y.o_mirror2c) + size_t(l0) * lb2;
    b2s = h->D(y.o_mirror2s) + size_t(l0) * lbs;
  } else {
    b1 = h->PD(y.p_pool1) + size_t(l0) * lb1;
    b2 = h->PD(y.p_pool2c) + size_t(l0) * lb2;
    b2s = h->PD(y.p_pool2s) + size_t(l0) * lbs;
    host = 1;
  }
  p.src[0] = PageSource{h->D(y.o_pool0) + size_t(l0) * lb0, lb0, y.plb[0], head_full, d_table(h, 0), d_mask(h, 0),
                        d_posmap(h, 0), nullptr, 0, 0, 0, SRC_FULL, kSwizzle, 0, cap32(y.cap[0])};
  p.src[1] = PageSource{b1, lb1, y.plb[1], head_full, d_table(h, 1), d_mask(h, 1), d_posmap(h, 1), nullptr, 0, 0, 0,
                        SRC_FULL, kSwizzle, host, cap32(y.cap[1])};
  p.src[2] = PageSource{b2, lb2, y.plb[2], int64_t(2) * kPage * y.D, d_table(h, 2), d_mask(h, 2), d_posmap(h, 2),
                        b2s, lbs, y.scale_rec, h->cfg.t2_scale_gran == TKV_SCALE_PER_TOKEN_HEAD ? 1 : 0, SRC_INT8, 0,
                        host, cap32(y.cap[2])};
  p.nsrc = 3;
}

int64_t attn_bytes_per_layer(tkv_ctx* h) {
  const Layout& y = h->y;
  const int64_t full = int64_t(2) * y.Hkv * y.D * y.esz;
  const int64_t i8 = int64_t(2) * y.Hkv * y.D +
                     (h->cfg.t2_scale_gran == TKV_SCALE_PER_TOKEN ? 8 : int64_t(2) * y.Hkv * 2);
  const bool t2_read = h->cfg.t2_mode == TKV_T2_ATTEND;
  int64_t bytes = 0;
  for (const Seq& sq : h->seqs)
    for (int64_t i = 0; i < sq.N; ++i) {
      const int t = sq.tier[i];
      if (t <= 1) bytes += full;
      else if (t == 2 && t2_read) bytes += i8;
    }
  return bytes;
}

tkv_status do_reclassify(tkv_ctx* h);

tkv_status decode_step_device(tkv_ctx* h, const void* q, const void* k_new, const void* v_new, void* out) {
  const Layout& y = h->y;
  const int B = static_cast<int>(h->seqs.size());
  // ---- capacity checks before any mutation
  int need_pages = 0;
  for (int b = 0; b < B; ++b) {
    const Seq& sq = h->seqs[b];
    if (sq.N + 1 > y.maxtok) return fail(h, TKV_ERR_CAPACITY, "sequence %d is full (%lld tokens)", b, (long long)sq.N);
    if (sq.holes[0].empty()) {
      ++need_pages;
      if (int64_t(sq.pages[0].size()) + 1 > y.maxp) return fail(h, TKV_ERR_CAPACITY, "sequence %d: T0 page list full", b);
    }
  }
  if (h->next_page[0] + need_pages - int64_t(h->free_pages[0].size()) > y.cap[0])
    return fail(h, TKV_ERR_CAPACITY, "T0 pool full");

  // ---- append: every sequence's new token goes to T0 (recent window)
  AppendParams ap{};
  ap.B = B; ap.L = y.L; ap.Hkv = y.Hkv; ap.D = y.D; ap.esz = y.esz;
  ap.k = static_cast<const char*>(k_new); ap.v = static_cast<const char*>(v_new);
  ap.pool0 = h->D(y.o_pool0); ap.layer_bytes = y.cap[0] * y.plb[0]; ap.page_bytes = y.plb[0];
  ap.mask0 = d_mask(h, 0); ap.posmap0 = d_posmap(h, 0); ap.table0 = d_table(h, 0);
  ap.table_stride = static_cast<int32_t>(y.maxp);
  ap.err = reinterpret_cast<int32_t*>(h->D(y.o_err));
  ap.cap0 = cap32(y.cap[0]);
  for (int b = 0; b < B; ++b) {
    Seq& sq = h->seqs[b];
    const int64_t pos = sq.N;
    sq.tier.push_back(0);
    sq.loc.push_back(-1);
    sq.N += 1;
    const size_t np_before = sq.pages[0].size();
    std::vector<int32_t> loc;
    int inserted_at = -1;
    place(h, sq, b, 0, {pos}, &loc, &inserted_at);
    ap.page[b] = loc[0] / kPage;
    ap.slot[b] = loc[0] % kPage;
    ap.new_page[b] = sq.pages[0].size() != np_before;
    ap.insert_at[b] = ap.new_page[b] ? inserted_at : -1;
    ap.np0[b] = static_cast<int32_t>(np_before);
    ap.pos[b] = pos;
  }
  LK(h, launch_append(ap, h->cs), B > 0);

  // ---- per layer group: prefetch T1/T2 (copy stream, STREAM mode), attention + fused scores (compute stream)
  AttnParams p{};
  p.B = B; p.Hq = y.Hq; p.Hkv = y.Hkv; p.D = y.D; p.G = y.G;
  p.table_stride = static_cast<int32_t>(y.maxp);
  const bool t2_read = h->cfg.t2_mode == TKV_T2_ATTEND;
  std::vector<int64_t> ntot(B), cost(B);
  p.page_base[0] = 0;
  for (int b = 0; b < B; ++b) {
    const Seq& sq = h->seqs[b];
    p.npages[0][b] = static_cast<int32_t>(sq.pages[0].size());
    p.npages[1][b] = static_cast<int32_t>(sq.pages[1].size());
    p.npages[2][b] = t2_read ? static_cast<int32_t>(sq.pages[2].size()) : 0;
    ntot[b] = p.npages[0][b] + p.npages[1][b] + p.npages[2][b];
    cost[b] = int64_t(kCostFull) * (p.npages[0][b] + p.npages[1][b]) + int64_t(kCostI8) * p.npages[2][b];
    p.page_base[b + 1] = p.page_base[b] + static_cast<int32_t>(ntot[b]);
  }
  if (p.page_base[B] > y.total_pages) return fail(h, TKV_ERR_INTERNAL, "page lists exceed the pools");
  p.chunk_pages = plan_chunks(ntot, cost, y.Hkv, h->cfg.split_pages, h->resident_ctas, p.chunk_first);
  plan_unit_order(cost, p.chunk_first, p.order, p.order_chunk_first);
  const int total_chunks = p.chunk_first[B];
  if (total_chunks > y.max_chunks) return fail(h, TKV_ERR_INTERNAL, "chunk table overflow");
  p.total_chunks = total_chunks;
  p.q_stride_b = int64_t(y.L) * y.Hq * y.D;
  p.q_stride_l = int64_t(y.Hq) * y.D;
  p.out_stride_b = int64_t(y.L) * y.Hq * y.D;
  p.out_stride_l = int64_t(y.Hq) * y.D;
  p.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(double(y.D)));
  // two buffers of partials and spilled logits, by launch parity
  const size_t part_o_n = size_t(y.Lg) * y.max_chunks * y.Hkv * y.G * y.D;
  const size_t part_mz_n = size_t(y.Lg) * y.max_chunks * y.Hkv * y.G;
  const size_t spill_n = size_t(y.Lg) * y.Hkv * y.spill_stride;
  float* part_o = reinterpret_cast<float*>(h->D(y.o_part_o));
  float* part_m = reinterpret_cast<float*>(h->D(y.o_part_m));
  float* part_z = reinterpret_cast<float*>(h->D(y.o_part_z));
  float* spill = reinterpret_cast<float*>(h->D(y.o_spill));
  p.spill_stride_h = y.spill_stride;
  p.spill_stride_l = int64_t(y.Hkv) * y.spill_stride;
  p.spill_stride_b = 0;
  float* acc = reinterpret_cast<float*>(h->D(y.o_acc));
  p.acc_stride_h = y.total_pages * kPage;
  p.acc_stride_l = int64_t(y.Hkv) * p.acc_stride_h;
  p.acc_stride_b = 0;
  EpCounters* ring = reinterpret_cast<EpCounters*>(h->D(y.o_err) + kEpOffset);
  p.err = reinterpret_cast<int32_t*>(h->D(y.o_err));
  p.wait_limit_ns = h->wait_limit_ns;
  const bool timing = h->cfg.flags & TKV_FLAG_TIMING;
  const int64_t abytes = attn_bytes_per_layer(h);
  const bool stream = y.mode == TKV_HOST_TIERS_STREAM;
  // epilogue bytes per token and KV head (G logits, the accumulator read and
  // write) against its K and V bytes
  const double ep_share = (4.0 * y.G + 8.0) / (2.0 * y.D * y.esz);

  // Each attention launch first finishes the previous launch's layers (their
  // output merge and score epilogue) in its CTAs' tails; the last launch's
  // epilogue is a launch of its own after the loop.
  for (int l0 = 0; l0 < y.L; l0 += y.Lg) {
    const int nl = std::min(y.Lg, y.L - l0);
    int slot = h->slot_rr;
    if (stream && l0 == 0 && h->ahead_valid) {
      slot = h->ahead_slot;  // staged at the end of the previous step
      h->ahead_valid = false;
      if (h->xs != h->cs) CK(h, cudaStreamWaitEvent(h->cs, h->ev_ready[slot], 0));
    } else if (stream) {
      h->slot_rr ^= 1;
      tkv_status st = enqueue_prefetch(h, l0, nl, slot, static_cast<uint32_t>(h->last_launch_seq));
      if (st) return st;
      if (h->xs != h->cs) CK(h, cudaStreamWaitEvent(h->cs, h->ev_ready[slot], 0));
    }
    fill_sources(h, l0, slot, p);
    // consecutive launches alternate parity, across steps too (a step may have an odd launch count)
    const int par = static_cast<int>(h->attn_launch_seq & 1);
    h->attn_launch_seq += 1;
    p.started = reinterpret_cast<uint32_t*>(h->D(y.o_err) + kStartedWordOffset);
    p.launch_seq = static_cast<uint32_t>(h->attn_launch_seq);
    if (timing) {
      unsigned long long* spans = reinterpret_cast<unsigned long long*>(h->D(y.o_span));
      p.span = spans + 2 * (h->attn_launch_seq % kSpanSlots);
      p.span_next = spans + 2 * ((h->attn_launch_seq + 1) % kSpanSlots);
    }
    p.has_prev = l0 > 0;
    {
      // a share of the launch's grid (resident CTAs, at most one per unit)
      const int64_t grid = std::min<int64_t>(h->resident_ctas, int64_t(total_chunks) * y.Hkv * nl);
      p.ep_first_ctas = p.has_prev && kEpFirstDiv > 0 && ep_share >= kEpFirstShare
                            ? static_cast<int32_t>(grid / kEpFirstDiv) : 0;
    }
    p.prev_nlayers = p.nlayers;
    p.nlayers = nl;
    p.prev_first_of_step = p.first_of_step;
    p.first_of_step = l0 == 0;
    // counters rotate over four launches: this one's, the previous one's
    // (leftover items), and the one after next, which this launch zeroes
    p.ep_own = ring + h->attn_launch_seq % 4;
    p.ep_prev = ring + (h->attn_launch_seq + 3) % 4;
    p.ep_clear = ring + (h->attn_launch_seq + 2) % 4;
    p.acc = acc;
    p.prev_part_o = p.part_o;
    p.prev_part_m = p.part_m;
    p.prev_part_z = p.part_z;
    p.prev_spill = p.spill;
    p.prev_out = p.out;
    p.part_o = part_o + par * part_o_n;
    p.part_m = part_m + par * part_mz_n;
    p.part_z = part_z + par * part_mz_n;
    p.spill = spill + par * spill_n;
    p.q = static_cast<const char*>(q) + size_t(l0) * y.Hq * y.D * y.esz;
    p.out = static_cast<char*>(out) + size_t(l0) * y.Hq * y.D * y.esz;
    p.stall_first_page = h->stall_next ? 1 : 0;
    h->stall_next = false;
    TimedPair tp{};
    if (timing) {
      tkv_status st = timed_pair(h, 0, &tp);
      if (st) return st;
      CK(h, cudaEventRecord(tp.a, h->cs));
    }
    LK(h, launch_attention_part(p, h->cfg.kv_dtype, total_chunks, h->cs, 0), total_chunks > 0);
    if (total_chunks > 0) h->last_launch_seq = h->attn_launch_seq;
    if (timing) {
      CK(h, cudaEventRecord(tp.b, h->cs));
      h->pending.push_back(tp);
    }
    if (stream) CK(h, cudaEventRecord(h->ev_free[slot], h->cs));
    h->stats.attn_launches += 1;
    h->stats.attn_layers += nl;
    h->stats.attn_bytes += abytes * nl;
  }
  {
    TimedPair tc{};
    if (timing) {
      if (tkv_status st = timed_pair(h, 2, &tc)) return st;
      CK(h, cudaEventRecord(tc.a, h->cs));
    }
    LK(h, launch_attention_part(p, h->cfg.kv_dtype, total_chunks, h->cs, 1), total_chunks > 0);
    if (timing) {
      CK(h, cudaEventRecord(tc.b, h->cs));
      h->pending.push_back(tc);
    }
  }

  // ---- fold this step's score increments into s (float64)
  FoldParams fp{};
  fp.B = B; fp.Hkv = y.Hkv; fp.nslices = y.Lg;
  fp.max_slots = 0;
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < 3; ++t) fp.npages[t][b] = p.npages[t][b];
    fp.max_slots = std::max<int64_t>(fp.max_slots, ntot[b] * kPage);
  }
  for (int b = 0; b <= B; ++b) fp.page_base[b] = p.page_base[b];
  for (int t = 0; t < 3; ++t) {
    fp.table[t] = d_table(h, t);
    fp.mask[t] = d_mask(h, t);
    fp.posmap[t] = d_posmap(h, t);
  }
  fp.table_stride = static_cast<int32_t>(y.maxp);
  fp.s = reinterpret_cast<double*>(h->D(y.o_s));
  fp.s_stride = y.maxtok;
  fp.acc = acc;
  fp.acc_stride_h = p.acc_stride_h;
  fp.acc_stride_l = p.acc_stride_l;
  fp.inv_lh = 1.0 / (double(y.L) * double(y.Hq));
  fp.err = reinterpret_cast<int32_t*>(h->D(y.o_err));
  for (int t = 0; t < 3; ++t) fp.cap[t] = cap32(y.cap[t]);
  LK(h, launch_fold(fp, h->cs), fp.B > 0 && fp.max_slots > 0);

  h->steps += 1;
  h->stats.steps += 1;
  if (h->pending.size() > 4096) {
    CK(h, cudaStreamSynchronize(h->cs));
    CK(h, cudaStreamSynchronize(h->xs));
    harvest(h);
  }
  if (h->steps % h->cfg.reclassify_interval == 0) return do_reclassify(h);
  // T1 / T2 change only at a reassignment: stage the next step's first layer
  // group now, so the host link stays busy while this step's tail runs and
  // while a caller waits for it (the next step uses the staged slot)
  if (stream && h->xs != h->cs) {
    const int slot = h->slot_rr;
    h->slot_rr ^= 1;
    if (tkv_status st = enqueue_prefetch(h, 0, std::min(y.Lg, y.L), slot, static_cast<uint32_t>(h->last_launch_seq)))
      return st;
    h->ahead_valid = true;
    h->ahead_slot = slot;
  }
  return TKV_OK;
}

tkv_status do_reclassify(tkv_ctx* h) {
  const Layout& y = h->y;
  const int B = static_cast<int>(h->seqs.size());
  h->ahead_valid = false;  // the reassignment may move T1 / T2 pages: restage
  if (B == 0) return fail(h, TKV_ERR_STATE, "no sequence to reclassify");
  // the reassignment reads the scores of every step enqueued so far: drain them
  // first (this also keeps queued decode work out of the reassignment's time)
  if (tkv_status st0 = sync_all(h)) return st0;
  const auto t_start = std::chrono::steady_clock::now();

  // ---- classifier kernel: new tiers on the device
  ClassifyParams cp{};
  cp.B = B;
  cp.s = reinterpret_cast<const double*>(h->D(y.o_s));
  cp.old_tier = h->d_tier;
  cp.new_tier = h->d_tier_new;
  cp.stride = y.maxtok;
  for (int b = 0; b < B; ++b) {
    const Seq& sq = h->seqs[b];
    const int64_t N = sq.N;
    int64_t n0, n1, n2;
    if (h->cfg.budget_mode == TKV_BUDGET_PERCENT) {
      n1 = h->cfg.budget[1] * N / 100;
      n2 = h->cfg.budget[2] * N / 100;
      const int64_t n3 = h->cfg.budget[3] * N / 100;
      n0 = N - n1 - n2 - n3;
    } else {
      n0 = h->cfg.budget[0]; n1 = h->cfg.budget[1]; n2 = h->cfg.budget[2];
    }
    cp.N[b] = N; cp.prompt_len[b] = sq.prompt_len; cp.n0[b] = n0; cp.n1[b] = n1; cp.n2[b] = n2;
  }
  cp.n_sink = h->cfg.n_sink;
  cp.recent_window = h->cfg.recent_window;
  cp.keys = reinterpret_cast<unsigned long long*>(h->D(y.o_keys));
  cp.state = reinterpret_cast<ClassifyState*>(h->D(y.o_cls_state));
  cp.slice_ties = reinterpret_cast<long long*>(h->D(y.o_cls_ties));
  cp.max_slices = classify_slices(y.maxtok);
  // the device tier array must reflect appends since the last reassignment
  {
    char* arena = h->P(y.p_arena);
    for (int b = 0; b < B; ++b) std::memcpy(arena + size_t(b) * y.maxtok, h->seqs[b].tier.data(), h->seqs[b].N);
    int64_t nmax = 0;
    for (const Seq& sq : h->seqs) nmax = std::max(nmax, sq.N);
    CK(h, cudaMemcpy2DAsync(h->d_tier, y.maxtok, arena, y.maxtok, nmax, B, cudaMemcpyHostToDevice, h->cs));
    int nl = 0;
    CK(h, launch_classify(cp, h->cs, &nl));
    h->stats.kernel_launches += nl;
    CK(h, cudaMemcpy2DAsync(arena, y.maxtok, h->d_tier_new, y.maxtok, nmax, B, cudaMemcpyDeviceToHost, h->cs));
    tkv_status st = sync_all(h);
    if (st) return st;
  }
  const auto t_classified = std::chrono::steady_clock::now();
  const uint8_t* new_tiers = reinterpret_cast<const uint8_t*>(h->P(y.p_arena));

  // ---- allocator on a copy of the bookkeeping: a capacity failure changes nothing
  std::vector<Seq> seqs = h->seqs;
  int64_t next_page_save[3] = {h->next_page[0], h->next_page[1], h->next_page[2]};
  MinHeap free_save[3] = {h->free_pages[0], h->free_pages[1], h->free_pages[2]};
  std::vector<uint32_t> mask_save[3];
  std::vector<int32_t> posmap_save[3], table_save[3];
  for (int t = 0; t < 3; ++t) {
    mask_save[t] = h->mask[t];
    posmap_save[t] = h->posmap[t];
    table_save[t] = h->table[t];
  }
  auto restore = [&]() {
    for (int t = 0; t < 3; ++t) {
      h->next_page[t] = next_page_save[t];
      h->free_pages[t] = free_save[t];
      h->mask[t].swap(mask_save[t]);
      h->posmap[t].swap(posmap_save[t]);
      h->table[t].swap(table_save[t]);
    }
  };

  std::vector<Mover> phase1, phase2, compaction;
  int64_t d2h = 0, h2d = 0;
  const bool overflow = fault_fires(h, TKV_FAULT_CLASSIFY_OVERFLOW);
  const int64_t row_full = int64_t(y.L) * 2 * y.Hkv * y.D * y.esz;
  const int64_t row_i8 = int64_t(y.L) * (2 * y.Hkv * y.D + (h->cfg.t2_scale_gran == TKV_SCALE_PER_TOKEN ? 8 : 4 * y.Hkv));
  for (int b = 0; b < B; ++b) {
    Seq& sq = seqs[b];
    const uint8_t* nt = new_tiers + size_t(b) * y.maxtok;
    std::vector<int64_t> moved;
    for (int64_t i = 0; i < sq.N; ++i)
      if (nt[i] != sq.tier[i]) {
        if (sq.tier[i] == 3 || nt[i] > 3) {
          restore();
          return fail(h, TKV_ERR_INTERNAL, "classifier revived an evicted token or wrote tier %d", int(nt[i]));
        }
        moved.push_back(i);
      }
    // source locations before vacating; slots vacated by tokens whose data moves
    std::vector<int32_t> src_loc(moved.size());
    std::vector<uint8_t> src_tier(moved.size());
    std::vector<int64_t> busy;  // tier * 2^40 + loc of slots whose old data still has to be read
    for (size_t m = 0; m < moved.size(); ++m) {
      src_loc[m] = sq.loc[moved[m]];
      src_tier[m] = sq.tier[moved[m]];
      if (nt[moved[m]] != 3) busy.push_back((int64_t(src_tier[m]) << 40) | src_loc[m]);
    }
    std::sort(busy.begin(), busy.end());
    for (int t = 0; t < 3; ++t)
      for (size_t m = 0; m < moved.size(); ++m)
        if (src_tier[m] == t) vacate(h, sq, t, moved[m]);
    std::vector<int32_t> dst_loc(moved.size(), -1);
    for (int t = 0; t < 3; ++t) {
      std::vector<int64_t> arrivals;
      std::vector<size_t> idx;
      for (size_t m = 0; m < moved.size(); ++m)
        if (nt[moved[m]] == t) {
          arrivals.push_back(moved[m]);
          idx.push_back(m);
        }
      std::vector<int32_t> locs;
      // an injected overflow fires at the last placement, after every other sequence's
      // vacates, placements and compaction have touched the bookkeeping
      const bool inject_now = overflow && b == B - 1 && t == 2;
      if (inject_now || !place(h, sq, b, t, arrivals, &locs)) {
        restore();
        return fail(h, TKV_ERR_CAPACITY, "tier %d pool or page list full during reassignment%s", t,
                    inject_now ? " (injected host-side fault)" : "");
      }
      for (size_t a = 0; a < idx.size(); ++a) dst_loc[idx[a]] = locs[a];
    }
    compact_t0(h, sq, b, compaction);
    for (size_t m = 0; m < moved.size(); ++m) {
      const int64_t pos = moved[m];
      const int dt = nt[pos];
      if (dt == 0) dst_loc[m] = sq.loc[pos];  // compaction may have moved a T0 arrival
      if (dt == 3) {
        sq.tier[pos] = 3;
        sq.loc[pos] = -1;
        continue;
      }
      Mover mv{b, src_tier[m], src_loc[m], dt, dst_loc[m], -1};
      const bool recycled = std::binary_search(busy.begin(), busy.end(), (int64_t(dt) << 40) | dst_loc[m]);
      if (recycled) {
        mv.temp_row = static_cast<int32_t>(phase2.size());
        phase2.push_back(mv);
      } else {
        phase1.push_back(mv);
      }
      const bool mirrored = y.mode == TKV_HOST_TIERS_MIRROR;  // T1 / T2 sources read from the device copy
      if (src_tier[m] == 1 && !mirrored) h2d += row_full;
      if (src_tier[m] == 2 && !mirrored) h2d += row_i8;
      if (dt == 1) d2h += row_full;
      if (dt == 2) d2h += row_i8;
    }
  }
  if (int64_t(phase2.size()) > y.temp_rows) {
    restore();
    return fail(h, TKV_ERR_CAPACITY, "%zu movers need staging but max_staged_movers is %lld",
                phase2.size(), (long long)y.temp_rows);
  }

  // ---- commit the bookkeeping, then move the data
  const auto t_allocated = std::chrono::steady_clock::now();
  h->seqs.swap(seqs);
  char* arena = h->P(y.p_arena);
  const size_t moff = align_up(size_t(y.maxb) * y.maxtok);
  Mover* hm = reinterpret_cast<Mover*>(arena + moff);
  std::memcpy(hm, phase2.data(), phase2.size() * sizeof(Mover));
  std::memcpy(hm + phase2.size(), phase1.data(), phase1.size() * sizeof(Mover));
  std::memcpy(hm + phase2.size() + phase1.size(), compaction.data(), compaction.size() * sizeof(Mover));
  const size_t nmov = phase1.size() + phase2.size() + compaction.size();
  Mover* dm = reinterpret_cast<Mover*>(h->D(y.o_movers));
  if (nmov) CK(h, cudaMemcpyAsync(dm, hm, nmov * sizeof(Mover), cudaMemcpyHostToDevice, h->cs));
  MoveParams mp{};
  mp.L = y.L; mp.Hkv = y.Hkv; mp.D = y.D; mp.kv_dtype = h->cfg.kv_dtype;
  mp.pools.base[0] = h->D(y.o_pool0);
  mp.pools.base[1] = h->PD(y.p_pool1);
  mp.pools.base[2] = h->PD(y.p_pool2c);
  for (int t = 0; t < 3; ++t) {
    mp.pools.layer_bytes[t] = y.cap[t] * y.plb[t];
    mp.pools.page_bytes[t] = y.plb[t];
  }
  mp.pools.t2_scales = h->PD(y.p_pool2s);
  mp.pools.t2_scale_layer_bytes = y.cap[2] * y.scale_rec;
  mp.pools.t2_scale_page_bytes = y.scale_rec;
  mp.pools.scale_per_head = h->cfg.t2_scale_gran == TKV_SCALE_PER_TOKEN_HEAD;
  if (y.mode == TKV_HOST_TIERS_MIRROR) {
    mp.pools.mirror[1] = h->D(y.o_mirror1);
    mp.pools.mirror[2] = h->D(y.o_mirror2c);
    mp.pools.mirror_scales = h->D(y.o_mirror2s);
  }
  mp.pools.scale_f16 = h->cfg.t2_scale_dtype == TKV_SCALE_F16;
  for (int t = 0; t < 3; ++t) mp.pools.cap[t] = cap32(y.cap[t]);
  mp.temp = h->D(y.o_temp);
  mp.temp_rows = y.temp_rows;
  mp.err = reinterpret_cast<int32_t*>(h->D(y.o_err));
  // Every source is read before any slot is written that a mover vacated:
  // phase 1 (destinations no mover vacated) reads its sources and writes at
  // once, for all layers; then, layer by layer, phase 2 gathers its sources
  // into the staging rows and scatters them to the recycled slots.
  mp.mode = MOVE_DIRECT;
  mp.layer0 = 0;
  LK(h, launch_move(mp, dm + phase2.size(), int64_t(phase1.size()), y.L, h->cs), !phase1.empty());
  // all layers at once when the staging rows hold them, else one layer per launch pair
  const int per = int64_t(phase2.size()) * y.L <= y.temp_rows ? y.L : 1;
  for (int l = 0; l < y.L && !phase2.empty(); l += per) {
    mp.layer0 = l;
    mp.mode = MOVE_GATHER;
    LK(h, launch_move(mp, dm, int64_t(phase2.size()), per, h->cs), true);
    mp.mode = MOVE_SCATTER;
    LK(h, launch_move(mp, dm, int64_t(phase2.size()), per, h->cs), true);
  }
  // T0 compaction last: every slot it writes has been read by the moves above
  mp.mode = MOVE_DIRECT;
  mp.layer0 = 0;
  LK(h, launch_move(mp, dm + phase2.size() + phase1.size(), int64_t(compaction.size()), y.L, h->cs), !compaction.empty());
  tkv_status st = upload_metadata(h);
  if (st) return st;
  std::swap(h->d_tier, h->d_tier_new);
  st = sync_all(h);
  if (st) return st;

  h->stats.reclassifies += 1;
  h->stats.movers += int64_t(nmov);
  h->stats.d2h_move_bytes += d2h;
  h->stats.h2d_move_bytes += h2d;
  if (h->cfg.flags & TKV_FLAG_TIMING) {
    using ms = std::chrono::duration<double, std::milli>;
    const auto t_end = std::chrono::steady_clock::now();
    h->stats.reclassify_ms += ms(t_end - t_start).count();
    h->stats.classify_ms += ms(t_classified - t_start).count();
    h->stats.allocate_ms += ms(t_allocated - t_classified).count();
    h->stats.move_ms += ms(t_end - t_allocated).count();
  }
  return TKV_OK;
}

tkv_status seq_ok(tkv_ctx* h, int32_t seq) {
  if (seq < 0 || seq >= int32_t(h->seqs.size())) return fail(h, TKV_ERR_INVALID_ARG, "no sequence %d", seq);
  return TKV_OK;
}

}  // namespace

// ============================================================ C ABI
extern "C" {

tkv_status tkv_workspace_size(const tkv_config* cfg, size_t* dev_bytes, size_t* pinned_bytes) {
  if (!cfg || !dev_bytes || !pinned_bytes) return fail(nullptr, TKV_ERR_INVALID_ARG, "null argument");
  const std::string why = validate(*cfg);
  if (!why.empty()) return fail(nullptr, TKV_ERR_INVALID_ARG, "%s", why.c_str());
  const Layout y = make_layout(*cfg);
  *dev_bytes = y.dev_bytes;
  *pinned_bytes = y.pinned_bytes;
  return TKV_OK;
}

tkv_status tkv_create(const tkv_config* cfg, void* dev_ws, size_t dev_bytes, void* pinned_ws,
                      size_t pinned_bytes, tkv_stream compute, tkv_stream copy, tkv_handle* out) {
  if (!cfg || !out) return fail(nullptr, TKV_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const std::string why = validate(*cfg);
  if (!why.empty()) return fail(nullptr, TKV_ERR_INVALID_ARG, "%s", why.c_str());
  const Layout y = make_layout(*cfg);
  if (!dev_ws || !pinned_ws) return fail(nullptr, TKV_ERR_INVALID_ARG, "null workspace");
  if (reinterpret_cast<uintptr_t>(dev_ws) % kAlign || reinterpret_cast<uintptr_t>(pinned_ws) % 64)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "workspace not aligned (device 256 B, pinned 64 B)");
  if (dev_bytes < y.dev_bytes || pinned_bytes < y.pinned_bytes)
    return fail(nullptr, TKV_ERR_CAPACITY, "workspace too small: need %zu device and %zu pinned bytes",
                y.dev_bytes, y.pinned_bytes);
  // fault injection: the set-up call that fails (0: none), and a site the environment arms on the handle
  int32_t setup_fault = g_create_fault.exchange(0);
  int32_t env_site = TKV_FAULT_NONE, env_countdown = 0;
  if (fault_from_env(&env_site, &env_countdown) && env_site == TKV_FAULT_ALLOC && setup_fault == 0)
    setup_fault = env_countdown;
  tkv_ctx* h = new (std::nothrow) tkv_ctx();
  if (!h) return fail(nullptr, TKV_ERR_INTERNAL, "out of host memory");
  h->cfg = *cfg;
  h->y = y;
  h->dev = static_cast<char*>(dev_ws);
  h->pin = static_cast<char*>(pinned_ws);
  h->cs = static_cast<cudaStream_t>(compute);
  h->xs = copy ? static_cast<cudaStream_t>(copy) : h->cs;
  bool enqueued = false;  // clearing of the caller's workspace was enqueued on the compute stream
  auto bail = [&](tkv_status st) {
    if (enqueued) (void)cudaStreamSynchronize(h->cs);  // the workspace goes back to the caller idle
    for (int i = 0; i < 2; ++i) {
      if (h->ev_ready[i]) cudaEventDestroy(h->ev_ready[i]);
      if (h->ev_free[i]) cudaEventDestroy(h->ev_free[i]);
    }
    delete h;
    (void)cudaGetLastError();
    return st;
  };
  // the set-up calls below, counted for fault injection
  auto setup_fails = [&]() { return setup_fault > 0 && --setup_fault == 0; };
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) return bail(fail_cuda(nullptr, "cudaGetDevice", e));
  void* mapped = nullptr;
  if (setup_fails()) return bail(injected(nullptr, "cudaHostGetDevicePointer"));
  e = cudaHostGetDevicePointer(&mapped, pinned_ws, 0);
  if (e != cudaSuccess) return bail(fail_cuda(nullptr, "cudaHostGetDevicePointer (pinned workspace must be page-locked)", e));
  h->pin_dev = static_cast<char*>(mapped);
  for (int i = 0; i < 2; ++i) {
    if (setup_fails()) return bail(injected(nullptr, "cudaEventCreate"));
    if ((e = cudaEventCreateWithFlags(&h->ev_ready[i], cudaEventDisableTiming)) != cudaSuccess)
      return bail(fail_cuda(nullptr, "cudaEventCreate", e));
    if (setup_fails()) return bail(injected(nullptr, "cudaEventCreate"));
    if ((e = cudaEventCreateWithFlags(&h->ev_free[i], cudaEventDisableTiming)) != cudaSuccess)
      return bail(fail_cuda(nullptr, "cudaEventCreate", e));
  }
  h->d_tier = reinterpret_cast<uint8_t*>(h->D(y.o_tier));
  h->d_tier_new = reinterpret_cast<uint8_t*>(h->D(y.o_tier_new));
  h->resident_ctas = resident_attention_ctas(cfg->kv_dtype, y.G, y.D);
  {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      h->wait_value = reinterpret_cast<WaitValue32Fn>(fn);
    (void)cudaGetLastError();
  }
  // zero what must start at zero: pools (holes must hold finite values), tables,
  // masks, accumulators, scores, the error word; posmaps start at -1
  struct Z { size_t off, bytes; int val; } zs[] = {
      {y.o_pool0, size_t(y.L) * y.cap[0] * y.plb[0], 0},
      {y.o_table, 3 * size_t(y.maxb) * y.maxp * 4, 0},
      {y.o_mask, size_t(y.cap[0] + y.cap[1] + y.cap[2]) * 4, 0},
      {y.o_posmap, size_t(y.cap[0] + y.cap[1] + y.cap[2]) * kPage * 4, 0xff},
      {y.o_tier, size_t(y.maxb) * y.maxtok, 0},
      {y.o_s, size_t(y.maxb) * y.maxtok * 8, 0},
      {y.o_acc, size_t(y.Lg) * y.Hkv * y.total_pages * kPage * 4, 0},
      {y.o_err, kErrRegion, 0},
      // device mirrors of the host tiers start as the (zeroed) host pools do
      {y.o_mirror1, y.mode == TKV_HOST_TIERS_MIRROR ? size_t(y.L) * y.cap[1] * y.plb[1] : 0, 0},
      {y.o_mirror2c, y.mode == TKV_HOST_TIERS_MIRROR ? size_t(y.L) * y.cap[2] * y.plb[2] : 0, 0},
      {y.o_mirror2s, y.mode == TKV_HOST_TIERS_MIRROR ? size_t(y.L) * y.cap[2] * y.scale_rec : 0, 0}};
  for (const Z& z : zs) {
    if (!z.bytes) continue;
    if (setup_fails()) return bail(injected(nullptr, "cudaMemsetAsync"));
    enqueued = true;
    if ((e = cudaMemsetAsync(h->D(z.off), z.val, z.bytes, h->cs)) != cudaSuccess)
      return bail(fail_cuda(nullptr, "cudaMemsetAsync", e));
  }
  {
    std::vector<unsigned long long> init(2 * size_t(kSpanSlots), 0ull);
    for (int i = 0; i < kSpanSlots; ++i) init[2 * size_t(i)] = ~0ull;
    if (setup_fails()) return bail(injected(nullptr, "cudaMemcpy"));
    if ((e = cudaMemcpy(h->D(y.o_span), init.data(), init.size() * 8, cudaMemcpyHostToDevice)) != cudaSuccess)
      return bail(fail_cuda(nullptr, "cudaMemcpy", e));
  }
  if (setup_fails()) return bail(injected(nullptr, "cudaStreamSynchronize"));
  if ((e = cudaStreamSynchronize(h->cs)) != cudaSuccess) return bail(fail_cuda(nullptr, "cudaStreamSynchronize", e));
  for (int t = 0; t < 3; ++t) {
    h->mask[t].assign(size_t(y.cap[t]), 0u);
    h->posmap[t].assign(size_t(y.cap[t]) * kPage, -1);
    h->table[t].assign(size_t(y.maxb) * y.maxp, 0);
  }
  if (env_site != TKV_FAULT_NONE && env_site != TKV_FAULT_ALLOC) {
    h->fault_site = env_site;
    h->fault_countdown = env_countdown;
  }
  *out = h;
  return TKV_OK;
}

tkv_status tkv_destroy(tkv_handle h) {
  if (!h) return TKV_OK;
  cudaStreamSynchronize(h->cs);
  if (h->xs != h->cs) cudaStreamSynchronize(h->xs);
  harvest(h);
  for (auto& tp : h->spare) {
    cudaEventDestroy(tp.a);
    cudaEventDestroy(tp.b);
  }
  for (int i = 0; i < 2; ++i) {
    cudaEventDestroy(h->ev_ready[i]);
    cudaEventDestroy(h->ev_free[i]);
  }
  delete h;
  return TKV_OK;
}

tkv_status tkv_append(tkv_handle h, int32_t seq, const void* k, const void* v, int64_t n_tokens,
                      int32_t is_prompt) {
  if (tkv_status st = check_usable(h)) return st;
  const Layout& y = h->y;
  if (!k || !v || n_tokens < 0) return fail(h, TKV_ERR_INVALID_ARG, "bad k/v or n_tokens");
  if (seq < 0 || seq > int32_t(h->seqs.size())) return fail(h, TKV_ERR_INVALID_ARG, "sequence %d does not exist and is not the next one", seq);
  if (seq == int32_t(h->seqs.size()) && seq >= y.maxb) return fail(h, TKV_ERR_CAPACITY, "max_batch sequences already exist");
  if (n_tokens == 0) return TKV_OK;
  const int64_t N0 = seq < int32_t(h->seqs.size()) ? h->seqs[seq].N : 0;
  const int64_t P0 = seq < int32_t(h->seqs.size()) ? h->seqs[seq].prompt_len : 0;
  if (N0 + n_tokens > y.maxtok) return fail(h, TKV_ERR_CAPACITY, "sequence %d would exceed max_tokens", seq);
  if (is_prompt && N0 != P0) return fail(h, TKV_ERR_INVALID_ARG, "prompt tokens must precede generated tokens");
  {
    const int64_t holes = seq < int32_t(h->seqs.size()) ? int64_t(h->seqs[seq].holes[0].size()) : 0;
    const int64_t newp = ceil_div(std::max<int64_t>(0, n_tokens - holes), kPage);
    const int64_t have = seq < int32_t(h->seqs.size()) ? int64_t(h->seqs[seq].pages[0].size()) : 0;
    if (h->next_page[0] + newp > y.cap[0] || have + newp > y.maxp)
      return fail(h, TKV_ERR_CAPACITY, "T0 pool too small for the prefill");
  }
  if (seq == int32_t(h->seqs.size())) h->seqs.emplace_back();
  Seq& sq = h->seqs[seq];
  std::vector<int64_t> pos(static_cast<size_t>(n_tokens));
  for (int64_t i = 0; i < n_tokens; ++i) pos[i] = N0 + i;
  sq.tier.resize(size_t(N0 + n_tokens), 0);
  sq.loc.resize(size_t(N0 + n_tokens), -1);
  sq.N = N0 + n_tokens;
  if (is_prompt) sq.prompt_len += n_tokens;
  std::vector<int32_t> locs;
  if (!place(h, sq, seq, 0, pos, &locs)) return fail(h, TKV_ERR_INTERNAL, "T0 placement failed after the capacity check");
  char* arena = h->P(y.p_arena);
  const size_t loff = y.arena_bytes - align_up(size_t(y.maxtok) * 4);
  std::memcpy(arena + loff, locs.data(), locs.size() * 4);
  int32_t* dl = reinterpret_cast<int32_t*>(h->D(y.o_locs));
  CK(h, cudaMemcpyAsync(dl, arena + loff, locs.size() * 4, cudaMemcpyHostToDevice, h->cs));
  PrefillParams pp{};
  pp.L = y.L; pp.Hkv = y.Hkv; pp.D = y.D; pp.esz = y.esz; pp.n = n_tokens;
  pp.k = static_cast<const char*>(k); pp.v = static_cast<const char*>(v); pp.loc = dl;
  pp.pool0 = h->D(y.o_pool0); pp.layer_bytes = y.cap[0] * y.plb[0]; pp.page_bytes = y.plb[0];
  pp.err = reinterpret_cast<int32_t*>(h->D(y.o_err));
  pp.cap0 = cap32(y.cap[0]);
  LK(h, launch_prefill(pp, h->cs), n_tokens > 0);
  if (tkv_status st = upload_metadata(h)) return st;
  return sync_all(h);
}

tkv_status tkv_decode_step(tkv_handle h, const void* q, const void* k_new, const void* v_new, void* out) {
  if (tkv_status st = check_usable(h)) return st;
  if (!q || !k_new || !v_new || !out) return fail(h, TKV_ERR_INVALID_ARG, "null pointer");
  if (h->seqs.empty()) return fail(h, TKV_ERR_STATE, "no sequence: append a prefill first");
  return decode_step_device(h, q, k_new, v_new, out);
}

tkv_status tkv_decode_step_host(tkv_handle h, const void* q, const void* k_new, const void* v_new, void* out) {
  if (tkv_status st = check_usable(h)) return st;
  if (!q || !k_new || !v_new || !out) return fail(h, TKV_ERR_INVALID_ARG, "null pointer");
  if (h->seqs.empty()) return fail(h, TKV_ERR_STATE, "no sequence: append a prefill first");
  const Layout& y = h->y;
  const int B = static_cast<int>(h->seqs.size());
  const size_t qb = size_t(B) * y.L * y.Hq * y.D * y.esz;
  const size_t kb = size_t(B) * y.L * y.Hkv * y.D * y.esz;
  char* io = h->D(y.o_io);
  char* dq = io + y.io_q;
  char* dk = io + y.io_k;
  char* dv = dk + align_up(size_t(y.maxb) * y.L * y.Hkv * y.D * y.esz);
  char* dout = io + y.io_out;
  // the inputs land in the I/O area, which holds no state: a failed copy changes nothing
  const struct { char* dst; const void* src; size_t n; const char* what; } in[] = {
      {dq, q, qb, "cudaMemcpyAsync (query to device)"},
      {dk, k_new, kb, "cudaMemcpyAsync (new keys to device)"},
      {dv, v_new, kb, "cudaMemcpyAsync (new values to device)"}};
  bool issued = false;
  for (const auto& c : in) {
    tkv_status st = TKV_OK;
    if (fault_fires(h, TKV_FAULT_H2D)) {
      st = injected(h, c.what);
    } else if (cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, h->cs); e != cudaSuccess) {
      (void)cudaGetLastError();
      st = fail(h, TKV_ERR_CUDA, "%s failed: %s", c.what, cudaGetErrorString(e));
    }
    if (st) {
      // earlier copies may still read the caller's buffers: let them land before returning
      if (issued && cudaStreamSynchronize(h->cs) != cudaSuccess) h->broken = true;
      return st;
    }
    issued = true;
  }
  if (tkv_status st = decode_step_device(h, dq, dk, dv, dout)) return st;
  if (fault_fires(h, TKV_FAULT_D2H)) return injected(h, "cudaMemcpyAsync (output to host)");
  CK_SOFT(h, "cudaMemcpyAsync (output to host)", cudaMemcpyAsync(out, dout, qb, cudaMemcpyDeviceToHost, h->cs));
  CK(h, cudaStreamSynchronize(h->cs));
  return TKV_OK;
}

tkv_status tkv_reclassify(tkv_handle h) {
  if (tkv_status st = check_usable(h)) return st;
  return do_reclassify(h);
}

tkv_status tkv_prefetch(tkv_handle h, int32_t layer, int32_t slot) {
  if (tkv_status st = check_usable(h)) return st;
  if (layer < 0 || layer >= h->y.L || slot < 0 || slot > 1) return fail(h, TKV_ERR_INVALID_ARG, "bad layer or slot");
  h->ahead_valid = false;  // the caller may overwrite the staged slot
  return enqueue_prefetch(h, layer, std::min(h->y.Lg, h->y.L - layer), slot);
}

tkv_status tkv_synchronize(tkv_handle h) {
  if (tkv_status st = check_usable(h)) return st;
  return sync_all(h);
}

tkv_status tkv_test_stall_next_attention(tkv_handle h, uint64_t wait_limit_ns) {
  if (tkv_status st = check_usable(h)) return st;
  if (wait_limit_ns < 1000000ull || wait_limit_ns > 2000000000ull)
    return fail(h, TKV_ERR_INVALID_ARG, "wait limit must be 1 ms .. 2 s");
  h->stall_next = true;
  h->wait_limit_ns = wait_limit_ns;
  return TKV_OK;
}

tkv_status tkv_test_inject_fault(tkv_handle h, int32_t site, int32_t countdown) {
  if (site < TKV_FAULT_NONE || site > TKV_FAULT_CLASSIFY_OVERFLOW) return fail(h, TKV_ERR_INVALID_ARG, "unknown fault site %d", site);
  if (site != TKV_FAULT_NONE && countdown < 1) return fail(h, TKV_ERR_INVALID_ARG, "countdown must be >= 1");
  if (site == TKV_FAULT_ALLOC) {
    if (h) return fail(h, TKV_ERR_INVALID_ARG, "the allocation site arms the next tkv_create: pass no handle");
    g_create_fault.store(countdown);
    return TKV_OK;
  }
  if (!h) {
    if (site != TKV_FAULT_NONE) return fail(nullptr, TKV_ERR_INVALID_ARG, "null handle");
    g_create_fault.store(0);
    return TKV_OK;
  }
  h->fault_site = site;
  h->fault_countdown = site == TKV_FAULT_NONE ? 0 : countdown;
  return TKV_OK;
}

int32_t tkv_debug_build(void) { return kDebugBuild ? 1 : 0; }

tkv_status tkv_test_plant_bad_page(tkv_handle h, int32_t seq, int32_t tier, int64_t index, int32_t* planted) {
  if (tkv_status st = check_usable(h)) return st;
  if (!kDebugBuild) return fail(h, TKV_ERR_STATE, "the page-table test hook needs the debug build (TKV_DEBUG)");
  if (tkv_status st = seq_ok(h, seq)) return st;
  if (tier < 0 || tier > 2) return fail(h, TKV_ERR_INVALID_ARG, "tier must be 0, 1 or 2");
  if (index < 0 || index >= int64_t(h->seqs[seq].pages[tier].size()))
    return fail(h, TKV_ERR_INVALID_ARG, "index %lld outside the page list", (long long)index);
  if (!planted) return fail(h, TKV_ERR_INVALID_ARG, "null output");
  if (tkv_status st = sync_all(h)) return st;
  const int32_t id = cap32(h->y.cap[tier]);
  int32_t* at = d_table(h, tier) + size_t(seq) * h->y.maxp + size_t(index);
  CK(h, cudaMemcpy(at, &id, 4, cudaMemcpyHostToDevice));
  *planted = id;
  return TKV_OK;
}

tkv_status tkv_test_plan_attention(int32_t batch, const int64_t* full_pages, const int64_t* i8_pages,
                                   int32_t n_kv_heads, int32_t split_pages, int32_t resident_ctas,
                                   int32_t* chunk_first, int32_t* order, int32_t* order_chunk_first,
                                   int32_t* page_bound) {
  if (batch < 1 || batch > kMaxBatch) return fail(nullptr, TKV_ERR_INVALID_ARG, "batch must be 1..64");
  if (!full_pages || !i8_pages || !chunk_first || !order || !order_chunk_first || !page_bound)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "null pointer");
  if (n_kv_heads < 1 || resident_ctas < 1 || split_pages < 0)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "bad n_kv_heads, resident_ctas or split_pages");
  std::vector<int64_t> ntot(batch), cost(batch);
  for (int b = 0; b < batch; ++b) {
    if (full_pages[b] < 0 || i8_pages[b] < 0 || full_pages[b] + i8_pages[b] > kMaxSeqPages)
      return fail(nullptr, TKV_ERR_INVALID_ARG, "page count of sequence %d outside 0..16384", b);
    ntot[b] = full_pages[b] + i8_pages[b];
    cost[b] = int64_t(kCostFull) * full_pages[b] + int64_t(kCostI8) * i8_pages[b];
  }
  *page_bound = plan_chunks(ntot, cost, n_kv_heads, split_pages, resident_ctas, chunk_first);
  plan_unit_order(cost, chunk_first, order, order_chunk_first);
  return TKV_OK;
}

tkv_status tkv_num_sequences(tkv_handle h, int32_t* n) {
  if (!h || !n) return fail(h, TKV_ERR_INVALID_ARG, "null argument");
  *n = static_cast<int32_t>(h->seqs.size());
  return TKV_OK;
}

tkv_status tkv_seq_len(tkv_handle h, int32_t seq, int64_t* n) {
  if (!h || !n) return fail(h, TKV_ERR_INVALID_ARG, "null argument");
  if (tkv_status st = seq_ok(h, seq)) return st;
  *n = h->seqs[seq].N;
  return TKV_OK;
}

tkv_status tkv_get_scores(tkv_handle h, int32_t seq, double* host_out, int64_t n) {
  if (tkv_status st = check_usable(h)) return st;
  if (tkv_status st = seq_ok(h, seq)) return st;
  if (!host_out || n < 0 || n > h->seqs[seq].N) return fail(h, TKV_ERR_INVALID_ARG, "bad output or n");
  if (tkv_status st = sync_all(h)) return st;
  if (fault_fires(h, TKV_FAULT_D2H)) return injected(h, "cudaMemcpy (scores to host)");
  CK_SOFT(h, "cudaMemcpy (scores to host)",
          cudaMemcpy(host_out, h->D(h->y.o_s) + size_t(seq) * h->y.maxtok * 8, size_t(n) * 8, cudaMemcpyDeviceToHost));
  return TKV_OK;
}

tkv_status tkv_set_scores(tkv_handle h, int32_t seq, const double* host_in, int64_t n) {
  if (tkv_status st = check_usable(h)) return st;
  if (tkv_status st = seq_ok(h, seq)) return st;
  if (!host_in || n < 0 || n > h->seqs[seq].N) return fail(h, TKV_ERR_INVALID_ARG, "bad input or n");
  std::vector<double> s(host_in, host_in + n);
  for (double& x : s) {
    if (std::isnan(x)) return fail(h, TKV_ERR_INVALID_ARG, "NaN score");
    if (x == 0.0) x = 0.0;
  }
  if (tkv_status st = sync_all(h)) return st;
  if (fault_fires(h, TKV_FAULT_H2D)) return injected(h, "cudaMemcpy (scores to device)");
  CK_SOFT(h, "cudaMemcpy (scores to device)",
          cudaMemcpy(h->D(h->y.o_s) + size_t(seq) * h->y.maxtok * 8, s.data(), size_t(n) * 8, cudaMemcpyHostToDevice));
  return TKV_OK;
}

tkv_status tkv_get_tiers(tkv_handle h, int32_t seq, uint8_t* host_out, int64_t n) {
  if (!h) return fail(nullptr, TKV_ERR_INVALID_ARG, "null handle");
  if (tkv_status st = seq_ok(h, seq)) return st;
  if (!host_out || n < 0 || n > h->seqs[seq].N) return fail(h, TKV_ERR_INVALID_ARG, "bad output or n");
  std::memcpy(host_out, h->seqs[seq].tier.data(), size_t(n));
  return TKV_OK;
}

tkv_status tkv_get_page_table(tkv_handle h, int32_t seq, int32_t tier, int32_t* pages, uint16_t* valid_mask,
                              int32_t* positions, int64_t cap, int64_t* n_out) {
  if (!h || !n_out) return fail(h, TKV_ERR_INVALID_ARG, "null argument");
  if (tkv_status st = seq_ok(h, seq)) return st;
  if (tier < 0 || tier > 2) return fail(h, TKV_ERR_INVALID_ARG, "tier must be 0, 1 or 2");
  const std::vector<int32_t>& pl = h->seqs[seq].pages[tier];
  *n_out = int64_t(pl.size());
  const int64_t n = std::min<int64_t>(cap, int64_t(pl.size()));
  for (int64_t i = 0; i < n; ++i) {
    const int32_t pg = pl[i];
    if (pages) pages[i] = pg;
    if (valid_mask) valid_mask[i] = static_cast<uint16_t>(h->mask[tier][pg]);
    if (positions)
      for (int j = 0; j < kPage; ++j) positions[i * kPage + j] = h->posmap[tier][size_t(pg) * kPage + j];
  }
  return TKV_OK;
}

tkv_status tkv_get_t2_row(tkv_handle h, int32_t seq, int64_t pos, int8_t* codes, void* scales) {
  if (tkv_status st = check_usable(h)) return st;
  if (tkv_status st = seq_ok(h, seq)) return st;
  const Seq& sq = h->seqs[seq];
  if (pos < 0 || pos >= sq.N || sq.tier[pos] != 2) return fail(h, TKV_ERR_INVALID_ARG, "position %lld is not in T2", (long long)pos);
  if (!codes || !scales) return fail(h, TKV_ERR_INVALID_ARG, "null output");
  if (tkv_status st = sync_all(h)) return st;
  const Layout& y = h->y;
  const int64_t page = sq.loc[pos] / kPage, slot = sq.loc[pos] % kPage;
  const bool per_head = h->cfg.t2_scale_gran == TKV_SCALE_PER_TOKEN_HEAD;
  for (int l = 0; l < y.L; ++l) {
    const char* pg = h->P(y.p_pool2c) + (size_t(l) * y.cap[2] + page) * y.plb[2];
    const char* sc = h->P(y.p_pool2s) + (size_t(l) * y.cap[2] + page) * y.scale_rec;
    for (int kv = 0; kv < 2; ++kv) {
      for (int hh = 0; hh < y.Hkv; ++hh)
        std::memcpy(codes + ((size_t(l) * 2 + kv) * y.Hkv + hh) * y.D,
                    pg + ((size_t(hh) * 2 + kv) * kPage + slot) * y.D, size_t(y.D));
      if (per_head) {
        for (int hh = 0; hh < y.Hkv; ++hh)
          std::memcpy(static_cast<char*>(scales) + ((size_t(l) * 2 + kv) * y.Hkv + hh) * 2,
                      sc + ((size_t(hh) * 2 + kv) * kPage + slot) * 2, 2);
      } else {
        std::memcpy(static_cast<char*>(scales) + (size_t(l) * 2 + kv) * 4, sc + (size_t(kv) * kPage + slot) * 4, 4);
      }
    }
  }
  return TKV_OK;
}

tkv_status tkv_get_kv_row(tkv_handle h, int32_t seq, int64_t pos, void* k, void* v) {
  if (tkv_status st = check_usable(h)) return st;
  if (tkv_status st = seq_ok(h, seq)) return st;
  const Seq& sq = h->seqs[seq];
  if (pos < 0 || pos >= sq.N || sq.tier[pos] > 1) return fail(h, TKV_ERR_INVALID_ARG, "position %lld is not in T0 or T1", (long long)pos);
  if (!k || !v) return fail(h, TKV_ERR_INVALID_ARG, "null output");
  if (tkv_status st = sync_all(h)) return st;
  const Layout& y = h->y;
  const int t = sq.tier[pos];
  const int64_t page = sq.loc[pos] / kPage, slot = sq.loc[pos] % kPage;
  const size_t rb = size_t(y.D) * y.esz;
  std::vector<char> raw(rb);
  if (t == 0 && fault_fires(h, TKV_FAULT_D2H)) return injected(h, "cudaMemcpy (T0 row to host)");
  for (int l = 0; l < y.L; ++l)
    for (int kv = 0; kv < 2; ++kv)
      for (int hh = 0; hh < y.Hkv; ++hh) {
        char* dst = static_cast<char*>(kv ? v : k) + (size_t(l) * y.Hkv + hh) * rb;
        const size_t off = (size_t(l) * y.cap[t] + page) * y.plb[t] + ((size_t(hh) * 2 + kv) * kPage + slot) * rb;
        if (t == 0)
          CK_SOFT(h, "cudaMemcpy (T0 row to host)", cudaMemcpy(raw.data(), h->D(y.o_pool0) + off, rb, cudaMemcpyDeviceToHost));
        else
          std::memcpy(raw.data(), h->P(y.p_pool1) + off, rb);
        for (size_t c = 0; c < rb / 16; ++c)  // undo the chunk swizzle of the stored row
          std::memcpy(dst + c * 16, raw.data() + swz_offset(int(slot), int64_t(c) * 16, kSwizzle), 16);
      }
  return TKV_OK;
}

tkv_status tkv_get_stats(tkv_handle h, tkv_stats* out) {
  if (!h || !out) return fail(h, TKV_ERR_INVALID_ARG, "null argument");
  if (!h->broken) {
    if (tkv_status st = sync_all(h)) return st;
  }
  for (int t = 0; t < 4; ++t) h->stats.tier_counts[t] = 0;
  for (const Seq& sq : h->seqs)
    for (int64_t i = 0; i < sq.N; ++i) h->stats.tier_counts[sq.tier[i]] += 1;
  h->stats.attn_span_ms = 0.0;
  if ((h->cfg.flags & TKV_FLAG_TIMING) && !h->broken && h->attn_launch_seq > h->span_from) {
    std::vector<unsigned long long> sp(2 * size_t(kSpanSlots));
    CK(h, cudaMemcpy(sp.data(), h->D(h->y.o_span), sp.size() * 8, cudaMemcpyDeviceToHost));
    const int64_t lo = std::max<int64_t>(h->span_from, h->attn_launch_seq - kSpanSlots);
    for (int64_t q = lo + 1; q <= h->attn_launch_seq; ++q) {  // launch q used slot q % kSpanSlots
      const size_t i = 2 * size_t(q % kSpanSlots);
      if (sp[i + 1] > sp[i]) h->stats.attn_span_ms += double(sp[i + 1] - sp[i]) * 1e-6;
    }
  }
  *out = h->stats;
  return TKV_OK;
}

tkv_status tkv_reset_stats(tkv_handle h) {
  if (!h) return fail(nullptr, TKV_ERR_INVALID_ARG, "null handle");
  if (!h->broken) {
    if (tkv_status st = sync_all(h)) return st;
  }
  h->stats = tkv_stats{};
  h->span_from = h->attn_launch_seq;
  return TKV_OK;
}

const char* tkv_last_error(tkv_handle h) {
  if (h) return h->err.c_str();
  return g_last_error.c_str();
}

// ------------------------------------------------------------ stateless kernels
namespace {
struct PagedScratch {
  size_t o_err, o_part_o, o_part_m, o_part_z, o_spill, bytes;
  int64_t max_chunks, spill_stride;
};
PagedScratch paged_scratch(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t max_pages) {
  PagedScratch s{};
  const int G = Hq / Hkv;
  s.max_chunks = int64_t(B) * (ceil_div(max_pages, 8) + 1);
  s.spill_stride = int64_t(max_pages) * G * kPage;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  s.o_err = take(kErrRegion);   // error word, then the launch's epilogue counters
  s.o_part_o = take(size_t(s.max_chunks) * Hkv * G * D * 4);
  s.o_part_m = take(size_t(s.max_chunks) * Hkv * G * 4);
  s.o_part_z = take(size_t(s.max_chunks) * Hkv * G * 4);
  s.o_spill = take(size_t(B) * Hkv * s.spill_stride * 4);
  s.bytes = o;
  return s;
}
}  // namespace

tkv_status tkv_paged_attention_scratch_size(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                                            int32_t head_dim, int32_t max_pages, size_t* scratch_bytes) {
  if (!scratch_bytes || batch < 1 || batch > kMaxBatch || n_kv_heads < 1 || n_q_heads % n_kv_heads ||
      max_pages < 1)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "bad paged-attention shape");
  *scratch_bytes = paged_scratch(batch, n_q_heads, n_kv_heads, head_dim, max_pages).bytes;
  return TKV_OK;
}

tkv_status tkv_paged_attention(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                               int32_t kv_dtype, const void* q, const void* pool, const int32_t* page_table,
                               const uint32_t* slot_mask, const int32_t* page_counts, int32_t max_pages,
                               void* out, float* alpha_sum, void* scratch, size_t scratch_bytes,
                               tkv_stream stream) {
  if (batch < 1 || batch > kMaxBatch || n_kv_heads < 1 || n_q_heads % n_kv_heads || max_pages < 1)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "bad paged-attention shape");
  if (kv_dtype != TKV_DTYPE_F32 && kv_dtype != TKV_DTYPE_BF16) return fail(nullptr, TKV_ERR_INVALID_ARG, "kv_dtype");
  const int G = n_q_heads / n_kv_heads;
  if (!attention_supported(kv_dtype, G, head_dim)) return fail(nullptr, TKV_ERR_INVALID_ARG, "unsupported group size or head_dim");
  if (!q || !pool || !page_table || !slot_mask || !page_counts || !out || !scratch)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "null pointer");
  const PagedScratch s = paged_scratch(batch, n_q_heads, n_kv_heads, head_dim, max_pages);
  if (scratch_bytes < s.bytes) return fail(nullptr, TKV_ERR_CAPACITY, "scratch too small: need %zu bytes", s.bytes);
  if (reinterpret_cast<uintptr_t>(scratch) % kAlign) return fail(nullptr, TKV_ERR_INVALID_ARG, "scratch not 256-byte aligned");
  if (reinterpret_cast<uintptr_t>(alpha_sum) % 16) return fail(nullptr, TKV_ERR_INVALID_ARG, "alpha_sum not 16-byte aligned");
  const int esz = kv_dtype == TKV_DTYPE_BF16 ? 2 : 4;
  AttnParams p{};
  p.B = batch; p.Hq = n_q_heads; p.Hkv = n_kv_heads; p.D = head_dim; p.G = G;
  p.table_stride = max_pages;
  std::vector<int64_t> ntot(batch), cost(batch);
  if (max_pages > kMaxSeqPages) return fail(nullptr, TKV_ERR_INVALID_ARG, "max_pages above 16384");
  for (int b = 0; b < batch; ++b) {
    if (page_counts[b] < 1 || page_counts[b] > max_pages) return fail(nullptr, TKV_ERR_INVALID_ARG, "page_counts[%d] out of 1..max_pages", b);
    p.npages[0][b] = page_counts[b];
    ntot[b] = page_counts[b];
    cost[b] = int64_t(kCostFull) * page_counts[b];
  }
  p.chunk_pages = plan_chunks(ntot, cost, n_kv_heads, 0, resident_attention_ctas(kv_dtype, G, head_dim), p.chunk_first);
  plan_unit_order(cost, p.chunk_first, p.order, p.order_chunk_first);
  if (p.chunk_first[batch] > s.max_chunks) return fail(nullptr, TKV_ERR_INTERNAL, "chunk plan exceeds the scratch");
  const int64_t head_full = int64_t(2) * kPage * head_dim * esz;
  // the caller's pool size is not passed in: its page ids are the caller's to keep in range
  p.src[0] = PageSource{static_cast<const char*>(pool), 0, head_full * n_kv_heads, head_full, page_table, slot_mask,
                        nullptr, nullptr, 0, 0, 0, SRC_FULL, 0, 0, INT32_MAX};
  p.nsrc = 1;
  p.total_chunks = p.chunk_first[batch];
  p.nlayers = 1;
  for (int b = 0; b <= batch; ++b) p.page_base[b] = 0;
  p.q = q; p.q_stride_b = int64_t(n_q_heads) * head_dim;
  p.out = out; p.out_stride_b = int64_t(n_q_heads) * head_dim;
  p.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(double(head_dim)));
  char* sc = static_cast<char*>(scratch);
  p.part_o = reinterpret_cast<float*>(sc + s.o_part_o);
  p.part_m = reinterpret_cast<float*>(sc + s.o_part_m);
  p.part_z = reinterpret_cast<float*>(sc + s.o_part_z);
  p.spill = reinterpret_cast<float*>(sc + s.o_spill);
  p.spill_stride_h = s.spill_stride;
  p.spill_stride_b = int64_t(n_kv_heads) * s.spill_stride;
  p.acc = alpha_sum;
  p.acc_stride_b = int64_t(n_kv_heads) * max_pages * kPage;
  p.acc_stride_h = int64_t(max_pages) * kPage;
  p.err = reinterpret_cast<int32_t*>(sc + s.o_err);
  p.ep_own = reinterpret_cast<EpCounters*>(sc + s.o_err + kEpOffset);
  p.wait_limit_ns = 2000000000ull;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(sc + s.o_err, 0, kErrRegion, st);
  if (e != cudaSuccess) return fail_cuda(nullptr, "cudaMemsetAsync", e);
  e = launch_attention(p, kv_dtype, p.chunk_first[batch], st);
  if (e != cudaSuccess) return fail_cuda(nullptr, "attention launch", e);
  return TKV_OK;
}

// ------------------------------------------------------------ allocation-free form
// For callers that cannot allocate device memory: the scratch of the paged
// attention lives in a fixed array of this file, set up once per device.
}  // extern "C"
namespace {
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device
__device__ __align__(256) char g_static_scratch[kStaticScratchBytes];
constexpr int kMaxDevices = 256;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};
}  // namespace
extern "C" {

tkv_status tkv_paged_attention_noalloc(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                       int32_t kv_dtype, const void* q, const void* pool,
                                       const int32_t* page_table, const uint32_t* slot_mask,
                                       const int32_t* page_counts, int32_t max_pages, void* out,
                                       float* alpha_sum, tkv_stream stream) {
  if (batch < 1 || batch > kMaxBatch || n_kv_heads < 1 || n_q_heads % n_kv_heads || max_pages < 1)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "bad paged-attention shape");
  // the checks tkv_paged_attention makes on the shape come first, so that an
  // unsupported shape is not reported as one that needs a caller buffer
  if (kv_dtype != TKV_DTYPE_F32 && kv_dtype != TKV_DTYPE_BF16) return fail(nullptr, TKV_ERR_INVALID_ARG, "kv_dtype");
  if (!attention_supported(kv_dtype, n_q_heads / n_kv_heads, head_dim))
    return fail(nullptr, TKV_ERR_INVALID_ARG, "unsupported group size or head_dim");
  const size_t need = paged_scratch(batch, n_q_heads, n_kv_heads, head_dim, max_pages).bytes;
  if (need > kStaticScratchBytes)
    return fail(nullptr, TKV_ERR_CAPACITY,
                "this shape needs %zu bytes of scratch; the allocation-free form has %zu: use "
                "tkv_paged_attention with a caller buffer", need, kStaticScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(nullptr, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return fail(nullptr, TKV_ERR_INVALID_ARG, "device index out of range");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      // once per device, with that device current: the array's device address
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_static_scratch);
      if (e != cudaSuccess) return fail_cuda(nullptr, "cudaGetSymbolAddress(static scratch)", e);
      g_static_addr[dev] = ptr;
    }
    scratch = g_static_addr[dev];
  }
  return tkv_paged_attention(batch, n_q_heads, n_kv_heads, head_dim, kv_dtype, q, pool, page_table, slot_mask,
                             page_counts, max_pages, out, alpha_sum, scratch, kStaticScratchBytes, stream);
}

tkv_status tkv_paged_attention_noalloc_status(int32_t* host_out, tkv_stream stream) {
  if (!host_out) return fail(nullptr, TKV_ERR_INVALID_ARG, "null output");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(nullptr, "cudaGetDevice", e);
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (dev < 0 || dev >= kMaxDevices || !g_static_addr[dev])
      return fail(nullptr, TKV_ERR_STATE, "no allocation-free call has run on this device");
  }
  // the status word is the first int32 of the array (offset 0 of the scratch layout)
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaMemcpyFromSymbolAsync(host_out, g_static_scratch, sizeof(int32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return fail_cuda(nullptr, "cudaMemcpyFromSymbolAsync", e);
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_cuda(nullptr, "cudaStreamSynchronize", e);
  return TKV_OK;
}

namespace {
// scratch of the stateless classifier: keys [B][stride], state [B], slice tie counts [B][slices][3]
struct ClassifyScratch {
  size_t o_keys, o_state, o_ties, bytes;
  int64_t slices;
};
ClassifyScratch classify_scratch(int32_t batch, int64_t stride) {
  ClassifyScratch c{};
  c.slices = classify_slices(stride);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  c.o_keys = take(size_t(batch) * stride * 8);
  c.o_state = take(size_t(batch) * sizeof(ClassifyState));
  c.o_ties = take(size_t(batch) * c.slices * 3 * 8);
  c.bytes = o;
  return c;
}
}  // namespace

tkv_status tkv_classify_scratch_size(int32_t batch, int64_t stride, size_t* scratch_bytes) {
  if (!scratch_bytes || batch < 1 || batch > kMaxBatch || stride < 1) return fail(nullptr, TKV_ERR_INVALID_ARG, "bad shape");
  *scratch_bytes = classify_scratch(batch, stride).bytes;
  return TKV_OK;
}

tkv_status tkv_classify(int32_t batch, const double* scores, const uint8_t* old_tier, uint8_t* new_tier,
                        int64_t stride, const int64_t* params, int32_t n_sink, int32_t recent_window,
                        void* scratch, size_t scratch_bytes, tkv_stream stream) {
  if (batch < 1 || batch > kMaxBatch || stride < 1 || !scores || !old_tier || !new_tier || !params || !scratch)
    return fail(nullptr, TKV_ERR_INVALID_ARG, "bad classify arguments");
  const ClassifyScratch cs = classify_scratch(batch, stride);
  if (scratch_bytes < cs.bytes) return fail(nullptr, TKV_ERR_CAPACITY, "scratch too small: need %zu bytes", cs.bytes);
  if (reinterpret_cast<uintptr_t>(scratch) % kAlign) return fail(nullptr, TKV_ERR_INVALID_ARG, "scratch not 256-byte aligned");
  if (n_sink < 0 || recent_window < 0) return fail(nullptr, TKV_ERR_INVALID_ARG, "negative protection");
  ClassifyParams cp{};
  cp.B = batch;
  cp.s = scores; cp.old_tier = old_tier; cp.new_tier = new_tier; cp.stride = stride;
  for (int b = 0; b < batch; ++b) {
    const int64_t* r = params + 5 * b;
    if (r[0] < 0 || r[0] > stride || r[1] < 0 || r[2] < 0 || r[3] < 0 || r[4] < 0)
      return fail(nullptr, TKV_ERR_INVALID_ARG, "bad params for sequence %d", b);
    cp.N[b] = r[0]; cp.prompt_len[b] = r[1]; cp.n0[b] = r[2]; cp.n1[b] = r[3]; cp.n2[b] = r[4];
  }
  cp.n_sink = n_sink; cp.recent_window = recent_window;
  char* sc = static_cast<char*>(scratch);
  cp.keys = reinterpret_cast<unsigned long long*>(sc + cs.o_keys);
  cp.state = reinterpret_cast<ClassifyState*>(sc + cs.o_state);
  cp.slice_ties = reinterpret_cast<long long*>(sc + cs.o_ties);
  cp.max_slices = cs.slices;
  int nl = 0;
  cudaError_t e = launch_classify(cp, static_cast<cudaStream_t>(stream), &nl);
  if (e != cudaSuccess) return fail_cuda(nullptr, "classify launch", e);
  return TKV_OK;
}

tkv_status tkv_quantize_rows(const void* x, int32_t kv_dtype, int64_t rows, int32_t row_len, int8_t* codes,
                             void* scales, int32_t scale_dtype, tkv_stream stream) {
  if (!x || !codes || !scales || rows < 0 || row_len < 1) return fail(nullptr, TKV_ERR_INVALID_ARG, "bad quantize arguments");
  if (kv_dtype != TKV_DTYPE_F32 && kv_dtype != TKV_DTYPE_BF16) return fail(nullptr, TKV_ERR_INVALID_ARG, "kv_dtype");
  if (scale_dtype != TKV_SCALE_F32 && scale_dtype != TKV_SCALE_F16) return fail(nullptr, TKV_ERR_INVALID_ARG, "scale_dtype");
  cudaError_t e = launch_quantize_rows(x, kv_dtype, rows, row_len, codes, scales, scale_dtype == TKV_SCALE_F16,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(nullptr, "quantize launch", e);
  return TKV_OK;
}

}  // extern "C"
