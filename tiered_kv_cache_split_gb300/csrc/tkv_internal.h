// Internal declarations shared by the translation units of libtkv.so.
// Not part of the public interface (include/tkv.h is).
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace tkv {

constexpr int kPage = 16;          // tokens per page
constexpr int kMaxBatch = 64;      // sequences per handle (kernel parameters carry per-sequence arrays)
#ifndef TKV_ATTN_WARPS
#define TKV_ATTN_WARPS 4
#endif
#ifndef TKV_ATTN_STAGES
#define TKV_ATTN_STAGES 8
#endif
constexpr int kAttnWarps = TKV_ATTN_WARPS;    // consumer warps per attention CTA (+ 1 producer warp)
constexpr int kAttnStages = TKV_ATTN_STAGES;  // shared-memory ring of page stages per CTA
// Page i goes to ring stage i % stages and to consumer warp i % warps. With the
// stage count a multiple of the warp count every stage has a single consumer,
// so each warp waits on a stage's mbarrier phases one after another; otherwise
// a warp would skip phases and a parity wait could match a stale phase.
static_assert(kAttnStages % kAttnWarps == 0, "ring stages must be a multiple of consumer warps");
constexpr int kMaxChunkPages = 256;    // pages one attention CTA may take
constexpr int kMaxChunksPerSeq = 128;  // chunks one sequence may be split into
constexpr int kMaxSeqPages = 16384;    // pages of one sequence (all tiers)
constexpr int kSpanSlots = 4096;       // attention launches whose device span is kept

// Chunks of a sequence's page list (T0, T1, then T2 pages) are balanced by
// cost, in half-page units per page: a T2 page carries half the bytes of a
// full-precision page but is widened in shared memory first, and measured
// about 1.5 times as long to process.
constexpr int kCostFull = 2, kCostI8 = 3;
// Page index at cost c of a list of n01 full-precision pages followed by 8-bit ones.
__host__ __device__ inline int page_at_cost(int64_t c, int n01) {
  const int64_t full = static_cast<int64_t>(kCostFull) * n01;
  if (c <= full) return static_cast<int>(c / kCostFull);
  return n01 + static_cast<int>((c - full) / kCostI8);
}
// A chunk of cost at most this holds at most kMaxChunkPages pages.
constexpr int64_t kMaxChunkCost = static_cast<int64_t>(kCostFull) * (kMaxChunkPages - 1);

// Device-side error codes written into the handle's error word.
enum DevError : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_INDEX = 2 };

// Index checks of the debug build (compiled with -DTKV_DEBUG; release builds
// compile them away). A failing check stores DEV_BAD_INDEX in the error word,
// then the site, the index and its bound after it (the first failure wins),
// and the access it guards is skipped; the next synchronising call reports
// TKV_ERR_INTERNAL with those details. No check traps.
enum DebugSite : int {
  DBG_NONE = 0,
  DBG_ATTN_LIST = 1,   // attention: page-list index against the table row
  DBG_ATTN_PAGE = 2,   // attention: page id against its pool
  DBG_FOLD_PAGE = 3,   // score fold: page id against its pool
  DBG_FOLD_POS = 4,    // score fold: position held by a slot against the score row
  DBG_APPEND_PAGE = 5, // append: page id of the new token against the T0 pool
  DBG_APPEND_LIST = 6, // append: T0 page list length against the table row
  DBG_PREFILL_PAGE = 7,// prefill: page id against the T0 pool
  DBG_MOVE_SRC = 8,    // mover: source page id against its pool
  DBG_MOVE_DST = 9,    // mover: destination page id against its pool
  DBG_MOVE_TEMP = 10   // mover: staging row against the staging area
};
constexpr int kDebugSites = 11;
// error word layout: int32 [0] code, [1] site; int64 [1] index, [2] bound

#ifdef TKV_DEBUG
constexpr bool kDebugBuild = true;
__device__ __forceinline__ bool index_ok(int32_t* err, int site, int64_t i, int64_t bound) {
  if (i >= 0 && i < bound) return true;
  if (err && atomicCAS(err, 0, DEV_BAD_INDEX) == 0) {
    err[1] = site;
    reinterpret_cast<long long*>(err)[1] = static_cast<long long>(i);
    reinterpret_cast<long long*>(err)[2] = static_cast<long long>(bound);
  }
  return false;
}
#else
constexpr bool kDebugBuild = false;
__device__ __forceinline__ bool index_ok(int32_t*, int, int64_t, int64_t) { return true; }
#endif

enum SrcKind : int { SRC_FULL = 0, SRC_INT8 = 1 };

// Full-precision K and V blocks of a page (16 rows of head_dim elements) are
// stored swizzled: the 16-byte chunk c of row r sits at chunk c ^ (r & 7) of
// that row, so that 8 consecutive rows of one column chunk fall in 8 distinct
// shared-memory bank groups once a block is copied to shared memory verbatim.
// 8-bit T2 blocks are stored unswizzled.
constexpr int kSwizzle = 7;
__host__ __device__ inline int64_t swz_offset(int row, int64_t byte_in_row, int swz) {
  return (((byte_in_row >> 4) ^ (row & swz)) << 4) | (byte_in_row & 15);
}

// Work counters of one attention launch: claim[z] hands out the epilogue
// items of its layer z, and units hands out the launch's work units after each
// CTA's first (fetch-and-add; values past the count mean none is left). Four
// sets rotate over consecutive launches.
constexpr int kMaxLaunchLayers = 32;
struct EpCounters {
  int32_t claim[kMaxLaunchLayers];
  int32_t units;
};

// One page source of the attention kernel: a page pool (or one layer of it).
struct PageSource {
  const char* base;          // page 0 of this source at the launch's first layer
  int64_t layer_bytes;       // bytes from one layer of the source to the next
  int64_t page_bytes;        // bytes per page record (all KV heads)
  int64_t head_bytes;        // bytes per KV head in a page record (its K block then V block)
  const int32_t* table;      // [B][table_stride] page ids in page order
  const uint32_t* mask;      // [pages] valid-slot bits
  const int32_t* posmap;     // [pages][16] position held by each slot (-1 hole); may be null
  const char* scales;        // int8 sources: scale records of page 0 at the launch's first layer
  int64_t scale_layer_bytes; // bytes from one layer of the scale records to the next
  int64_t scale_page_bytes;  // bytes per page of scale records
  int32_t scale_per_head;    // 0: [2][16] float32 per page; 1: [Hkv][2][16] float16
  int32_t kind;              // SrcKind
  int32_t swz;               // full-precision blocks: kSwizzle (library pools) or 0 (plain)
  int32_t host;              // 1: pages sit in pinned host memory (device-mapped) and are read
                             // in place with plain loads, never with bulk copies
  int32_t pages;             // pool capacity in pages (debug index checks; INT32_MAX: unknown)
};

// One attention launch covers `nlayers` consecutive layers (gridDim.z) of the
// same chunk plan. Work unit (layer z, chunk c, KV head h) has index
// (z * total_chunks + c) * Hkv + h in the partial buffers; its logits and
// score increments sit at (page_base[b] + k) * 16 + row of its (z, b, h)
// region (k = page index in the sequence's list).
struct AttnParams {
  int32_t B, Hq, Hkv, D, G;
  int32_t nsrc;
  PageSource src[3];
  int32_t table_stride;
  int32_t npages[3][kMaxBatch];
  int32_t chunk_first[kMaxBatch + 1];   // prefix sums of chunks per sequence
  // Order in which the launch's units are handed out: the sequences by
  // decreasing chunk cost (order[r] = sequence of rank r), and prefix sums of
  // their chunk counts in that order. Largest units first keeps the CTAs'
  // finishing times close.
  int32_t order[kMaxBatch];
  int32_t order_chunk_first[kMaxBatch + 1];
  int32_t page_base[kMaxBatch + 1];     // spill / score slot base of each sequence, in pages
  int32_t chunk_pages;                  // upper bound of pages per chunk
  int32_t total_chunks;                 // chunk_first[B]
  int32_t nlayers;                      // layers in this launch
  const void* q;          // element (z, b, h, e) at q[z * q_stride_l + b * q_stride_b + h * D + e]
  int64_t q_stride_b, q_stride_l;
  void* out;
  int64_t out_stride_b, out_stride_l;
  float qscale;           // log2(e) / sqrt(D): logits are kept in base 2
  float* part_o;          // [unit][G][D]
  float* part_m;          // [unit][G]
  float* part_z;          // [unit][G]
  float* spill;           // logits of (z, b, h): spill + z * spill_stride_l + b * spill_stride_b
  int64_t spill_stride_l, spill_stride_b, spill_stride_h;   //  + h * spill_stride_h + (page_base[b] + k) * G * 16
  float* acc;             // score increments of (z, b, h): acc + z * acc_stride_l + b * acc_stride_b
  int64_t acc_stride_l, acc_stride_b, acc_stride_h;         //  + h * acc_stride_h + (page_base[b] + k) * 16 (may be null)
  int32_t* err;
  unsigned long long wait_limit_ns;     // bounded waits give up after this long
  int32_t stall_first_page;             // test hook: the CTA running unit 0 never issues its first page's copy
  // The previous launch of the same step (same chunk plan), whose output merge
  // and score epilogue each CTA of this launch runs after its own pages
  // (has_prev != 0); it covered prev_nlayers layers.
  int32_t has_prev;
  int32_t prev_nlayers;
  // CTAs blockIdx.x < ep_first_ctas take the previous launch's epilogue items
  // before their first unit, overlapping them with the others' page streams;
  // every CTA takes items left over once the units run out
  int32_t ep_first_ctas;
  // The first launch of a step covers layers 0 .. Lg-1, so its epilogue items
  // are the first to touch every accumulator slot of the step: they write
  // instead of adding (and the fold does not clear). 0 for a stateless call.
  int32_t first_of_step;
  int32_t prev_first_of_step;
  EpCounters* ep_own;     // this launch's counters (zero at launch; claimed by the next launch or the combine)
  EpCounters* ep_prev;    // the previous launch's counters (its epilogue items)
  EpCounters* ep_clear;   // counters of the launch after next, zeroed by this launch (or null)
  uint32_t* started;      // if set, the first CTA writes launch_seq here at entry
  uint32_t launch_seq;
  // if set: span[0] = min CTA start, span[1] = max CTA end (%globaltimer ns) of
  // this launch; span_next (the next launch's pair) is reset to (max, 0)
  unsigned long long* span;
  unsigned long long* span_next;
  const float* prev_part_o;
  const float* prev_part_m;
  const float* prev_part_z;
  const float* prev_spill;
  void* prev_out;
};

// attention.cu
cudaError_t launch_attention(const AttnParams& p, int kv_dtype, int total_chunks, cudaStream_t s);
// part 0: the page-streaming attention kernel; part 1: the combine / score kernel
cudaError_t launch_attention_part(const AttnParams& p, int kv_dtype, int total_chunks, cudaStream_t s, int part);
int attention_supported(int kv_dtype, int G, int D);
// attention CTAs that fit on the current device at once (SMs x CTAs per SM)
int resident_attention_ctas(int kv_dtype, int G, int D);

// classify.cu
// Per-sequence state of the radix select (device scratch, zeroed per call).
struct ClassifyState {
  unsigned long long ncand, nprot;      // candidates and protected positions
  unsigned long long prefix[3];         // boundary keys, narrowed 8 bits per pass
  long long rem[3];                     // rank of each boundary among keys with its prefix
  int done[3];                          // boundary past the last candidate
  unsigned int hist[3][256];            // digit histograms of the current pass
};

struct ClassifyParams {
  int32_t B;
  const double* s;
  const uint8_t* old_tier;
  uint8_t* new_tier;
  int64_t stride;
  int64_t N[kMaxBatch], prompt_len[kMaxBatch], n0[kMaxBatch], n1[kMaxBatch], n2[kMaxBatch];
  int32_t n_sink, recent_window;
  unsigned long long* keys;  // scratch [B][stride]
  ClassifyState* state;      // scratch [B]
  long long* slice_ties;     // scratch [B][max_slices][3]
  int64_t max_slices;        // slices of 4096 positions per sequence the scratch holds
};
// slices of 4096 positions needed for sequences of up to `stride` positions
int64_t classify_slices(int64_t stride);
// launches the select's kernels (their count in *launches)
cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t s, int* launches);

// movement.cu
struct AppendParams {
  int32_t B, L, Hkv, D, esz;
  const char* k;           // [B][L][Hkv][D]
  const char* v;
  char* pool0;             // T0 pool, layer-major [L][pages][Hkv][2][16][D]
  int64_t layer_bytes;     // bytes of one layer of the T0 pool
  int64_t page_bytes;      // bytes of one page record
  uint32_t* mask0;
  int32_t* posmap0;
  int32_t* table0;
  int32_t table_stride;
  int32_t page[kMaxBatch], slot[kMaxBatch], np0[kMaxBatch], new_page[kMaxBatch];
  int32_t insert_at[kMaxBatch];  // list index the new page takes (-1: none); later entries shift right
  int64_t pos[kMaxBatch];
  int32_t* err;            // error word (debug index checks)
  int32_t cap0;            // T0 pool capacity in pages
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);

struct PrefillParams {
  int32_t L, Hkv, D, esz;
  int64_t n;               // tokens
  const char* k;           // [L][n][Hkv][D]
  const char* v;
  const int32_t* loc;      // [n] page * 16 + slot
  char* pool0;
  int64_t layer_bytes, page_bytes;
  int32_t* err;            // error word (debug index checks)
  int32_t cap0;            // T0 pool capacity in pages
};
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t s);

// A token whose tier changes; loc = page * 16 + slot in that tier's pool.
struct Mover {
  int32_t b, src_tier, src_loc, dst_tier, dst_loc, temp_row;
};

struct TierPools {
  char* base[3];           // layer-major page pools (T1, T2 in host memory, device-mapped)
  char* mirror[3];         // device-resident copies of the T1 / T2 pools (same layout) or null:
                           // tokens entering T1 / T2 are written to both, sources are read from the copy
  char* mirror_scales;
  int64_t layer_bytes[3];
  int64_t page_bytes[3];   // page record bytes (T2: int8 codes)
  char* t2_scales;         // layer-major scale records
  int64_t t2_scale_layer_bytes, t2_scale_page_bytes;
  int32_t scale_per_head, scale_f16;
  int32_t cap[3];          // pool capacities in pages
};

enum MoveMode : int { MOVE_DIRECT = 0, MOVE_GATHER = 1, MOVE_SCATTER = 2 };

struct MoveParams {
  int32_t L, Hkv, D, kv_dtype;
  TierPools pools;
  char* temp;              // staging rows of one layer: [rows][2][Hkv][D] in the KV dtype
  int32_t mode;
  int32_t layer0;          // the launch covers layers [layer0, layer0 + gridDim.y)
  int32_t* err;            // error word (debug index checks)
  int64_t temp_rows;       // staging rows `temp` holds
};
cudaError_t launch_move(const MoveParams& p, const Mover* movers, int64_t count, int layers, cudaStream_t s);

// s[b][pos] += (sum over layer slices and KV heads of acc at the slot holding
// pos) / (L * Hq); slots follow the attention page order (T0, T1, then T2 page
// lists) from the sequence's page base. The step's first launch wrote every
// slot it reads, so nothing is cleared.
struct FoldParams {
  int32_t B, Hkv, nslices;
  int32_t npages[3][kMaxBatch];
  int32_t page_base[kMaxBatch + 1];
  const int32_t* table[3];
  int32_t table_stride;
  const uint32_t* mask[3];
  const int32_t* posmap[3];
  int64_t max_slots;       // largest 16 * (pages of a sequence)
  double* s;               // [B][s_stride]
  int64_t s_stride;
  float* acc;              // [nslices][Hkv][acc_stride_h]
  int64_t acc_stride_l, acc_stride_h;
  double inv_lh;           // 1 / (L * Hq)
  int32_t* err;            // error word (debug index checks)
  int32_t cap[3];          // pool capacities in pages
};
cudaError_t launch_fold(const FoldParams& p, cudaStream_t s);

cudaError_t launch_quantize_rows(const void* x, int kv_dtype, int64_t rows, int row_len,
                                 int8_t* codes, void* scales, int scale_f16, cudaStream_t s);

}  // namespace tkv
