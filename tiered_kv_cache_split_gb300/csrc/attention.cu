// Split-K paged decode attention over the retained tiers, with the cumulative
// attention score of "Not All Thoughts Need HBM" (Methodology 2) fused into
// the softmax epilogue.
//
// One CTA serves one (sequence b, KV head, chunk of pages) and all G query
// heads that share that KV head, so every K/V byte is read from HBM once.
// Pages come from up to three sources in page order: the T0 pool in HBM, the
// T1 staging copy prefetched from pinned host DDR, and the T2 staging copy of
// 8-bit codes (Methodology 1, 3, 4). A producer warp streams the chunk's pages
// into a shared-memory ring with 1-D bulk TMA copies (cp.async.bulk, mbarrier
// transaction counts, L2 evict-first) as far ahead as the ring allows; the
// consumer warps take pages round-robin, each waiting on the page's "full"
// barrier and releasing the stage through its "empty" barrier.
//
// Two page processors share that pipeline and the epilogue:
//  * attn_split_mma_kernel (bf16 KV, G >= 2): the G query heads of a KV head
//    form the M side of bf16 tensor-core MMAs (mma.sync m16n8k16, fp32
//    accumulate): S^T = Q K^T over 16-key pages, then O^T += V^T P^T, with the
//    QK accumulators reused as the PV operand in registers. K and V tiles are
//    read with ldmatrix from the swizzled page layout (conflict-free). 8-bit
//    pages are widened to bf16 in shared memory first (the codes are exact in
//    bf16); their scales multiply the logits and the probabilities.
//  * attn_split_fma_kernel (fp32 KV, or one query head per KV head): fp32
//    registers and packed fp32x2 FMAs; the partial dot products of a
//    (head, row) are reduced across 8 lanes by a transposing butterfly.
// Per page both keep an online softmax per head in base 2 (log2(e)/sqrt(d)
// applied to the logits) and spill the raw logits. The warps of a CTA merge
// (m, Z, O) in shared memory and the CTA writes its partial; no CTA ever waits
// on another. A layer's epilogue — the global (M, Z) of each head from the
// partials, the merged output (each chunk's CTA merges a slice), and the exact
// softmax weights alpha = exp2(l - M) / Z of the chunk's slots summed over the
// G heads, added to a slot-indexed score accumulator (the fused score
// epilogue) — runs in the NEXT layer's attention launch, in each CTA after its
// own pages, so CTAs that finish early absorb it while the last ones stream.
// The last layer's epilogue (or a lone layer's) is attn_combine_kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "tkv_internal.h"

namespace tkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier; gives up after limit_ns nanoseconds
// (or 2^30 polls, whichever comes first).
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n"
      " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// D = A * B + D for one m16n8k16 bf16 tile with fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float i8f(uint32_t w, int byte) {
  return static_cast<float>(static_cast<int8_t>((w >> (8 * byte)) & 0xffu));
}
__device__ __forceinline__ int swz_chunk(int chunk, int row, int swz) { return chunk ^ (row & swz); }

// Pages of a CTA pass through ring positions 0, 1, 2, ...; position i uses
// ring stage i % kAttnStages and consumer warp i % kAttnWarps, and its page
// index and flags sit at slot i % kMeta (the producer resolves at most 32
// positions ahead of those still in the ring).
constexpr int kMeta = 64;

template <typename T, int G, int D>
struct Shape {
  static constexpr int GP = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
  static constexpr int ESZ = sizeof(T);
  static constexpr int ROWB = D * ESZ;        // bytes per full-precision row
  static constexpr int NCH = ROWB / 16;       // 16-byte chunks per row
  static constexpr int CPL = NCH / 8;         // chunks per lane in the fp32 QK
  static constexpr int EPC = 16 / ESZ;        // elements per chunk
  static constexpr int QE = CPL * EPC;        // fp32-QK elements per lane
  static constexpr int QP = QE / 2;
  static constexpr int VPL = D / 32;          // fp32-PV output elements per lane
  static constexpr int BLK = kPage * ROWB;    // K (or V) block of one page and head
  static constexpr int STAGE = 2 * BLK + 128; // + T2 scale record
  static constexpr int NV = GP * 4;           // fp32-QK partials per lane
  static constexpr int NL = NV >= 8 ? NV / 8 : 1;
  static_assert(CPL >= 1 && NCH % 8 == 0, "row must hold a multiple of 8 chunks");
  // a consumer warp's (O, m, Z) of a unit fits the stage of its unit-end marker
  static_assert((G * D + 2 * GP) * 4 <= STAGE, "merge data must fit a ring stage");
  static_assert(D % 32 == 0, "head_dim must be a multiple of 32");
};

// Shared-memory floats an epilogue item needs for its per-chunk output factors.
constexpr int kEpilogueFactors = kMaxChunksPerSeq * 8;

// Shared-memory layout of the attention CTA. The fp32 kernel also keeps the
// scaled query and per-warp probabilities in shared memory.
template <typename T, int G, int D, bool FMA>
struct Smem {
  using S = Shape<T, G, D>;
  static constexpr int RING = kAttnStages * S::STAGE;
  static_assert(RING >= kEpilogueFactors * 4, "the idle ring must hold the epilogue's chunk factors");
  static constexpr int QS = FMA ? S::GP * D * 4 : 0;
  static constexpr int PSW = S::GP * kPage + 8;   // floats per warp: p[GP][16], corr[GP]
  static constexpr int PS = FMA ? kAttnWarps * PSW * 4 : 0;
  static constexpr int PG = kMeta * 8;     // per ring position: page index, flags word
  static constexpr int DESC = kMeta * 16;  // producer's copy descriptors per ring position
  static constexpr int BARS = (2 * kAttnStages + 1) * 8;  // full[stages], empty[stages], merge
  static constexpr int MERGE = kAttnWarps * (G * D + 2 * S::GP) * 4;
  static constexpr int BODY = ((RING > MERGE ? RING : MERGE) + 127) / 128 * 128;
  static constexpr int off_q = BODY;
  static constexpr int off_p = off_q + QS;
  static constexpr int off_pg = off_p + PS;
  static constexpr int off_desc = (off_pg + PG + 15) / 16 * 16;
  static constexpr int off_bar = off_desc + DESC;
  static constexpr int TOTAL = off_bar + BARS;
};

// Resolves page-list index k of sequence b to (source, pool page id).
__device__ __forceinline__ void page_ref(const AttnParams& p, int b, int k, int& src, int& page) {
  int kk = k;
  src = 0;
  if (kk >= p.npages[0][b]) {
    kk -= p.npages[0][b];
    src = 1;
    if (kk >= p.npages[1][b]) {
      kk -= p.npages[1][b];
      src = 2;
    }
  }
  page = index_ok(p.err, DBG_ATTN_LIST, kk, p.table_stride) ? p.src[src].table[static_cast<int64_t>(b) * p.table_stride + kk]
                                                              : -1;
}

// What a CTA needs to know about its work item.
struct Work {
  int b, kvh, z, cf, jc, nch, ntot, k0, npg;  // the chunk: pages [k0, k0 + npg) of sequence b at layer z
};

// Index of work unit (layer z, chunk, KV head) in the partial buffers.
__device__ __forceinline__ int64_t unit_index(const AttnParams& p, int z, int chunk, int kvh) {
  return (static_cast<int64_t>(z) * p.total_chunks + chunk) * p.Hkv + kvh;
}

__device__ __forceinline__ Work find_work_at(const AttnParams& p, int chunk, int kvh, int z) {
  Work wk;
  wk.kvh = kvh;
  wk.z = z;
  int b = 0;
  while (b + 1 < p.B && p.chunk_first[b + 1] <= chunk) ++b;
  wk.b = b;
  wk.cf = p.chunk_first[b];
  wk.jc = chunk - wk.cf;
  wk.nch = p.chunk_first[b + 1] - wk.cf;
  const int n01 = p.npages[0][b] + p.npages[1][b];
  wk.ntot = n01 + p.npages[2][b];
  // cost-balanced split of the sequence's pages over its chunks
  const int64_t cost = static_cast<int64_t>(kCostFull) * n01 + static_cast<int64_t>(kCostI8) * p.npages[2][b];
  wk.k0 = page_at_cost((wk.jc * cost) / wk.nch, n01);
  wk.npg = page_at_cost(((wk.jc + 1) * cost) / wk.nch, n01) - wk.k0;
  if (wk.npg > kMaxChunkPages) {  // the host plan never makes one
    if (threadIdx.x == 0) atomicExch(p.err, DEV_BAD_INDEX);
    wk.npg = 0;
  }
  return wk;
}

// Metadata ring records other than pages (meta_k >= 0): a pad, the end of the
// CTA's last unit, or the end of a unit that names the CTA's next unit n (-3 - n).
constexpr int kMetaPad = -2, kMetaLast = -1;
__device__ __forceinline__ int end_marker(int next) { return next < 0 ? kMetaLast : -3 - next; }
__device__ __forceinline__ int marker_next(int k) { return -3 - k; }

// A CTA's first unit, and the unit it runs after unit u: the next unhanded one
// of the launch's counter, or with no counter a static stride.
__device__ __forceinline__ int first_unit(const AttnParams& p) {
  if (p.ep_own == nullptr) return static_cast<int>(blockIdx.x);
  return atomicAdd(&p.ep_own->units, 1);
}
__device__ __forceinline__ int claim_next_unit(const AttnParams& p, int u) {
  if (p.ep_own == nullptr) return u + static_cast<int>(gridDim.x);
  return atomicAdd(&p.ep_own->units, 1);
}

// Work unit u of a launch, in hand-out order: the sequences by decreasing chunk
// cost (p.order), and within a sequence over (layer, KV head, chunk), chunk
// fastest. A persistent CTA claims its units one at a time (first_unit,
// claim_next_unit), so the largest units go first and the CTAs finish close
// together. A unit's result does not depend on the CTA that runs it.
__device__ __forceinline__ Work unit_work(const AttnParams& p, int u) {
  const int per = p.Hkv * p.nlayers;  // units per chunk of a sequence
  int r = 0;
  while (r + 1 < p.B && p.order_chunk_first[r + 1] * per <= u) ++r;
  const int b = p.order[r];
  const int nch = p.chunk_first[b + 1] - p.chunk_first[b];
  const int v = u - p.order_chunk_first[r] * per;
  const int rest = v / nch;
  return find_work_at(p, p.chunk_first[b] + v % nch, rest % p.Hkv, rest / p.Hkv);
}
__device__ __forceinline__ int launch_units(const AttnParams& p) { return p.total_chunks * p.Hkv * p.nlayers; }

// This work unit's spilled logits (k-th page of the sequence at slot (k * G + g) * 16 + row).
__device__ __forceinline__ float* spill_of(const AttnParams& p, float* spill, const Work& wk) {
  return spill + wk.z * p.spill_stride_l + static_cast<int64_t>(wk.b) * p.spill_stride_b +
         static_cast<int64_t>(wk.kvh) * p.spill_stride_h + static_cast<int64_t>(p.page_base[wk.b]) * p.G * kPage;
}

// Initialises the ring's full and empty barriers (thread 0); a CTA barrier
// must follow before any thread uses them.
template <typename L>
__device__ __forceinline__ void init_barriers(char* smem) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bar);
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2 * kAttnStages; ++s) mbar_init(smem_u32(bars + s), 1);
    mbar_init(smem_u32(bars + 2 * kAttnStages), kAttnWarps);  // one arrival per consumer warp
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
}

// Barrier among the consumer warps only (the producer warp runs ahead).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kAttnWarps * 32) : "memory");
}

// A page's copy, resolved once: the source address of its (KV head) record
// with flags in the low bits (bit 0: 8-bit page, bit 1: per-head scales), and
// for 8-bit pages the address of its scale record.
struct PageCopy {
  unsigned long long src;
  unsigned long long scales;
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Producer lane: bulk-copy page i of the chunk into ring stage st, completing
// the stage's "full" barrier with the page's byte count.
template <typename S>
__device__ __forceinline__ void issue_page(const PageCopy& c, int st, char* ring, uint32_t full0,
                                           uint64_t policy) {
  const bool i8 = c.src & 1ull;
  const char* gsrc = reinterpret_cast<const char*>(c.src & ~15ull);
  const uint32_t dst = smem_u32(ring + st * S::STAGE);
  const uint32_t bar = full0 + st * 8;
  const uint32_t bytes = i8 ? 2u * kPage * (S::ROWB / S::ESZ) : 2u * S::BLK;
  const uint32_t sbytes = i8 ? ((c.src & 2ull) ? 64u : 128u) : 0u;
  mbar_expect_tx(bar, bytes + sbytes);
  bulk_g2s(dst, gsrc, bytes, bar, policy);
  if (sbytes) bulk_g2s(dst + 2 * S::BLK, reinterpret_cast<const char*>(c.scales), sbytes, bar, policy);
}

// Per-page word the producer publishes for the consumers: valid-slot bits in
// the low 16 bits, then the page's source traits, so that the consumers never
// index the source table.
constexpr uint32_t kFlagI8 = 1u << 16, kFlagPerHead = 1u << 17, kFlagHost = 1u << 21;
constexpr int kFlagSwzShift = 18;
__device__ __forceinline__ uint32_t page_flags(uint32_t valid, bool i8, bool per_head, int swz, bool host) {
  return (valid & 0xffffu) | (i8 ? kFlagI8 : 0u) | (per_head ? kFlagPerHead : 0u) |
         (static_cast<uint32_t>(swz & 7) << kFlagSwzShift) | (host ? kFlagHost : 0u);
}

// Resolves page i of the chunk (source, pool page, valid mask and traits, copy
// descriptor) and publishes it in shared memory.
__device__ __forceinline__ void resolve_page(const AttnParams& p, const Work& wk, int k, int slot, int32_t* meta_k,
                                             uint32_t* meta_f, PageCopy* desc) {
  int src, page;
  page_ref(p, wk.b, k, src, page);
  const PageSource& ps = p.src[src];
  // debug build: a page id outside its pool reads page 0 with no valid slot instead
  const bool page_ok = index_ok(p.err, DBG_ATTN_PAGE, page, ps.pages);
  if (!page_ok) page = 0;
  meta_k[slot] = k;
  const bool i8 = ps.kind == SRC_INT8;
  meta_f[slot] = page_flags(page_ok ? ps.mask[page] : 0u, i8, ps.scale_per_head != 0, ps.swz, ps.host != 0);
  PageCopy c;
  c.src = reinterpret_cast<unsigned long long>(ps.base + wk.z * ps.layer_bytes + static_cast<int64_t>(page) * ps.page_bytes +
                                               static_cast<int64_t>(wk.kvh) * ps.head_bytes) |
          (i8 ? 1ull : 0ull) | ((i8 && ps.scale_per_head) ? 2ull : 0ull) | (ps.host ? 4ull : 0ull);
  c.scales = i8 ? reinterpret_cast<unsigned long long>(ps.scales + wk.z * ps.scale_layer_bytes +
                                                       static_cast<int64_t>(page) * ps.scale_page_bytes +
                                                       (ps.scale_per_head ? static_cast<int64_t>(wk.kvh) * 64 : 0))
                : 0ull;
  desc[slot] = c;
}

// Producer warp: read a page that sits in pinned host memory into its ring
// stage with plain 16-byte loads (K block then V block; for an 8-bit page the
// codes, then its scale record at the stage's scale area). All loads of a
// batch are issued before any store, so the warp keeps 8 x 512 B in flight over
// the host link.
template <typename S>
__device__ __forceinline__ void load_host_page(const PageCopy& c, char* stage, int lane) {
  const bool i8 = c.src & 1ull;
  const uint4* src = reinterpret_cast<const uint4*>(c.src & ~15ull);
  uint4* dst = reinterpret_cast<uint4*>(stage);
  const int n = (i8 ? 2 * kPage * (S::ROWB / S::ESZ) : 2 * S::BLK) / 16;
  constexpr int kBatch = 8;
  for (int base = 0; base < n; base += 32 * kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + j * 32 + lane;
      if (i < n) v[j] = src[i];
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = base + j * 32 + lane;
      if (i < n) dst[i] = v[j];
    }
  }
  if (i8) {
    const int sn = ((c.src & 2ull) ? 64 : 128) / 16;
    if (lane < sn)
      reinterpret_cast<uint4*>(stage + 2 * S::BLK)[lane] = reinterpret_cast<const uint4*>(c.scales)[lane];
  }
  __syncwarp();
}

// The producer warp's job, for each work unit of this persistent CTA in turn
// (from `first`; at the start of each unit it claims the next): resolve the unit's pages (one lane per page, 32 per round; the first
// round's copies go out at once, later rounds are resolved while the ring is
// full) and keep the ring full; then pad positions (kMetaPad) up to a multiple
// of the consumer warp count, and one unit-end marker per consumer warp (the
// claimed next unit, or kMetaLast; flags word = the first marker's position),
// each completed by a plain arrive. Every unit thus starts at a multiple of the
// warp count, so its page j always goes to consumer warp j % warps and the
// result does not depend on which CTA runs the unit. The ring runs on across
// units, so the next unit's pages stream in while the consumers merge the last
// one. Returns the ring positions handled (lane 0).
template <typename S>
__device__ int produce(const AttnParams& p, int first, int32_t* meta_k, uint32_t* meta_f, PageCopy* desc, char* ring,
                       uint32_t full0, uint32_t empty0, volatile int* abort_flag) {
  static_assert(kMeta >= 32 + kAttnStages + 2 * kAttnWarps, "metadata ring too small");
  const int lane = threadIdx.x & 31;
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  int pos = 0, issued = 0;
  bool ok = true;  // lane 0: no bounded wait gave up
  auto stage_free = [&](int i) {  // position i's stage has been released by position i - stages
    return i < kAttnStages || mbar_wait(empty0 + (i % kAttnStages) * 8, ((i / kAttnStages) - 1) & 1, p.wait_limit_ns);
  };
  // test hook: the CTA that runs unit 0 withholds its first page, so that a
  // consumer's bounded wait runs out (nothing is in flight for that stage)
  const bool stall = p.stall_first_page && first == 0;
  // Lane 0 waits for each stage and issues its bulk copy; a page in pinned host
  // memory is instead read by the whole warp with plain loads (load_host_page)
  // and its stage completed with a plain arrive.
  auto issue = [&](int n) {
    for (int j = 0; j < n; ++j) {
      const int i = pos + j;
      int go = 0;
      if (lane == 0) go = ok && stage_free(i);
      go = __shfl_sync(kFull, go, 0);
      if (!go) {
        if (lane == 0 && ok) {
          ok = false;
          *abort_flag = 1;
        }
        break;
      }
      const int st = i % kAttnStages;
      const PageCopy c = desc[i % kMeta];
      if (c.src & 4ull) {
        if (!(stall && i == 0)) {
          load_host_page<S>(c, ring + st * S::STAGE, lane);
          if (lane == 0) mbar_arrive(full0 + st * 8);
        }
      } else if (lane == 0 && !(stall && i == 0)) {
        issue_page<S>(c, st, ring, full0, policy);
      }
      if (lane == 0) ++issued;
    }
    pos += n;
    __syncwarp();
  };
  const int units = launch_units(p);
  for (int u = first; u < units;) {
    // claim the unit to run after this one now, so the claim's latency hides behind this unit's pages
    int next = 0;
    if (lane == 0) next = claim_next_unit(p, u);
    next = __shfl_sync(kFull, next, 0);
    if (next >= units) next = -1;
    const Work wk = unit_work(p, u);
    for (int r = 0; r < wk.npg; r += 32) {
      const int n = min(32, wk.npg - r);
      if (lane < n) resolve_page(p, wk, wk.k0 + r + lane, (pos + lane) % kMeta, meta_k, meta_f, desc);
      __syncwarp();
      issue(n);
    }
    const int pad = (kAttnWarps - pos % kAttnWarps) % kAttnWarps;
    if (lane == 0 && ok) {
      for (int j = 0; j < pad + kAttnWarps; ++j) {
        const int i = pos + j;
        if (!stage_free(i)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        meta_k[i % kMeta] = j < pad ? kMetaPad : end_marker(next);
        meta_f[i % kMeta] = static_cast<uint32_t>(pos + pad);
        mbar_arrive(full0 + (i % kAttnStages) * 8);
        ++issued;
      }
    }
    pos += pad + kAttnWarps;
    __syncwarp();
    if (!__shfl_sync(kFull, ok ? 1 : 0, 0) || next < 0) break;
    u = next;
  }
  return issued;
}

// Stage of the unit-end marker that consumer warp ww takes when the unit's
// markers start at ring position `first`, a multiple of the warp count
// (position i goes to warp i % warps).
__device__ __forceinline__ int marker_stage(int first, int ww) { return (first + ww) % kAttnStages; }

// Merges the consumer warps' (O, m, Z) of a unit — each warp's in the stage of
// its unit-end marker, laid out [G][D] floats, then m[GP], Z[GP] — into the
// unit's partial: O relative to the unit's max M, and (M, Z) per head. Run by
// the consumer threads (ctid < warps * 32).
template <typename T, int G, int D>
__device__ void merge_partial(const AttnParams& p, const Work& wk, const char* ring, int first, int ctid) {
  using S = Shape<T, G, D>;
  const float* mo[kAttnWarps];
#pragma unroll
  for (int ww = 0; ww < kAttnWarps; ++ww)
    mo[ww] = reinterpret_cast<const float*>(ring + marker_stage(first, ww) * S::STAGE);
  const int64_t pidx = unit_index(p, wk.z, wk.cf + wk.jc, wk.kvh);
  for (int idx = ctid; idx < G * D; idx += kAttnWarps * 32) {
    const int g = idx / D;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kAttnWarps; ++ww) M = fmaxf(M, mo[ww][G * D + g]);
    float o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int ww = 0; ww < kAttnWarps; ++ww) {
        const float mw = mo[ww][G * D + g];
        if (mw != -INFINITY) o += mo[ww][idx] * exp2f(mw - M);
      }
    }
    p.part_o[pidx * G * D + idx] = o;
  }
  if (ctid < G) {
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kAttnWarps; ++ww) M = fmaxf(M, mo[ww][G * D + ctid]);
    float Z = 0.f;
    if (M != -INFINITY)
#pragma unroll
      for (int ww = 0; ww < kAttnWarps; ++ww) {
        const float mw = mo[ww][G * D + ctid];
        if (mw != -INFINITY) Z += mo[ww][G * D + S::GP + ctid] * exp2f(mw - M);
      }
    p.part_m[pidx * G + ctid] = M;
    p.part_z[pidx * G + ctid] = Z;
  }
}

// Barrier of the consumer warps at a unit end (an mbarrier with one arrival
// per warp, so that a warp whose own wait gave up cannot hold the others for
// ever: they give up too). Returns false when the wait gave up.
__device__ __forceinline__ bool consumers_meet(uint32_t bar, uint32_t& phase, int lane, uint64_t limit_ns) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = __all_sync(kFull, mbar_wait(bar, phase & 1u, limit_ns));
  ++phase;
  return ok;
}

// After an abort: wait (bounded) for the copies still in flight to land.
__device__ void drain(int issued, uint32_t full0, uint64_t limit_ns) {
  const int lo = issued > kAttnStages ? issued - kAttnStages : 0;
  for (int i = lo; i < issued; ++i) (void)mbar_wait(full0 + (i % kAttnStages) * 8, (i / kAttnStages) & 1, limit_ns);
}



__device__ __forceinline__ float t2_scale(const char* stage_scales, bool per_head, int idx) {
  return per_head ? __half2float(reinterpret_cast<const __half*>(stage_scales)[idx])
                  : reinterpret_cast<const float*>(stage_scales)[idx];
}

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// The epilogue of one (layer, sequence, KV head) group of a finished layer, run
// by NT threads (tid < NT, NT a multiple of 32): global (M, Z) of each head from
// the group's chunk partials (one warp per head), the merged output, and the
// exact softmax weights alpha = exp2(l - M) / Z of every slot of the sequence's
// pages, summed over the G heads and added to the score accumulator at slot
// 16 * k + row of the sequence's page list (the fused score epilogue of
// Methodology 2). Masked slots hold -inf logits, so they add exactly 0 and no
// page metadata is read. `sync` synchronises the NT threads. `wk` describes the
// group: its first chunk, with k0 = 0 and npg = all the sequence's pages.
struct LayerBufs {
  const float* part_o;
  const float* part_m;
  const float* part_z;
  const float* spill;
  void* out;
  float* acc;   // score accumulator slice of the launch's first layer
  bool first;   // the launch is a step's first: its items write the slices instead of adding to them
};

// Every epilogue item is read after the grid that wrote it has finished, so the
// read-only path is safe.
__device__ __forceinline__ float ld_part(const float* p) { return __ldg(p); }
#ifndef TKV_EPILOGUE_QUADS
#define TKV_EPILOGUE_QUADS 2
#endif
constexpr int kEpilogueQuads = TKV_EPILOGUE_QUADS;  // four-row groups in flight per thread in the logit pass
// four consecutive floats; p is 16-byte aligned (page slots start on multiples of 16 floats)
__device__ __forceinline__ float4 ld_part4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// One epilogue item: (1) the group's (M, 1/Z) per head from its chunk partials,
// and each chunk's output factor exp2(m_j - M) / Z into sF ([chunk][8], -1 for a
// chunk with no valid slot); (2) the G * D outputs, sum over chunks of factor x
// partial output, every thread's loads independent of one another; (3) the
// logit pass into the score accumulator.
template <typename T, int G, int D, int NT, typename Sync>
__device__ void layer_epilogue(const AttnParams& p, const LayerBufs& lb, const Work& wk, int tid,
                               float* sM, float* sIZ, float* sF, Sync sync) {
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t base = unit_index(p, wk.z, wk.cf, wk.kvh);  // partial of chunk j: base + j * Hkv
  const int nch = wk.nch;
  for (int g = warp; g < G; g += NT / 32) {
    // one round of loads: up to 64 chunks per lane pair (m, z) in registers
    float mj[2], zj[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int j = lane + 32 * r;
      const int64_t pj = (base + static_cast<int64_t>(j) * p.Hkv) * G + g;
      mj[r] = j < nch ? ld_part(lb.part_m + pj) : -INFINITY;
      zj[r] = j < nch ? ld_part(lb.part_z + pj) : 0.f;
    }
    float M = fmaxf(mj[0], mj[1]);
    for (int j = lane + 64; j < nch; j += 32)
      M = fmaxf(M, ld_part(lb.part_m + (base + static_cast<int64_t>(j) * p.Hkv) * G + g));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, m));
    float Z = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int r = 0; r < 2; ++r)
        if (mj[r] != -INFINITY) Z += zj[r] * exp2f(mj[r] - M);
      for (int j = lane + 64; j < nch; j += 32) {
        const int64_t pj = (base + static_cast<int64_t>(j) * p.Hkv) * G + g;
        const float m2 = ld_part(lb.part_m + pj);
        if (m2 != -INFINITY) Z += ld_part(lb.part_z + pj) * exp2f(m2 - M);
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) Z += __shfl_xor_sync(kFull, Z, m);
    const float IZ = Z > 0.f ? 1.f / Z : 0.f;
    if (lane == 0) {
      sM[g] = M;
      sIZ[g] = IZ;
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int j = lane + 32 * r;
      if (j < nch) sF[j * 8 + g] = (M != -INFINITY && mj[r] != -INFINITY) ? exp2f(mj[r] - M) * IZ : -1.f;
    }
    for (int j = lane + 64; j < nch; j += 32) {
      const float m2 = ld_part(lb.part_m + (base + static_cast<int64_t>(j) * p.Hkv) * G + g);
      sF[j * 8 + g] = (M != -INFINITY && m2 != -INFINITY) ? exp2f(m2 - M) * IZ : -1.f;
    }
  }
  sync();
  {
    // the G * D outputs: each thread's EPT elements, chunk by chunk
    constexpr int EPT = (G * D + NT - 1) / NT;
    T* out = reinterpret_cast<T*>(lb.out) + wk.z * p.out_stride_l + static_cast<int64_t>(wk.b) * p.out_stride_b +
             static_cast<int64_t>(wk.kvh) * G * D;
    float o[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) o[e] = 0.f;
#pragma unroll 2
    for (int j = 0; j < nch; ++j) {
      const float* po = lb.part_o + (base + static_cast<int64_t>(j) * p.Hkv) * G * D;
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const int idx = tid + e * NT;
        if (idx < G * D) {
          const float f = sF[j * 8 + idx / D];
          if (f >= 0.f) o[e] += ld_part(po + idx) * f;
        }
      }
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = tid + e * NT;
      if (idx < G * D) store_out(out + idx, o[e]);
    }
  }
  if (lb.acc == nullptr) return;
  const float* __restrict__ spill_b = spill_of(p, const_cast<float*>(lb.spill), wk);
  float* __restrict__ accb = lb.acc + wk.z * p.acc_stride_l + static_cast<int64_t>(wk.b) * p.acc_stride_b +
                             static_cast<int64_t>(wk.kvh) * p.acc_stride_h + static_cast<int64_t>(p.page_base[wk.b]) * kPage;
  float M[G], IZ[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = sM[g];
    IZ[g] = sIZ[g];
  }
  // Each thread takes four consecutive rows of a page at a time (16-byte loads
  // of every head's logits and of the accumulator), U quads in flight: the
  // pass is bound by load latency, so bytes in flight per load decide its speed.
  constexpr int U = kEpilogueQuads;
  const int quads = wk.npg * (kPage / 4);
  for (int first = tid; first < quads; first += NT * U) {
    float4 l[U][G], old[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int qd = first + u * NT;
      if (qd < quads) {
        const int64_t k = wk.k0 + (qd >> 2);
        const int r0 = (qd & 3) * 4;
#pragma unroll
        for (int g = 0; g < G; ++g) l[u][g] = ld_part4(spill_b + (k * G + g) * kPage + r0);
        old[u] = lb.first ? make_float4(0.f, 0.f, 0.f, 0.f)
                          : __ldcg(reinterpret_cast<const float4*>(accb + k * kPage + r0));  // chunks share lines
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int qd = first + u * NT;
      if (qd < quads) {
        const int64_t k = wk.k0 + (qd >> 2);
        const int r0 = (qd & 3) * 4;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          a.x += exp2f(l[u][g].x - M[g]) * IZ[g];
          a.y += exp2f(l[u][g].y - M[g]) * IZ[g];
          a.z += exp2f(l[u][g].z - M[g]) * IZ[g];
          a.w += exp2f(l[u][g].w - M[g]) * IZ[g];
        }
        *reinterpret_cast<float4*>(accb + k * kPage + r0) =
            make_float4(old[u].x + a.x, old[u].y + a.y, old[u].z + a.z, old[u].w + a.w);
      }
    }
  }
}

// Epilogue item `item` of a launch: group (layer z, sequence b, KV head) with
// item = (z * B + b) * Hkv + kvh, covering all of the sequence's pages. One item
// per group computes the global (M, Z) once and streams the group's logits in
// one pass (latency-bound work: fewer, larger items keep more loads in flight).
__device__ __forceinline__ Work epilogue_work(const AttnParams& p, int item) {
  const int kvh = item % p.Hkv, rest = item / p.Hkv;
  const int b = rest % p.B, z = rest / p.B;
  Work wk = find_work_at(p, p.chunk_first[b], kvh, z);
  wk.jc = 0;
  wk.k0 = 0;
  wk.npg = wk.ntot;
  return wk;
}
__device__ __forceinline__ int epilogue_items_per_layer(const AttnParams& p) { return p.B * p.Hkv; }

// Claims an epilogue item of a finished launch: the next unclaimed (KV head,
// chunk) of its first layer that has one left, as layer * per_layer + index,
// or -1 when none is left. Every claim is one fetch-and-add on that layer's
// counter, so CTAs that finish together never retry against one another.
__device__ __forceinline__ int claim_item(EpCounters* ctr, int nlayers, int per_layer) {
  for (int z = 0; z < nlayers; ++z) {
    if (*reinterpret_cast<volatile int32_t*>(ctr->claim + z) >= per_layer) continue;  // layer handed out
    const int i = atomicAdd(ctr->claim + z, 1);
    if (i < per_layer) return z * per_layer + i;
  }
  return -1;
}

// The epilogue of a launch's items, as a kernel of its own launched as a
// programmatic dependent of that attention launch (for a lone call, and for the
// last launch of a decode step): CTAs claim the launch's items.
constexpr int kCombineThreads = 256;

template <typename T, int G, int D>
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  __shared__ float sM[8], sIZ[8];
  __shared__ float sF[kEpilogueFactors];
  __shared__ int s_item;
  const int per_layer = epilogue_items_per_layer(p);
  // wait here until the attention kernel's partials and spilled logits are complete and visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const LayerBufs lb{p.part_o, p.part_m, p.part_z, p.spill, p.out, p.acc, p.first_of_step != 0};
  for (;;) {
    __syncthreads();
    if (threadIdx.x == 0) s_item = claim_item(p.ep_own, p.nlayers, per_layer);
    __syncthreads();
    const int item = s_item;
    if (item < 0) break;
    layer_epilogue<T, G, D, kCombineThreads>(p, lb, epilogue_work(p, item), threadIdx.x, sM, sIZ, sF,
                                             [] { __syncthreads(); });
  }
}

// The previous launch's epilogue, run by all warps of an attention CTA: before
// its first unit (CTAs blockIdx.x < ep_first_ctas, while the others stream) and
// once the launch's units run out (any items left). The items — one per
// (layer, sequence, KV head) group of the previous launch — are handed out by
// that launch's counters. While a CTA runs items its page ring is idle, so the
// items' chunk factors sit in the ring's first stages. (Running each group's
// item in its own launch, by the CTA that finishes the group, measured slower:
// the last groups' items form a tail and an item stalls its CTA's ring.)
template <typename T, int G, int D>
__device__ __forceinline__ void prev_launch_epilogue(const AttnParams& p, int tid, float* sM, float* sIZ,
                                                     float* sF, volatile int* s_item) {
  if (!p.has_prev) return;
  constexpr int NT = (kAttnWarps + 1) * 32;
  const int per_layer = epilogue_items_per_layer(p);
  const LayerBufs lb{p.prev_part_o, p.prev_part_m, p.prev_part_z, p.prev_spill, p.prev_out, p.acc,
                     p.prev_first_of_step != 0};
  for (;;) {
    __syncthreads();
    if (tid == 0) *s_item = claim_item(p.ep_prev, p.prev_nlayers, per_layer);
    __syncthreads();
    const int item = *s_item;
    if (item < 0) break;
    layer_epilogue<T, G, D, NT>(p, lb, epilogue_work(p, item), tid, sM, sIZ, sF, [] { __syncthreads(); });
  }
}

// ===================================================================== MMA
// Four signed 8-bit codes (one word, byte 0 first) as two bf16x2 words, exactly,
// without conversion instructions: byte b + 128 placed in the low mantissa bits
// of 2^23 gives the float 2^23 + b + 128; subtracting 2^23 + 128 leaves b; the
// upper half of that float is its bf16 (|b| <= 128 needs 8 significant bits).
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;  // b + 128 as unsigned bytes
  const float2 bias = make_float2(-8388736.f, -8388736.f);
  const float2 one = make_float2(1.f, 1.f);
  const float2 a = ffma2(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                     __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441))), one, bias);
  const float2 b = ffma2(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                     __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443))), one, bias);
  lo = __byte_perm(__float_as_uint(a.x), __float_as_uint(a.y), 0x7632);
  hi = __byte_perm(__float_as_uint(b.x), __float_as_uint(b.y), 0x7632);
}

// Widens an 8-bit page (codes at stage + 0: K block then V block, unswizzled)
// into bf16 K and V blocks in the swizzled layout, in place. The V codes are
// widened first (their bf16 block lies past the codes), then the K codes, each
// block read whole into registers before it is written.
template <int D>
__device__ __forceinline__ void widen_i8_block(char* stage, int kv, int lane) {
  constexpr int ROWB = D * 2;
  constexpr int PER_BLOCK = kPage * D / 16;  // uint4 of codes in one block
  constexpr int PER_LANE = PER_BLOCK / 32;
  uint4 v[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) v[i] = reinterpret_cast<const uint4*>(stage + kv * kPage * D)[lane + 32 * i];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int vec = lane + 32 * i;                 // 16 codes: row r, columns [16c, 16c + 16)
    const int r = vec / (D / 16), c = vec % (D / 16);
    uint4 lo, hi;
    i8x4_to_bf16x4(v[i].x, lo.x, lo.y);
    i8x4_to_bf16x4(v[i].y, lo.z, lo.w);
    i8x4_to_bf16x4(v[i].z, hi.x, hi.y);
    i8x4_to_bf16x4(v[i].w, hi.z, hi.w);
    char* rowp = stage + kv * kPage * ROWB + r * ROWB;
    *reinterpret_cast<uint4*>(rowp + swz_chunk(2 * c, r, kSwizzle) * 16) = lo;
    *reinterpret_cast<uint4*>(rowp + swz_chunk(2 * c + 1, r, kSwizzle) * 16) = hi;
  }
  __syncwarp();
}

template <int D>
__device__ __forceinline__ void widen_i8_page(char* stage, int lane) {
  widen_i8_block<D>(stage, 1, lane);  // V codes [16 D, 32 D) -> bf16 V block [32 D, 64 D)
  widen_i8_block<D>(stage, 0, lane);  // K codes [0, 16 D)     -> bf16 K block [0, 32 D)
}

template <int G, int D>
__global__ void __launch_bounds__((kAttnWarps + 1) * 32, 3)
    attn_split_mma_kernel(const __grid_constant__ AttnParams p) {
  using T = __nv_bfloat16;
  using S = Shape<T, G, D>;
  using L = Smem<T, G, D, false>;
  constexpr int KS = D / 16;  // k-steps of QK over d, and m-tiles of PV over d
  static_assert(G >= 2 && G <= 8, "tensor-core path serves 2..8 query heads per KV head");
  extern __shared__ __align__(128) char smem[];
  __shared__ volatile int s_abort;
  __shared__ float s_epM[8], s_epIZ[8];  // previous launch's (M, 1 / Z) per head
  __shared__ volatile int s_item;
  __shared__ int s_first;

  const int tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;  // fragment row group and column pair
  if (tid == 0) s_abort = 0;
  if (tid == 0 && p.span) atomicMin(p.span, global_ns());
  if (tid == 0 && blockIdx.x == 0) {
    if (p.span_next) {
      p.span_next[0] = ~0ull;
      p.span_next[1] = 0ull;
    }
    if (p.ep_clear) {  // counters of the launch after next
      for (int z = 0; z < kMaxLaunchLayers; ++z) p.ep_clear->claim[z] = 0;
      p.ep_clear->units = 0;
    }
    if (p.started) {                  // tells the copy stream this launch is under way
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.started), "r"(p.launch_seq) : "memory");
    }
  }
  init_barriers<L>(smem);
  __syncthreads();
  // the first ep_first_ctas CTAs take epilogue items of the previous launch
  // before any unit (the ring is still idle), while the others start streaming
  if (static_cast<int>(blockIdx.x) < p.ep_first_ctas) {
    prev_launch_epilogue<T, G, D>(p, tid, s_epM, s_epIZ, reinterpret_cast<float*>(smem), &s_item);
    // the items wrote the ring's first stage through the generic proxy: order
    // those writes before the bulk copies that will fill it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (tid == 0) s_first = first_unit(p);
  __syncthreads();
  const int first = s_first;

  int32_t* meta_k = reinterpret_cast<int32_t*>(smem + L::off_pg);
  uint32_t* meta_f = reinterpret_cast<uint32_t*>(meta_k + kMeta);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bar);
  char* ring = smem;
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + kAttnStages * 8;
  const uint32_t merge_bar = full0 + 2 * kAttnStages * 8;
  const bool consumer = w < kAttnWarps;
  int issued = 0;
  if (!consumer)
    issued = produce<S>(p, first, meta_k, meta_f, reinterpret_cast<PageCopy*>(smem + L::off_desc), ring, full0,
                        empty0, &s_abort);

  const int units = launch_units(p);
  int u = first;
  Work wk{};
  uint32_t qa[KS][2];                    // Q fragments (A operand, heads as rows; rows 8..15 zero)
  float* spill_b = nullptr;
  // the unit's query fragments and logit spill
  auto start_unit = [&]() {
    wk = unit_work(p, u);
    const T* q = reinterpret_cast<const T*>(p.q) + wk.z * p.q_stride_l + static_cast<int64_t>(wk.b) * p.q_stride_b +
                 static_cast<int64_t>(wk.kvh) * G * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (g < G) {
        qa[ks][0] = *reinterpret_cast<const uint32_t*>(q + g * D + 16 * ks + 2 * t);
        qa[ks][1] = *reinterpret_cast<const uint32_t*>(q + g * D + 16 * ks + 2 * t + 8);
      } else {
        qa[ks][0] = qa[ks][1] = 0u;
      }
    }
    spill_b = spill_of(p, p.spill, wk);
  };
  if (consumer && u < units) start_unit();

  float m_run = -INFINITY, z_run = 0.f;  // softmax state of head g
  float o[KS][4];                        // O^T tiles: d rows, head columns
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  uint32_t mphase = 0;                   // merge-barrier phases completed
  // per-lane ldmatrix row / chunk selectors (matrix = lane / 8)
  const int lrow = ((lane >> 4) << 3) | (lane & 7);
  const int lchunk = (lane >> 3) & 1;

  for (int i = w; consumer && u < units; i += kAttnWarps) {
    const int st = i % kAttnStages;
    const bool ok = __all_sync(kFull, mbar_wait(full0 + st * 8, (i / kAttnStages) & 1, p.wait_limit_ns));
    if (!ok) {
      if (lane == 0) s_abort = 1;
      break;
    }
    char* stage = ring + st * S::STAGE;
    const int k = meta_k[i % kMeta];  // page index in the sequence's list, or a pad or unit-end record
    if (k == kMetaPad) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + st * 8);
      continue;
    }
    if (k < 0) {
      // ---- unit end: this warp's (O, m, Z) into its marker's stage, then merge
      const int first = static_cast<int>(meta_f[i % kMeta]);
      float* mo = reinterpret_cast<float*>(stage);
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d0 = 16 * mt + g;
        if (2 * t < G) {
          mo[(2 * t) * D + d0] = o[mt][0];
          mo[(2 * t) * D + d0 + 8] = o[mt][2];
        }
        if (2 * t + 1 < G) {
          mo[(2 * t + 1) * D + d0] = o[mt][1];
          mo[(2 * t + 1) * D + d0 + 8] = o[mt][3];
        }
      }
      if (t == 0 && g < G) {
        mo[G * D + g] = m_run;
        mo[G * D + S::GP + g] = z_run;
      }
      if (!consumers_meet(merge_bar, mphase, lane, p.wait_limit_ns)) {
        if (lane == 0) s_abort = 1;
        break;
      }
      merge_partial<T, G, D>(p, wk, ring, first, tid);
      if (!consumers_meet(merge_bar, mphase, lane, p.wait_limit_ns)) {  // every warp has read every stage
        if (lane == 0) s_abort = 1;
        break;
      }
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes before the next copy
        mbar_arrive(empty0 + st * 8);
      }
      if (k == kMetaLast) break;  // the producer claimed no further unit
      u = marker_next(k);
      start_unit();
      m_run = -INFINITY;
      z_run = 0.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      continue;
    }
    const uint32_t flags = meta_f[i % kMeta];
    const uint32_t mask = flags & 0xffffu;
    const bool i8 = (flags & kFlagI8) != 0;
    const bool host = (flags & kFlagHost) != 0;
    const int swz = i8 ? kSwizzle : static_cast<int>((flags >> kFlagSwzShift) & 7u);
    if (i8) widen_i8_page<D>(stage, lane);
    const uint32_t kbase = smem_u32(stage), vbase = kbase + S::BLK;

    // ---- S^T = Q K^T: two n-tiles of 8 keys -----------------------------------
    // even and odd k-steps accumulate separately: four independent MMA chains
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ks += 2) {
      uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
      ldsm_x4(kbase + lrow * S::ROWB + swz_chunk(2 * ks + lchunk, lrow, swz) * 16, b0, b1, b2, b3);
      ldsm_x4(kbase + lrow * S::ROWB + swz_chunk(2 * ks + 2 + lchunk, lrow, swz) * 16, c0, c1, c2, c3);
      mma_bf16(s0, qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
      mma_bf16(s1, qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
      mma_bf16(s2, qa[ks + 1][0], 0u, qa[ks + 1][1], 0u, c0, c1);
      mma_bf16(s3, qa[ks + 1][0], 0u, qa[ks + 1][1], 0u, c2, c3);
    }
    // this lane's logits: head g, keys 2t, 2t+1, 8+2t, 9+2t
    float l[4] = {s0[0] + s2[0], s0[1] + s2[1], s1[0] + s3[0], s1[1] + s3[1]};
    const int rows[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
    const char* sc = stage + 2 * S::BLK;
    const bool per_head = (flags & kFlagPerHead) != 0;
    float pmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float x = l[j] * p.qscale;
      if (i8) x *= t2_scale(sc, per_head, rows[j]);
      if (!((mask >> rows[j]) & 1u)) x = -INFINITY;
      l[j] = x;
      pmax = fmaxf(pmax, x);
    }
    pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 1));
    pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 2));
    const float m_new = fmaxf(m_run, pmax);
    float corr = 1.f, psum = 0.f, pr[4];
    if (m_new != -INFINITY) {
      corr = exp2f(m_run - m_new);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pr[j] = exp2f(l[j] - m_new);
        psum += pr[j];
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) pr[j] = 0.f;
    }
    psum += __shfl_xor_sync(kFull, psum, 1);
    psum += __shfl_xor_sync(kFull, psum, 2);
    z_run = z_run * corr + psum;
    m_run = m_new;
    if (g < G) {
      float* sp = spill_b + (static_cast<int64_t>(k) * G + g) * kPage;
      *reinterpret_cast<float2*>(sp + 2 * t) = make_float2(l[0], l[1]);
      *reinterpret_cast<float2*>(sp + 8 + 2 * t) = make_float2(l[2], l[3]);
    }
    if (i8) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        pr[j] = ((mask >> rows[j]) & 1u) ? pr[j] * t2_scale(sc, per_head, kPage + rows[j]) : 0.f;
    }
    const uint32_t pb0 = pack_bf16(pr[0], pr[1]), pb1 = pack_bf16(pr[2], pr[3]);

    // ---- rescale O^T columns (heads 2t, 2t+1) by their correction -------------
    const float ca = __shfl_sync(kFull, corr, 8 * t);
    const float cb = __shfl_sync(kFull, corr, 8 * t + 4);
    if (__any_sync(kFull, ca != 1.f || cb != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= ca;
        o[mt][1] *= cb;
        o[mt][2] *= ca;
        o[mt][3] *= cb;
      }
    }
    // holes may hold anything: a weight of 0 must not meet a NaN, so the V rows
    // of empty slots are zeroed in shared memory (partial pages only)
    if (mask != 0xffffu && !i8) {
      for (int e = lane; e < kPage * (S::ROWB / 16); e += 32) {
        const int r = e / (S::ROWB / 16);
        if (!((mask >> r) & 1u))
          *reinterpret_cast<uint4*>(stage + S::BLK + r * S::ROWB + (e % (S::ROWB / 16)) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    // ---- O^T += V^T P^T ----------------------------------------------------------
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vbase + lrow * S::ROWB + swz_chunk(2 * mt + lchunk, lrow, swz) * 16, a0, a1, a2, a3);
      mma_bf16(o[mt], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    if (lane == 0) {
      // the stage was written through the generic proxy (widened codes, zeroed
      // rows): order those writes before the next bulk copy into it
      if (i8 || host || mask != 0xffffu) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(empty0 + st * 8);
    }
  }

  __syncthreads();
  if (s_abort) {  // a bounded wait gave up: land the copies in flight; the unit's partial stays unwritten
    if (!consumer && lane == 0) {
      drain(issued, full0, p.wait_limit_ns);
      atomicExch(p.err, DEV_TIMEOUT);
    }
  }
  __syncthreads();
  // items left over once the units ran out (the ring is idle again)
  prev_launch_epilogue<T, G, D>(p, tid, s_epM, s_epIZ, reinterpret_cast<float*>(smem), &s_item);
  if (tid == 0 && p.span) atomicMax(p.span + 1, global_ns());
}

// ===================================================================== FP32
// Loads the lane's QE elements of one row of a full-precision page as pairs.
template <typename T, int G, int D>
__device__ __forceinline__ void load_row_qk(const char* rowp, int row, int c, int swz,
                                            float2 (&out)[Shape<T, G, D>::QP]) {
  using S = Shape<T, G, D>;
#pragma unroll
  for (int j = 0; j < S::CPL; ++j) {
    const char* cp = rowp + swz_chunk(c + 8 * j, row, swz) * 16;
    if constexpr (sizeof(T) == 2) {
      const uint4 w = *reinterpret_cast<const uint4*>(cp);
      out[j * 4 + 0] = make_float2(bf_lo(w.x), bf_hi(w.x));
      out[j * 4 + 1] = make_float2(bf_lo(w.y), bf_hi(w.y));
      out[j * 4 + 2] = make_float2(bf_lo(w.z), bf_hi(w.z));
      out[j * 4 + 3] = make_float2(bf_lo(w.w), bf_hi(w.w));
    } else {
      const float4 f = *reinterpret_cast<const float4*>(cp);
      out[j * 2 + 0] = make_float2(f.x, f.y);
      out[j * 2 + 1] = make_float2(f.z, f.w);
    }
  }
}

// The same elements of one row of an 8-bit page (codes as floats, unswizzled).
template <typename T, int G, int D>
__device__ __forceinline__ void load_row_qk_i8(const char* rowp, int c, float2 (&out)[Shape<T, G, D>::QP]) {
  using S = Shape<T, G, D>;
#pragma unroll
  for (int j = 0; j < S::CPL; ++j) {
    const char* cp = rowp + (c + 8 * j) * S::EPC;
    if constexpr (S::EPC == 8) {
      const uint2 w = *reinterpret_cast<const uint2*>(cp);
      out[j * 4 + 0] = make_float2(i8f(w.x, 0), i8f(w.x, 1));
      out[j * 4 + 1] = make_float2(i8f(w.x, 2), i8f(w.x, 3));
      out[j * 4 + 2] = make_float2(i8f(w.y, 0), i8f(w.y, 1));
      out[j * 4 + 3] = make_float2(i8f(w.y, 2), i8f(w.y, 3));
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(cp);
      out[j * 2 + 0] = make_float2(i8f(w, 0), i8f(w, 1));
      out[j * 2 + 1] = make_float2(i8f(w, 2), i8f(w, 3));
    }
  }
}

// The lane's VPL elements of one V row (full precision, swizzled, or 8-bit codes).
template <typename T, int D, bool I8>
__device__ __forceinline__ void load_row_pv(const char* rowp, int row, int lane, int swz, float (&v)[D / 32]) {
  constexpr int VPL = D / 32;
  if constexpr (I8) {
    if constexpr (VPL == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(rowp + lane * 4);
      v[0] = i8f(w, 0); v[1] = i8f(w, 1); v[2] = i8f(w, 2); v[3] = i8f(w, 3);
    } else {
      const uint32_t w = *reinterpret_cast<const uint16_t*>(rowp + lane * 2);
      v[0] = i8f(w, 0); v[1] = i8f(w, 1);
    }
  } else {
    const int byte = lane * VPL * static_cast<int>(sizeof(T));
    const char* ep = rowp + swz_chunk(byte >> 4, row, swz) * 16 + (byte & 15);
    if constexpr (sizeof(T) == 2) {
      if constexpr (VPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(ep);
        v[0] = bf_lo(w.x); v[1] = bf_hi(w.x); v[2] = bf_lo(w.y); v[3] = bf_hi(w.y);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(ep);
        v[0] = bf_lo(w); v[1] = bf_hi(w);
      }
    } else {
      if constexpr (VPL == 4) {
        const float4 f = *reinterpret_cast<const float4*>(ep);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
      } else {
        const float2 f = *reinterpret_cast<const float2*>(ep);
        v[0] = f.x; v[1] = f.y;
      }
    }
  }
}

template <typename T, int G, int D>
__global__ void __launch_bounds__((kAttnWarps + 1) * 32)
    attn_split_fma_kernel(const __grid_constant__ AttnParams p) {
  using S = Shape<T, G, D>;
  using L = Smem<T, G, D, true>;
  extern __shared__ __align__(128) char smem[];
  __shared__ volatile int s_abort;
  __shared__ float s_epM[8], s_epIZ[8];  // previous layer's (M, 1 / Z) per head
  __shared__ volatile int s_item;
  __shared__ int s_first;

  const int tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31;
  const int r = lane >> 3, c = lane & 7;
  if (tid == 0) s_abort = 0;
  if (tid == 0 && p.span) atomicMin(p.span, global_ns());
  if (tid == 0 && blockIdx.x == 0) {
    if (p.span_next) {
      p.span_next[0] = ~0ull;
      p.span_next[1] = 0ull;
    }
    if (p.ep_clear) {  // counters of the launch after next
      for (int z = 0; z < kMaxLaunchLayers; ++z) p.ep_clear->claim[z] = 0;
      p.ep_clear->units = 0;
    }
    if (p.started) {                  // tells the copy stream this launch is under way
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.started), "r"(p.launch_seq) : "memory");
    }
  }
  init_barriers<L>(smem);
  __syncthreads();
  // the first ep_first_ctas CTAs take epilogue items of the previous launch
  // before any unit (the ring is still idle), while the others start streaming
  if (static_cast<int>(blockIdx.x) < p.ep_first_ctas) {
    prev_launch_epilogue<T, G, D>(p, tid, s_epM, s_epIZ, reinterpret_cast<float*>(smem), &s_item);
    // the items wrote the ring's first stage through the generic proxy: order
    // those writes before the bulk copies that will fill it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (tid == 0) s_first = first_unit(p);
  __syncthreads();
  const int first = s_first;

  int32_t* meta_k = reinterpret_cast<int32_t*>(smem + L::off_pg);
  uint32_t* meta_f = reinterpret_cast<uint32_t*>(meta_k + kMeta);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bar);
  char* ring = smem;
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + kAttnStages * 8;
  const uint32_t merge_bar = full0 + 2 * kAttnStages * 8;
  const bool consumer = w < kAttnWarps;
  int issued = 0;
  if (!consumer)
    issued = produce<S>(p, first, meta_k, meta_f, reinterpret_cast<PageCopy*>(smem + L::off_desc), ring, full0,
                        empty0, &s_abort);

  float* q_s = reinterpret_cast<float*>(smem + L::off_q);
  float* p_s = reinterpret_cast<float*>(smem + L::off_p) + w * L::PSW;
  float* corr_s = p_s + S::GP * kPage;
  const int units = launch_units(p);
  int u = first;
  Work wk{};
  float* spill_b = nullptr;
  // the unit's scaled query (shared by the consumer warps) and logit spill
  auto start_unit = [&]() {
    wk = unit_work(p, u);
    const T* q = reinterpret_cast<const T*>(p.q) + wk.z * p.q_stride_l + static_cast<int64_t>(wk.b) * p.q_stride_b +
                 static_cast<int64_t>(wk.kvh) * G * D;
    for (int i = tid; i < S::GP * D; i += kAttnWarps * 32) {
      const int gg = i / D;
      float v = 0.f;
      if (gg < G) {
        if constexpr (sizeof(T) == 2)
          v = __bfloat162float(q[i]);
        else
          v = static_cast<float>(q[i]);
      }
      q_s[i] = v * p.qscale;
    }
    spill_b = spill_of(p, p.spill, wk);
  };
  if (consumer && u < units) start_unit();
  if (consumer) consumer_sync();
  uint32_t mphase = 0;                   // merge-barrier phases completed

  float m_run = -INFINITY, z_run = 0.f;  // for the head this lane owns
  float2 acc[G][S::VPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < S::VPL; ++e) acc[g][e] = make_float2(0.f, 0.f);

  // Which (head, row) logits this lane owns after the butterfly.
  const int own_g = S::NV >= 8 ? (c * S::NL) >> 2 : 0;
  const bool own_writer = S::NV >= 8 ? true : ((c & 1) == 0);
  const bool head_lead = r == 0 && (S::NV < 8 ? c == 0 : (c & ((8 / S::GP) - 1)) == 0);

  for (int i = w; consumer && u < units; i += kAttnWarps) {
    const int st = i % kAttnStages;
    const bool ok = __all_sync(kFull, mbar_wait(full0 + st * 8, (i / kAttnStages) & 1, p.wait_limit_ns));
    if (!ok) {
      if (lane == 0) s_abort = 1;
      break;
    }
    const int k = meta_k[i % kMeta];  // page index in the sequence's list, or a pad or unit-end record
    if (k == kMetaPad) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + st * 8);
      continue;
    }
    if (k < 0) {
      // ---- unit end: this warp's (O, m, Z) into its marker's stage, then merge
      const int first = static_cast<int>(meta_f[i % kMeta]);
      float* mo = reinterpret_cast<float*>(ring + st * S::STAGE);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < S::VPL; ++e) mo[g * D + lane * S::VPL + e] = acc[g][e].x + acc[g][e].y;
      if (own_writer && own_g < G && head_lead) {
        mo[G * D + own_g] = m_run;
        mo[G * D + S::GP + own_g] = z_run;
      }
      if (!consumers_meet(merge_bar, mphase, lane, p.wait_limit_ns)) {
        if (lane == 0) s_abort = 1;
        break;
      }
      merge_partial<T, G, D>(p, wk, ring, first, tid);
      if (!consumers_meet(merge_bar, mphase, lane, p.wait_limit_ns)) {  // every warp has read every stage
        if (lane == 0) s_abort = 1;
        break;
      }
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes before the next copy
        mbar_arrive(empty0 + st * 8);
      }
      if (k == kMetaLast) break;  // the producer claimed no further unit
      u = marker_next(k);
      start_unit();
      if (!consumers_meet(merge_bar, mphase, lane, p.wait_limit_ns)) {  // the new query is in place
        if (lane == 0) s_abort = 1;
        break;
      }
      m_run = -INFINITY;
      z_run = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < S::VPL; ++e) acc[g][e] = make_float2(0.f, 0.f);
      continue;
    }
    const uint32_t flags = meta_f[i % kMeta];
    const uint32_t mask = flags & 0xffffu;
    const bool i8 = (flags & kFlagI8) != 0;
    const bool per_head = (flags & kFlagPerHead) != 0;
    const bool host = (flags & kFlagHost) != 0;
    const int swz = static_cast<int>((flags >> kFlagSwzShift) & 7u);
    const char* stage = ring + st * S::STAGE;

    // ---- QK: 4 rows per lane, QE elements each, all heads -----------------
    float part[S::NV];
    {
      float2 kf[4][S::QP];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int row = r + 4 * ii;
        if (i8)
          load_row_qk_i8<T, G, D>(stage + row * D, c, kf[ii]);
        else
          load_row_qk<T, G, D>(stage + row * S::ROWB, row, c, swz, kf[ii]);
      }
#pragma unroll
      for (int g = 0; g < S::GP; ++g) {
        if (g < G) {
          float2 qv[S::QP];
#pragma unroll
          for (int j = 0; j < S::CPL; ++j) {
            const float* qp = q_s + g * D + (c + 8 * j) * S::EPC;
#pragma unroll
            for (int e4 = 0; e4 < S::EPC / 4; ++e4) {
              const float4 f = *reinterpret_cast<const float4*>(qp + 4 * e4);
              qv[j * (S::EPC / 2) + 2 * e4] = make_float2(f.x, f.y);
              qv[j * (S::EPC / 2) + 2 * e4 + 1] = make_float2(f.z, f.w);
            }
          }
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < S::QP; ++e) a = ffma2(qv[e], kf[ii][e], a);
            part[g * 4 + ii] = a.x + a.y;
          }
        } else {
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) part[g * 4 + ii] = 0.f;
        }
      }
    }
    // ---- transposing butterfly over the 8 lanes c --------------------------
    {
      int size = S::NV;
#pragma unroll
      for (int m = 4; m >= 1; m >>= 1) {
        const bool up = (lane & m) != 0;
        if (size >= 2) {
          const int half = size >> 1;
#pragma unroll
          for (int tt = 0; tt < S::NV / 2; ++tt) {
            if (tt < half) {
              const float send = up ? part[tt] : part[tt + half];
              const float keep = up ? part[tt + half] : part[tt];
              part[tt] = keep + __shfl_xor_sync(kFull, send, m);
            }
          }
          size = half;
        } else {
          part[0] += __shfl_xor_sync(kFull, part[0], m);
        }
      }
    }
    // part[0 .. NL) are this lane's logits: head own_g, rows r + 4 * (idx & 3).
    float lg[S::NL], pv[S::NL];
    float pmax = -INFINITY;
    const char* sc = stage + 2 * S::BLK;
#pragma unroll
    for (int tt = 0; tt < S::NL; ++tt) {
      const int idx = S::NV >= 8 ? c * S::NL + tt : (c >> 1);
      const int row = r + 4 * (idx & 3);
      float x = part[tt];
      if (i8) x *= t2_scale(sc, per_head, row);
      if (!((mask >> row) & 1u)) x = -INFINITY;
      lg[tt] = x;
      pmax = fmaxf(pmax, x);
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1)
      if (m < 8 / S::GP) pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, m));
    pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 8));
    pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 16));
    const float m_new = fmaxf(m_run, pmax);
    float corr = 1.f, psum = 0.f;
    if (m_new != -INFINITY) {
      corr = exp2f(m_run - m_new);
#pragma unroll
      for (int tt = 0; tt < S::NL; ++tt) {
        pv[tt] = exp2f(lg[tt] - m_new);
        psum += pv[tt];
      }
    } else {
#pragma unroll
      for (int tt = 0; tt < S::NL; ++tt) pv[tt] = 0.f;
    }
    // with one head, lanes c and c ^ 1 hold the same logits: sum each row once
#pragma unroll
    for (int m = 1; m < 8; m <<= 1)
      if (m < 8 / S::GP && !(S::NV < 8 && m == 1)) psum += __shfl_xor_sync(kFull, psum, m);
    psum += __shfl_xor_sync(kFull, psum, 8);
    psum += __shfl_xor_sync(kFull, psum, 16);
    z_run = z_run * corr + psum;
    m_run = m_new;

    // spill raw logits, publish p (times the V scale for 8-bit rows) and corr
    if (own_writer && own_g < G) {
#pragma unroll
      for (int tt = 0; tt < S::NL; ++tt) {
        const int idx = S::NV >= 8 ? c * S::NL + tt : (c >> 1);
        const int row = r + 4 * (idx & 3);
        spill_b[(static_cast<int64_t>(k) * G + own_g) * kPage + row] = lg[tt];
        float pw = pv[tt];
        if (i8) pw = ((mask >> row) & 1u) ? pw * t2_scale(sc, per_head, kPage + row) : 0.f;
        p_s[own_g * kPage + row] = pw;
      }
      if (head_lead) corr_s[own_g] = corr;
    }
    __syncwarp();

    // ---- PV ---------------------------------------------------------------
    {
      const bool rescale = __any_sync(kFull, own_g < G && corr != 1.f);
      if (rescale) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float cg = corr_s[g];
#pragma unroll
          for (int e = 0; e < S::VPL; ++e) {
            acc[g][e].x *= cg;
            acc[g][e].y *= cg;
          }
        }
      }
      const char* vblk = stage + (i8 ? kPage * D : S::BLK);
      const int vrow = i8 ? D : S::ROWB;
      const bool partial = mask != 0xffffu && !i8;
#pragma unroll 2
      for (int j = 0; j < kPage / 2; ++j) {
        float va[S::VPL], vb[S::VPL];
        if (i8) {
          load_row_pv<T, D, true>(vblk + (2 * j) * vrow, 2 * j, lane, 0, va);
          load_row_pv<T, D, true>(vblk + (2 * j + 1) * vrow, 2 * j + 1, lane, 0, vb);
        } else {
          load_row_pv<T, D, false>(vblk + (2 * j) * vrow, 2 * j, lane, swz, va);
          load_row_pv<T, D, false>(vblk + (2 * j + 1) * vrow, 2 * j + 1, lane, swz, vb);
        }
        if (partial) {  // holes may hold anything: weight 0 must not meet a NaN
          const bool oka = (mask >> (2 * j)) & 1u, okb = (mask >> (2 * j + 1)) & 1u;
#pragma unroll
          for (int e = 0; e < S::VPL; ++e) {
            va[e] = oka ? va[e] : 0.f;
            vb[e] = okb ? vb[e] : 0.f;
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 pp = *reinterpret_cast<const float2*>(p_s + g * kPage + 2 * j);
#pragma unroll
          for (int e = 0; e < S::VPL; ++e) acc[g][e] = ffma2(pp, make_float2(va[e], vb[e]), acc[g][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      // a page read in place was written to the stage through the generic proxy:
      // order those writes before the next bulk copy into it
      if (host) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(empty0 + st * 8);
    }
  }

  __syncthreads();
  if (s_abort) {  // a bounded wait gave up: land the copies in flight; the unit's partial stays unwritten
    if (!consumer && lane == 0) {
      drain(issued, full0, p.wait_limit_ns);
      atomicExch(p.err, DEV_TIMEOUT);
    }
  }
  __syncthreads();
  // items left over once the units ran out (the ring is idle again)
  prev_launch_epilogue<T, G, D>(p, tid, s_epM, s_epIZ, reinterpret_cast<float*>(smem), &s_item);
  if (tid == 0 && p.span) atomicMax(p.span + 1, global_ns());
}

// Persistent launch: as many CTAs as fit on the device at once (found once per
// kernel and device), at most one per work unit; each CTA claims its units one
// at a time from the launch's counter (first_unit, claim_next_unit).
template <typename K>
cudaError_t launch_kernel(K kern, int smem_bytes, const AttnParams& p, int total_chunks, cudaStream_t s,
                          int (&resident)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident[dev] == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, (kAttnWarps + 1) * 32, smem_bytes);
    if (e != cudaSuccess) return e;
    resident[dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  const int64_t units = static_cast<int64_t>(total_chunks) * p.Hkv * p.nlayers;
  const unsigned grid = static_cast<unsigned>(units < resident[dev] ? units : resident[dev]);
  kern<<<grid, (kAttnWarps + 1) * 32, smem_bytes, s>>>(p);
  return cudaGetLastError();
}

// part 0: the page-streaming kernel; part 1: the combine / score kernel
template <typename T, int G, int D>
cudaError_t launch_typed(const AttnParams& p, int total_chunks, cudaStream_t s, int part) {
  constexpr bool kMma = sizeof(T) == 2 && G >= 2;
  using L = Smem<T, G, D, !kMma>;
  if (part == 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(total_chunks, p.Hkv, p.nlayers);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel<T, G, D>, p);
  }
  if constexpr (sizeof(T) == 2 && G >= 2) {
    static int resident[64] = {};
    return launch_kernel(attn_split_mma_kernel<G, D>, L::TOTAL, p, total_chunks, s, resident);
  } else {
    static int resident[64] = {};
    return launch_kernel(attn_split_fma_kernel<T, G, D>, L::TOTAL, p, total_chunks, s, resident);
  }
}

template <typename T, int G, int D>
int resident_typed() {
  constexpr bool kMma = sizeof(T) == 2 && G >= 2;
  using L = Smem<T, G, D, !kMma>;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 304;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 304;
  cudaError_t e;
  if constexpr (sizeof(T) == 2 && G >= 2) {
    cudaFuncSetAttribute(attn_split_mma_kernel<G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_mma_kernel<G, D>, (kAttnWarps + 1) * 32, L::TOTAL);
  } else {
    cudaFuncSetAttribute(attn_split_fma_kernel<T, G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_fma_kernel<T, G, D>, (kAttnWarps + 1) * 32, L::TOTAL);
  }
  (void)cudaGetLastError();
  if (e != cudaSuccess || per_sm < 1) return 2 * sms;
  return sms * per_sm;
}

template <typename T>
int resident_g(int G, int D) {
#define TKV_CASE(GG, DD) \
  if (G == GG && D == DD) return resident_typed<T, GG, DD>();
  TKV_CASE(1, 64) TKV_CASE(1, 128)
  TKV_CASE(2, 64) TKV_CASE(2, 128)
  TKV_CASE(4, 64) TKV_CASE(4, 128)
  TKV_CASE(7, 64) TKV_CASE(7, 128)
  TKV_CASE(8, 64) TKV_CASE(8, 128)
#undef TKV_CASE
  return 304;
}

template <typename T>
cudaError_t dispatch_g(const AttnParams& p, int total_chunks, cudaStream_t s, int part) {
  const int G = p.G, D = p.D;
#define TKV_CASE(GG, DD) \
  if (G == GG && D == DD) return launch_typed<T, GG, DD>(p, total_chunks, s, part);
  TKV_CASE(1, 64) TKV_CASE(1, 128)
  TKV_CASE(2, 64) TKV_CASE(2, 128)
  TKV_CASE(4, 64) TKV_CASE(4, 128)
  TKV_CASE(7, 64) TKV_CASE(7, 128)
  TKV_CASE(8, 64) TKV_CASE(8, 128)
#undef TKV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

int resident_attention_ctas(int kv_dtype, int G, int D) {
  if (kv_dtype == 1) return resident_g<__nv_bfloat16>(G, D);
  return resident_g<float>(G, D);
}

int attention_supported(int kv_dtype, int G, int D) {
  (void)kv_dtype;
  const bool g_ok = G == 1 || G == 2 || G == 4 || G == 7 || G == 8;
  return g_ok && (D == 64 || D == 128);
}

cudaError_t launch_attention_part(const AttnParams& p, int kv_dtype, int total_chunks, cudaStream_t s, int part) {
  if (total_chunks <= 0 || p.nlayers <= 0) return cudaSuccess;
  if (total_chunks != p.total_chunks || p.nlayers > 65535) return cudaErrorInvalidValue;
  if (kv_dtype == 1) return dispatch_g<__nv_bfloat16>(p, total_chunks, s, part);
  return dispatch_g<float>(p, total_chunks, s, part);
}

cudaError_t launch_attention(const AttnParams& p, int kv_dtype, int total_chunks, cudaStream_t s) {
  cudaError_t e = launch_attention_part(p, kv_dtype, total_chunks, s, 0);
  if (e != cudaSuccess) return e;
  return launch_attention_part(p, kv_dtype, total_chunks, s, 1);
}

}  // namespace tkv
