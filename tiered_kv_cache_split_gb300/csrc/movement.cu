// Data movement of the four-tier cache ("Not All Thoughts Need HBM",
// Methodology 1 and 4): appending the decoded token to T0, moving tokens whose
// tier changed between the T0 pool (HBM) and the T1/T2 pools (pinned host
// memory, reached through device-mapped pointers over the host link),
// 8-bit quantisation into T2 and dequantisation out of it, and folding each
// step's score increments into the float64 scores.
//
// T2 quantisation (the page names 8 bits, not the scheme; read here as
// symmetric absmax): scale = absmax / 127 in IEEE float32 division (then
// rounded to float16 when stored so), code = clamp(rint(x / scale), -127, 127)
// with float32 division and round-half-even; an all-zero row has scale 0 and
// codes 0. A token leaving T2 carries storage(float32(code * scale)).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tkv_internal.h"

namespace tkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float load_elem(const char* p, int kv_dtype) {
  if (kv_dtype == 1) return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
  return *reinterpret_cast<const float*>(p);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}

// Scale and divisor of one row: scale = absmax / 127 (float32, then float16
// if stored so); the divisor is the stored scale as float32.
__device__ __forceinline__ float quant_scale(float absmax, int scale_f16, __half* h) {
  const float s32 = __fdiv_rn(absmax, 127.0f);
  if (scale_f16) {
    *h = __float2half_rn(s32);
    return __half2float(*h);
  }
  return s32;
}

__device__ __forceinline__ int8_t quant_code(float x, float divisor) {
  if (!(divisor > 0.f)) return 0;
  float q = rintf(__fdiv_rn(x, divisor));
  q = fminf(fmaxf(q, -127.f), 127.f);
  return static_cast<int8_t>(static_cast<int>(q));
}

// ---------------------------------------------------------------- append
// One block per (sequence, layer): the new token's K and V rows go to its T0
// slot (full-precision rows are stored swizzled: 16-byte chunk c of row r at
// chunk c ^ (r & 7)). Block (b, 0) also updates the page metadata, inserting a
// new page at its sorted place in the sequence's T0 page list.
__global__ void append_kernel(const __grid_constant__ AppendParams p) {
  const int b = blockIdx.x, l = blockIdx.y;
  const int page = p.page[b], slot = p.slot[b];
  // debug build: a page outside the pool or a page list that would outgrow its row skips the block
  if (!index_ok(p.err, DBG_APPEND_PAGE, page, p.cap0) ||
      (p.new_page[b] && !index_ok(p.err, DBG_APPEND_LIST, p.np0[b], p.table_stride)))
    return;
  const int row_bytes = p.D * p.esz;
  const int vec_per_row = row_bytes / 16;
  const int total = p.Hkv * 2 * vec_per_row;
  char* dst_page = p.pool0 + l * p.layer_bytes + static_cast<int64_t>(page) * p.page_bytes;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int v = i % vec_per_row;
    const int hk = i / vec_per_row;  // head * 2 + kv
    const int h = hk >> 1, kv = hk & 1;
    const char* src = (kv ? p.v : p.k) +
                      ((static_cast<int64_t>(b) * p.L + l) * p.Hkv + h) * row_bytes + v * 16;
    char* dst = dst_page + (static_cast<int64_t>(h) * 2 + kv) * kPage * row_bytes +
                static_cast<int64_t>(slot) * row_bytes + swz_offset(slot, v * 16, kSwizzle);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
  if (l != 0) return;
  if (p.new_page[b]) {
    int32_t* row = p.table0 + static_cast<int64_t>(b) * p.table_stride;
    const int lo = p.insert_at[b], np0 = p.np0[b];
    // shift entries [lo, np0) one place right, highest first, a block-width at a time
    for (int base = np0 - 1; base >= lo; base -= blockDim.x) {
      const int i = base - static_cast<int>(threadIdx.x);
      int32_t v = 0;
      if (i >= lo) v = row[i];
      __syncthreads();
      if (i >= lo) row[i + 1] = v;
      __syncthreads();
    }
    if (threadIdx.x == 0) row[lo] = page;
  }
  if (threadIdx.x == 0) {
    atomicOr(p.mask0 + page, 1u << slot);
    p.posmap0[static_cast<int64_t>(page) * kPage + slot] = static_cast<int32_t>(p.pos[b]);
  }
}

// ---------------------------------------------------------------- prefill
__global__ void prefill_kernel(const __grid_constant__ PrefillParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
  const int l = blockIdx.y;
  if (t >= p.n) return;
  const int loc = p.loc[t];
  const int page = loc >> 4, slot = loc & 15;
  if (!index_ok(p.err, DBG_PREFILL_PAGE, page, p.cap0)) return;  // debug build only
  const int row_bytes = p.D * p.esz;
  const int vec_per_row = row_bytes / 16;
  const int total = p.Hkv * 2 * vec_per_row;
  char* dst_page = p.pool0 + l * p.layer_bytes + static_cast<int64_t>(page) * p.page_bytes;
  for (int i = lane; i < total; i += 32) {
    const int v = i % vec_per_row;
    const int hk = i / vec_per_row;
    const int h = hk >> 1, kv = hk & 1;
    const char* src = (kv ? p.v : p.k) + ((static_cast<int64_t>(l) * p.n + t) * p.Hkv + h) * row_bytes + v * 16;
    char* dst = dst_page + (static_cast<int64_t>(h) * 2 + kv) * kPage * row_bytes +
                static_cast<int64_t>(slot) * row_bytes + swz_offset(slot, v * 16, kSwizzle);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

// ---------------------------------------------------------------- movers
// One block per (mover, layer) moves the token's K and V rows of every KV head.
// Full-precision rows move as 16-byte chunks: the swizzle only permutes the
// chunks of a row, so a chunk keeps its place in the row's logical order and
// is read and written whole (T1 and T2 pools are host memory reached over the
// host link, where wide accesses matter most). Rows that leave T2 are
// dequantised chunk by chunk; rows that enter T2 pass through shared memory as
// float32 for the absmax of their scale group.
constexpr int kMoveThreads = 128;

// Full-precision chunk c of row hk (= head * 2 + kv) of a location: a pool slot
// (tier 0 or 1), or a staging row of `temp` (one layer, plain layout [rows][2][Hkv][D]).
__device__ __forceinline__ char* full_chunk(const MoveParams& p, int tier, int loc, int temp_row, int l,
                                           int hk, int c, int64_t row_bytes) {
  if (tier < 0) {
    const int h = hk >> 1, kv = hk & 1;
    return p.temp + ((static_cast<int64_t>(temp_row) * 2 + kv) * p.Hkv + h) * row_bytes + c * 16;
  }
  const int page = loc >> 4, slot = loc & 15;
  const TierPools& P = p.pools;
  char* pg = P.base[tier] + l * P.layer_bytes[tier] + static_cast<int64_t>(page) * P.page_bytes[tier];
  return pg + (static_cast<int64_t>(hk) * kPage + slot) * row_bytes + ((c ^ (slot & kSwizzle)) << 4);
}

// The same chunk in a tier's device mirror (null when the tier has none).
__device__ __forceinline__ char* mirror_chunk(const MoveParams& p, int tier, int loc, int l, int hk, int c,
                                             int64_t row_bytes) {
  if (tier < 1 || p.pools.mirror[tier] == nullptr) return nullptr;
  const int page = loc >> 4, slot = loc & 15;
  const TierPools& P = p.pools;
  char* pg = P.mirror[tier] + l * P.layer_bytes[tier] + static_cast<int64_t>(page) * P.page_bytes[tier];
  return pg + (static_cast<int64_t>(hk) * kPage + slot) * row_bytes + ((c ^ (slot & kSwizzle)) << 4);
}

__device__ __forceinline__ float t2_scale_of(const TierPools& P, const char* sc, int hk, int slot) {
  const int kv = hk & 1;
  if (P.scale_per_head) {
    if (P.scale_f16) return __half2float(reinterpret_cast<const __half*>(sc)[hk * kPage + slot]);
    return reinterpret_cast<const float*>(sc)[hk * kPage + slot];
  }
  return reinterpret_cast<const float*>(sc)[kv * kPage + slot];
}

__global__ void __launch_bounds__(kMoveThreads) move_kernel(const __grid_constant__ MoveParams p,
                                                            const Mover* __restrict__ movers) {
  extern __shared__ float row_s[];  // [2][Hkv][D] float32 (rows entering T2)
  const Mover mv = movers[blockIdx.x];
  const int l = p.layer0 + blockIdx.y;
  const int tid = threadIdx.x;
  const int esz = p.kv_dtype == 1 ? 2 : 4;
  const int64_t row_bytes = static_cast<int64_t>(p.D) * esz;
  const int cpr = static_cast<int>(row_bytes / 16);  // 16-byte chunks per full-precision row
  const int epc = 16 / esz;                          // elements per chunk
  const int nchunk = 2 * p.Hkv * cpr;
  const TierPools& P = p.pools;
  const int st = p.mode == MOVE_SCATTER ? -1 : mv.src_tier;  // -1: the staging rows
  const int dt = p.mode == MOVE_GATHER ? -1 : mv.dst_tier;

  // staging row of this (mover, layer): one per mover when the launch covers one
  // layer, one per (mover, layer) when it covers several
  const int trow = mv.temp_row * static_cast<int>(gridDim.y) + static_cast<int>(blockIdx.y);
  // debug build: the mover's pages and staging row against their areas (skips the block)
  if (!(st < 0 || index_ok(p.err, DBG_MOVE_SRC, mv.src_loc >> 4, P.cap[st])) ||
      !(dt < 0 || index_ok(p.err, DBG_MOVE_DST, mv.dst_loc >> 4, P.cap[dt])) ||
      !((st >= 0 && dt >= 0) || index_ok(p.err, DBG_MOVE_TEMP, trow, p.temp_rows)))
    return;
  // With a device mirror of T1 / T2, sources there are read from the mirror (no
  // host-link read) and destinations there are written to the pool and the mirror.
  const bool src_mirror = st >= 1 && P.mirror[st] != nullptr;
  if (st != 2 && dt != 2) {  // full precision -> full precision
    for (int j = tid; j < nchunk; j += kMoveThreads) {
      const int hk = j / cpr, c = j % cpr;
      const char* from = src_mirror ? mirror_chunk(p, st, mv.src_loc, l, hk, c, row_bytes)
                                    : full_chunk(p, st, mv.src_loc, trow, l, hk, c, row_bytes);
      const uint4 v = *reinterpret_cast<const uint4*>(from);
      *reinterpret_cast<uint4*>(full_chunk(p, dt, mv.dst_loc, trow, l, hk, c, row_bytes)) = v;
      if (char* m = mirror_chunk(p, dt, mv.dst_loc, l, hk, c, row_bytes)) *reinterpret_cast<uint4*>(m) = v;
    }
    return;
  }

  if (st == 2) {  // leaving T2: dequantise to the destination's storage, chunk by chunk
    const int page = mv.src_loc >> 4, slot = mv.src_loc & 15;
    const char* pg = (src_mirror ? P.mirror[2] : P.base[2]) + l * P.layer_bytes[2] +
                     static_cast<int64_t>(page) * P.page_bytes[2];
    const char* sc = (src_mirror ? P.mirror_scales : P.t2_scales) + l * P.t2_scale_layer_bytes +
                     static_cast<int64_t>(page) * P.t2_scale_page_bytes;
    for (int j = tid; j < nchunk; j += kMoveThreads) {
      const int hk = j / cpr, c = j % cpr;
      const float scale = t2_scale_of(P, sc, hk, slot);
      const int8_t* codes = reinterpret_cast<const int8_t*>(pg + (static_cast<int64_t>(hk) * kPage + slot) * p.D + c * epc);
      uint4 out;
      if (esz == 2) {
        const uint2 w = *reinterpret_cast<const uint2*>(codes);
        uint32_t r[4];
        const uint32_t words[2] = {w.x, w.y};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t word = words[q >> 1];
          const int b0 = 2 * (q & 1);
          const float x0 = __fmul_rn(static_cast<float>(static_cast<int8_t>((word >> (8 * b0)) & 0xffu)), scale);
          const float x1 = __fmul_rn(static_cast<float>(static_cast<int8_t>((word >> (8 * b0 + 8)) & 0xffu)), scale);
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(x0, x1);
          r[q] = *reinterpret_cast<const uint32_t*>(&v2);
        }
        out = make_uint4(r[0], r[1], r[2], r[3]);
      } else {
        const uint32_t word = *reinterpret_cast<const uint32_t*>(codes);
        float f[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          f[q] = __fmul_rn(static_cast<float>(static_cast<int8_t>((word >> (8 * q)) & 0xffu)), scale);
        out = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
      }
      *reinterpret_cast<uint4*>(full_chunk(p, dt, mv.dst_loc, trow, l, hk, c, row_bytes)) = out;
      if (char* m = mirror_chunk(p, dt, mv.dst_loc, l, hk, c, row_bytes)) *reinterpret_cast<uint4*>(m) = out;
    }
    return;
  }

  // entering T2: stage the rows as float32, one scale per group, 16 codes per store
  const int HD = p.Hkv * p.D;
  for (int j = tid; j < nchunk; j += kMoveThreads) {
    const int hk = j / cpr, c = j % cpr;
    const int h = hk >> 1, kv = hk & 1;
    const char* from = src_mirror ? mirror_chunk(p, st, mv.src_loc, l, hk, c, row_bytes)
                                  : full_chunk(p, st, mv.src_loc, trow, l, hk, c, row_bytes);
    const uint4 v = *reinterpret_cast<const uint4*>(from);
    float* dst = row_s + kv * HD + h * p.D + c * epc;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (esz == 2) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dst[2 * q] = __uint_as_float(w[q] << 16);
        dst[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = __uint_as_float(w[q]);
    }
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  const int page = mv.dst_loc >> 4, slot = mv.dst_loc & 15;
  char* pg = P.base[2] + l * P.layer_bytes[2] + static_cast<int64_t>(page) * P.page_bytes[2];
  char* sc = P.t2_scales + l * P.t2_scale_layer_bytes + static_cast<int64_t>(page) * P.t2_scale_page_bytes;
  char* mpg = P.mirror[2] ? P.mirror[2] + l * P.layer_bytes[2] + static_cast<int64_t>(page) * P.page_bytes[2] : nullptr;
  char* msc = P.mirror[2] ? P.mirror_scales + l * P.t2_scale_layer_bytes + static_cast<int64_t>(page) * P.t2_scale_page_bytes
                          : nullptr;
  // scale groups: per token, one per K / V over all heads; per token and head, one per (head, K / V)
  const int ngroups = P.scale_per_head ? 2 * p.Hkv : 2;
  const int glen = P.scale_per_head ? p.D : HD;
  for (int gi = warp; gi < ngroups; gi += kMoveThreads / 32) {
    const int kv = P.scale_per_head ? (gi & 1) : gi;
    const int h0 = P.scale_per_head ? (gi >> 1) : 0;
    const float* x = row_s + kv * HD + h0 * p.D;
    float amax = 0.f;
    for (int i = lane; i < glen; i += 32) amax = fmaxf(amax, fabsf(x[i]));
    amax = warp_max(amax);
    __half h16;
    const float div = quant_scale(amax, P.scale_f16, &h16);
    for (int v = lane; v < glen / 16; v += 32) {  // 16 consecutive codes of one head row
      const int i0 = v * 16;
      const int h = h0 + i0 / p.D, e0 = i0 % p.D;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
          word |= (static_cast<uint32_t>(static_cast<uint8_t>(quant_code(x[i0 + 4 * q + bb], div)))) << (8 * bb);
        w[q] = word;
      }
      const int64_t at = ((static_cast<int64_t>(h) * 2 + kv) * kPage + slot) * p.D + e0;
      *reinterpret_cast<uint4*>(pg + at) = make_uint4(w[0], w[1], w[2], w[3]);
      if (mpg) *reinterpret_cast<uint4*>(mpg + at) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (lane == 0) {
      for (int copy = 0; copy < (mpg ? 2 : 1); ++copy) {
        char* scp = copy ? msc : sc;
        if (P.scale_per_head) {
          if (P.scale_f16)
            reinterpret_cast<__half*>(scp)[(h0 * 2 + kv) * kPage + slot] = h16;
          else
            reinterpret_cast<float*>(scp)[(h0 * 2 + kv) * kPage + slot] = div;
        } else {
          reinterpret_cast<float*>(scp)[kv * kPage + slot] = div;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- fold
// One thread per slot of a sequence's attention page list: the slot's position
// gets (sum over layer slices and KV heads of the accumulated weights) /
// (L * Hq) in float64. The next step's first launch overwrites the slots, so
// they are only read here (independent loads, no read-after-write chain).
__global__ void fold_kernel(const __grid_constant__ FoldParams p) {
  const int b = blockIdx.y;
  const int64_t slot = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int n0 = p.npages[0][b], n1 = p.npages[1][b], n2 = p.npages[2][b];
  if (slot >= static_cast<int64_t>(n0 + n1 + n2) * kPage) return;
  int k = static_cast<int>(slot >> 4), src = 0;
  const int row = static_cast<int>(slot & 15);
  if (k >= n0) {
    k -= n0;
    src = 1;
    if (k >= n1) {
      k -= n1;
      src = 2;
    }
  }
  const int page = p.table[src][static_cast<int64_t>(b) * p.table_stride + k];
  if (!index_ok(p.err, DBG_FOLD_PAGE, page, p.cap[src])) return;  // debug build only
  // the slot's metadata, then its (slice, KV head) values: every load is
  // independent, so they go out in batches of U and are added in slice order
  const uint32_t mword = p.mask[src][page];
  const int pos = p.posmap[src][static_cast<int64_t>(page) * kPage + row];
  const float* __restrict__ acc = p.acc + static_cast<int64_t>(p.page_base[b]) * kPage + slot;
  const int n = p.nslices * p.Hkv;
  constexpr int U = 16;
  double sum = 0.0;
  for (int i0 = 0; i0 < n; i0 += U) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u;
      v[u] = i < n ? __ldg(acc + static_cast<int64_t>(i / p.Hkv) * p.acc_stride_l +
                           static_cast<int64_t>(i % p.Hkv) * p.acc_stride_h)
                   : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u < n) sum += static_cast<double>(v[u]);
  }
  if ((mword >> row) & 1u) {
    if (pos >= 0 && index_ok(p.err, DBG_FOLD_POS, pos, p.s_stride))
      p.s[static_cast<int64_t>(b) * p.s_stride + pos] += sum * p.inv_lh;
  }
}

// ---------------------------------------------------------------- quantise rows
__global__ void quantize_rows_kernel(const char* __restrict__ x, int kv_dtype, int64_t rows,
                                     int row_len, int8_t* __restrict__ codes, void* scales,
                                     int scale_f16) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int esz = kv_dtype == 1 ? 2 : 4;
  const char* xr = x + r * row_len * esz;
  float amax = 0.f;
  for (int i = lane; i < row_len; i += 32) amax = fmaxf(amax, fabsf(load_elem(xr + static_cast<int64_t>(i) * esz, kv_dtype)));
  amax = warp_max(amax);
  __half h16;
  const float div = quant_scale(amax, scale_f16, &h16);
  for (int i = lane; i < row_len; i += 32)
    codes[r * row_len + i] = quant_code(load_elem(xr + static_cast<int64_t>(i) * esz, kv_dtype), div);
  if (lane == 0) {
    if (scale_f16)
      reinterpret_cast<__half*>(scales)[r] = h16;
    else
      reinterpret_cast<float*>(scales)[r] = div;
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  append_kernel<<<dim3(p.B, p.L), 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  const int warps = 8;
  prefill_kernel<<<dim3(static_cast<unsigned>((p.n + warps - 1) / warps), p.L), warps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_move(const MoveParams& p, const Mover* movers, int64_t count, int layers, cudaStream_t s) {
  if (count <= 0 || layers <= 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(2) * p.Hkv * p.D * sizeof(float);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(move_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (smem > 96 * 1024) return cudaErrorInvalidValue;
  move_kernel<<<dim3(static_cast<unsigned>(count), static_cast<unsigned>(layers)), kMoveThreads, smem, s>>>(p, movers);
  return cudaGetLastError();
}

cudaError_t launch_fold(const FoldParams& p, cudaStream_t s) {
  if (p.B == 0 || p.max_slots == 0) return cudaSuccess;
  fold_kernel<<<dim3(static_cast<unsigned>((p.max_slots + 255) / 256), p.B), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void* x, int kv_dtype, int64_t rows, int row_len,
                                 int8_t* codes, void* scales, int scale_f16, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int warps = 8;
  quantize_rows_kernel<<<static_cast<unsigned>((rows + warps - 1) / warps), warps * 32, 0, s>>>(
      static_cast<const char*>(x), kv_dtype, rows, row_len, codes, scales, scale_f16);
  return cudaGetLastError();
}

}  // namespace tkv
