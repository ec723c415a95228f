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

__device__ __forceinline__ void store_elem(char* p, float v, int kv_dtype) {
  if (kv_dtype == 1)
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
  else
    *reinterpret_cast<float*>(p) = v;
}

// Rounds a float32 to what the KV dtype stores (identity for float32).
__device__ __forceinline__ float storage_round(float v, int kv_dtype) {
  if (kv_dtype == 1) return __bfloat162float(__float2bfloat16_rn(v));
  return v;
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
// One block per (mover, layer); warp 0 moves the K row, warp 1 the V row.
// The row (all KV heads) is staged in shared memory as float32.
__global__ void move_kernel(const __grid_constant__ MoveParams p, const Mover* __restrict__ movers) {
  extern __shared__ float row_s[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Mover mv = movers[blockIdx.x];
  const int l = blockIdx.y;
  const int kv = warp;
  const int HD = p.Hkv * p.D;
  float* row = row_s + kv * HD;
  const int esz = p.kv_dtype == 1 ? 2 : 4;
  const TierPools& P = p.pools;
  const int64_t row_bytes = static_cast<int64_t>(p.D) * esz;

  // ---- read
  if (p.mode == MOVE_SCATTER) {
    const char* src = p.temp + ((static_cast<int64_t>(mv.temp_row) * p.L + l) * 2 + kv) * HD * esz;
    for (int i = lane; i < HD; i += 32) row[i] = load_elem(src + static_cast<int64_t>(i) * esz, p.kv_dtype);
  } else {
    const int t = mv.src_tier, page = mv.src_loc >> 4, slot = mv.src_loc & 15;
    if (t == 0 || t == 1) {
      const char* pg = P.base[t] + l * P.layer_bytes[t] + static_cast<int64_t>(page) * P.page_bytes[t];
      for (int i = lane; i < HD; i += 32) {
        const int h = i / p.D, e = i % p.D;
        const char* src = pg + ((static_cast<int64_t>(h) * 2 + kv) * kPage + slot) * row_bytes +
                          swz_offset(slot, static_cast<int64_t>(e) * esz, kSwizzle);
        row[i] = load_elem(src, p.kv_dtype);
      }
    } else {
      const char* pg = P.base[2] + l * P.layer_bytes[2] + static_cast<int64_t>(page) * P.page_bytes[2];
      const char* sc = P.t2_scales + l * P.t2_scale_layer_bytes + static_cast<int64_t>(page) * P.t2_scale_page_bytes;
      for (int i = lane; i < HD; i += 32) {
        const int h = i / p.D, e = i % p.D;
        const int8_t code = *reinterpret_cast<const int8_t*>(pg + ((static_cast<int64_t>(h) * 2 + kv) * kPage + slot) * p.D + e);
        float scale;
        if (P.scale_per_head)
          scale = __half2float(reinterpret_cast<const __half*>(sc)[(h * 2 + kv) * kPage + slot]);
        else
          scale = reinterpret_cast<const float*>(sc)[kv * kPage + slot];
        row[i] = storage_round(__fmul_rn(static_cast<float>(code), scale), p.kv_dtype);
      }
    }
  }
  __syncwarp();

  // ---- write
  if (p.mode == MOVE_GATHER) {
    char* dst = p.temp + ((static_cast<int64_t>(mv.temp_row) * p.L + l) * 2 + kv) * HD * esz;
    for (int i = lane; i < HD; i += 32) store_elem(dst + static_cast<int64_t>(i) * esz, row[i], p.kv_dtype);
    return;
  }
  const int t = mv.dst_tier, page = mv.dst_loc >> 4, slot = mv.dst_loc & 15;
  if (t == 0 || t == 1) {
    char* pg = P.base[t] + l * P.layer_bytes[t] + static_cast<int64_t>(page) * P.page_bytes[t];
    for (int i = lane; i < HD; i += 32) {
      const int h = i / p.D, e = i % p.D;
      char* dst = pg + ((static_cast<int64_t>(h) * 2 + kv) * kPage + slot) * row_bytes +
                  swz_offset(slot, static_cast<int64_t>(e) * esz, kSwizzle);
      store_elem(dst, row[i], p.kv_dtype);
    }
    return;
  }
  // into T2: 8-bit codes and scales
  char* pg = P.base[2] + l * P.layer_bytes[2] + static_cast<int64_t>(page) * P.page_bytes[2];
  char* sc = P.t2_scales + l * P.t2_scale_layer_bytes + static_cast<int64_t>(page) * P.t2_scale_page_bytes;
  if (!P.scale_per_head) {
    float amax = 0.f;
    for (int i = lane; i < HD; i += 32) amax = fmaxf(amax, fabsf(row[i]));
    amax = warp_max(amax);
    __half h16;
    const float div = quant_scale(amax, 0, &h16);
    for (int i = lane; i < HD; i += 32) {
      const int h = i / p.D, e = i % p.D;
      *reinterpret_cast<int8_t*>(pg + ((static_cast<int64_t>(h) * 2 + kv) * kPage + slot) * p.D + e) =
          quant_code(row[i], div);
    }
    if (lane == 0) reinterpret_cast<float*>(sc)[kv * kPage + slot] = div;
  } else {
    for (int h = 0; h < p.Hkv; ++h) {
      float amax = 0.f;
      for (int e = lane; e < p.D; e += 32) amax = fmaxf(amax, fabsf(row[h * p.D + e]));
      amax = warp_max(amax);
      __half h16;
      const float div = quant_scale(amax, P.scale_f16, &h16);
      for (int e = lane; e < p.D; e += 32)
        *reinterpret_cast<int8_t*>(pg + ((static_cast<int64_t>(h) * 2 + kv) * kPage + slot) * p.D + e) =
            quant_code(row[h * p.D + e], div);
      if (lane == 0) {
        if (P.scale_f16)
          reinterpret_cast<__half*>(sc)[(h * 2 + kv) * kPage + slot] = h16;
        else
          reinterpret_cast<float*>(sc)[(h * 2 + kv) * kPage + slot] = div;
      }
    }
  }
}

// ---------------------------------------------------------------- fold
// One thread per slot of a sequence's attention page list: the slot's position
// gets (sum over KV heads of the accumulated weights) / (L * Hq) in float64;
// the accumulator is cleared for the next step.
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
  double sum = 0.0;
  for (int h = 0; h < p.Hkv; ++h) {
    float* a = p.acc + (static_cast<int64_t>(b) * p.Hkv + h) * p.acc_stride + slot;
    sum += static_cast<double>(*a);
    *a = 0.f;
  }
  if ((p.mask[src][page] >> row) & 1u) {
    const int pos = p.posmap[src][static_cast<int64_t>(page) * kPage + row];
    if (pos >= 0) p.s[static_cast<int64_t>(b) * p.s_stride + pos] += sum * p.inv_lh;
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

cudaError_t launch_move(const MoveParams& p, const Mover* movers, int64_t count, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(2) * p.Hkv * p.D * sizeof(float);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(move_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (smem > 96 * 1024) return cudaErrorInvalidValue;
  move_kernel<<<dim3(static_cast<unsigned>(count), p.L), 64, smem, s>>>(p, movers);
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
