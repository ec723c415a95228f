// Tier reassignment of "Not All Thoughts Need HBM" (Methodology 1, 4) as a
// segmented radix select spread over many CTAs per sequence.
//
// Candidates are the positions that are neither protected (prompt, sinks,
// recent window) nor already evicted. Ranked by (score descending, position
// ascending), the first max(n0 - |P|, 0) go to T0, the next n1 to T1, the next
// n2 to T2 and the rest to T3. Instead of sorting, the kernels find the three
// boundary keys of that order: each score becomes a 64-bit key whose ascending
// order is descending score (-0 folded onto +0), and an 8-bit-digit
// most-significant-first radix select narrows the key of each boundary rank in
// 8 passes. Each pass is two launches: every CTA histograms its 4096-position
// slice of a sequence (three warp-aggregated histograms at once, one per
// boundary) into the sequence's global histogram, then one CTA per sequence
// picks the next digit of each boundary. Ties at a boundary key are broken by
// position: each slice counts its keys equal to each boundary key, an
// exclusive scan over the slices gives every slice its base rank, and the
// assignment pass ranks equal keys in position order inside each slice with a
// block-wide scan. Every candidate then compares (key, rank) against the three
// boundaries. The result is exact: the same tiers as a stable sort, bit for
// bit.
#include <cuda_runtime.h>

#include "tkv_internal.h"

namespace tkv {
namespace {

constexpr int kThreads = 512;
constexpr int kPer = 8;                       // consecutive positions per thread
constexpr int kSlice = kThreads * kPer;       // positions per CTA
constexpr unsigned long long kNone = ~0ull;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned long long desc_key(double s) {
  if (s == 0.0) s = 0.0;  // -0 and +0 tie
  const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(s));
  const unsigned long long ord = (bits >> 63) ? ~bits : (bits | (1ull << 63));
  return ~ord;  // ascending key = descending score
}

__device__ __forceinline__ int64_t protected_end(const ClassifyParams& p, int b) {
  return p.prompt_len[b] > p.n_sink ? p.prompt_len[b] : p.n_sink;
}
__device__ __forceinline__ int64_t recent_start(const ClassifyParams& p, int b) {
  return p.N[b] - p.recent_window > 0 ? p.N[b] - p.recent_window : 0;
}

// Block-wide sum of one value per thread (all threads get the total).
__device__ long long block_sum(long long v, long long* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  long long t = 0;
  if (w == 0) {
    t = lane < (kThreads / 32) ? red[lane] : 0;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) t += __shfl_xor_sync(kFull, t, m);
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// Block-wide exclusive scan of one value per thread, in thread order.
__device__ long long block_exclusive_scan(long long v, long long* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const long long t = __shfl_up_sync(kFull, incl, m);
    if (lane >= m) incl += t;
  }
  __syncthreads();
  if (lane == 31) red[w] = incl;
  __syncthreads();
  if (w == 0) {
    long long x = lane < (kThreads / 32) ? red[lane] : 0;
    long long xi = x;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const long long t = __shfl_up_sync(kFull, xi, m);
      if (lane >= m) xi += t;
    }
    if (lane < (kThreads / 32)) red[lane] = xi - x;  // exclusive prefix of warp totals
  }
  __syncthreads();
  return red[w] + incl - v;
}

// 1. keys of this slice; candidate and protected counts of the sequence.
__global__ void __launch_bounds__(kThreads) cls_keys(const __grid_constant__ ClassifyParams p) {
  const int b = blockIdx.y;
  const int64_t N = p.N[b];
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kSlice;
  if (lo >= N) return;
  const double* s = p.s + b * p.stride;
  const uint8_t* old = p.old_tier + b * p.stride;
  unsigned long long* keys = p.keys + b * p.stride;
  const int64_t pend = protected_end(p, b), rstart = recent_start(p, b);
  __shared__ long long red[33];
  long long ncand = 0, nprot = 0;
  const int64_t hi = lo + kSlice < N ? lo + kSlice : N;
  for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) {
    const bool prot = i < pend || i >= rstart;
    const bool cand = !prot && old[i] != 3;
    keys[i] = cand ? desc_key(s[i]) : kNone;
    ncand += cand;
    nprot += prot;
  }
  ncand = block_sum(ncand, red);
  nprot = block_sum(nprot, red);
  if (threadIdx.x == 0) {
    ClassifyState& st = p.state[b];
    atomicAdd(&st.ncand, static_cast<unsigned long long>(ncand));
    atomicAdd(&st.nprot, static_cast<unsigned long long>(nprot));
  }
}

// 2. the three boundary ranks of each sequence.
__global__ void cls_setup(const __grid_constant__ ClassifyParams p) {
  const int b = blockIdx.x, j = threadIdx.x;
  if (j >= 3) return;
  ClassifyState& st = p.state[b];
  const long long ncand = static_cast<long long>(st.ncand), nprot = static_cast<long long>(st.nprot);
  const long long a0 = p.n0[b] - nprot > 0 ? p.n0[b] - nprot : 0;
  const long long r = j == 0 ? a0 : j == 1 ? a0 + p.n1[b] : a0 + p.n1[b] + p.n2[b];
  st.rem[j] = r;
  st.done[j] = r >= ncand;  // boundary past the end: every candidate is before it
  st.prefix[j] = 0;
}

// 3a. one radix pass: this slice's digit histograms of the keys that still
// match each boundary's prefix, added into the sequence's global histograms.
__global__ void __launch_bounds__(kThreads) cls_hist(const __grid_constant__ ClassifyParams p, int pass) {
  const int b = blockIdx.y;
  const int64_t N = p.N[b];
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kSlice;
  if (lo >= N) return;
  ClassifyState& st = p.state[b];
  __shared__ unsigned int hist[3][256];
  for (int i = threadIdx.x; i < 3 * 256; i += kThreads) (&hist[0][0])[i] = 0;
  unsigned long long pre[3];
  int done[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    pre[j] = st.prefix[j];
    done[j] = st.done[j];
  }
  __syncthreads();
  if (done[0] && done[1] && done[2]) return;
  const int shift = 56 - 8 * pass;
  const int lane = threadIdx.x & 31;
  const unsigned long long* keys = p.keys + b * p.stride;
  const int64_t hi = lo + kSlice < N ? lo + kSlice : N;
  for (int64_t base = lo; base < hi; base += kThreads) {   // every lane of a warp iterates together
    const int64_t i = base + threadIdx.x;
    const unsigned long long key = i < hi ? keys[i] : kNone;
    const int digit = static_cast<int>((key >> shift) & 0xffu);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const bool take = key != kNone && !done[j] && (pass == 0 || (key >> (shift + 8)) == pre[j]);
      const unsigned grp = __match_any_sync(kFull, take ? digit : 256 + lane);
      if (take && lane == __ffs(grp) - 1) atomicAdd(&hist[j][digit], __popc(grp));
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 3 * 256; i += kThreads) {
    const unsigned v = (&hist[0][0])[i];
    if (v) atomicAdd(&st.hist[i / 256][i % 256], v);
  }
}

// 3b. the next digit of each open boundary; clears the histograms.
__global__ void cls_select(const __grid_constant__ ClassifyParams p) {
  const int b = blockIdx.x, j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (j >= 3) return;
  ClassifyState& st = p.state[b];
  if (lane == 0 && !st.done[j]) {
    long long rem = st.rem[j], cum = 0;
    int d = 0;
    for (; d < 256; ++d) {
      if (rem < cum + static_cast<long long>(st.hist[j][d])) break;
      cum += st.hist[j][d];
    }
    st.prefix[j] = (st.prefix[j] << 8) | static_cast<unsigned long long>(d & 0xff);
    st.rem[j] = rem - cum;
  }
  __syncwarp();
  for (int d = lane; d < 256; d += 32) st.hist[j][d] = 0;
}

// 4. per slice: how many keys equal each boundary key.
__global__ void __launch_bounds__(kThreads) cls_tie_count(const __grid_constant__ ClassifyParams p) {
  const int b = blockIdx.y;
  const int64_t N = p.N[b];
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kSlice;
  if (lo >= N) return;
  const ClassifyState& st = p.state[b];
  const unsigned long long* keys = p.keys + b * p.stride;
  __shared__ long long red[33];
  const int64_t hi = lo + kSlice < N ? lo + kSlice : N;
  for (int j = 0; j < 3; ++j) {
    long long c = 0;
    if (!st.done[j])
      for (int64_t i = lo + threadIdx.x; i < hi; i += kThreads) c += keys[i] == st.prefix[j];
    c = block_sum(c, red);
    if (threadIdx.x == 0) p.slice_ties[(static_cast<int64_t>(b) * p.max_slices + blockIdx.x) * 3 + j] = c;
  }
}

// 5. exclusive scan of the tie counts over a sequence's slices (position order).
__global__ void cls_tie_scan(const __grid_constant__ ClassifyParams p) {
  const int b = blockIdx.x, j = threadIdx.x;
  if (j >= 3) return;
  const int64_t n_slices = (p.N[b] + kSlice - 1) / kSlice;
  long long run = 0;
  for (int64_t c = 0; c < n_slices; ++c) {
    long long& x = p.slice_ties[(static_cast<int64_t>(b) * p.max_slices + c) * 3 + j];
    const long long t = x;
    x = run;
    run += t;
  }
}

// 6. assignment: thread t of a slice takes positions [lo + kPer t, lo + kPer (t + 1)),
// so a block scan of per-thread tie counts ranks equal keys in position order.
__global__ void __launch_bounds__(kThreads) cls_assign(const __grid_constant__ ClassifyParams p) {
  const int b = blockIdx.y;
  const int64_t N = p.N[b];
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kSlice;
  if (lo >= N) return;
  const ClassifyState& st = p.state[b];
  const unsigned long long* keys = p.keys + b * p.stride;
  const uint8_t* old = p.old_tier + b * p.stride;
  uint8_t* nt = p.new_tier + b * p.stride;
  const int64_t pend = protected_end(p, b), rstart = recent_start(p, b);
  __shared__ long long red[33];
  unsigned long long K[3];
  long long R[3], rank[3];
  int done[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    K[j] = st.prefix[j];
    R[j] = st.rem[j];
    done[j] = st.done[j];
  }
  const int64_t i0 = lo + static_cast<int64_t>(threadIdx.x) * kPer;
  unsigned long long key[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) key[e] = i0 + e < N ? keys[i0 + e] : kNone;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    long long c = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) c += key[e] != kNone && key[e] == K[j];
    rank[j] = p.slice_ties[(static_cast<int64_t>(b) * p.max_slices + blockIdx.x) * 3 + j] +
              block_exclusive_scan(c, red);
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int64_t i = i0 + e;
    if (i >= N) break;
    uint8_t t;
    if (i < pend || i >= rstart) {
      t = 0;
    } else if (old[i] == 3) {
      t = 3;
    } else {
      t = 3;
#pragma unroll
      for (int j = 2; j >= 0; --j) {
        const bool before = done[j] || key[e] < K[j] || (key[e] == K[j] && rank[j] < R[j]);
        if (before) t = static_cast<uint8_t>(j);
      }
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) rank[j] += key[e] != kNone && key[e] == K[j];
    nt[i] = t;
  }
}

}  // namespace

int64_t classify_slices(int64_t stride) { return (stride + kSlice - 1) / kSlice; }

cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t s, int* launches) {
  *launches = 0;
  if (p.B <= 0) return cudaSuccess;
  int64_t nmax = 1;
  for (int b = 0; b < p.B; ++b) nmax = p.N[b] > nmax ? p.N[b] : nmax;
  const unsigned slices = static_cast<unsigned>((nmax + kSlice - 1) / kSlice);
  if (slices > p.max_slices) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(p.state, 0, sizeof(ClassifyState) * p.B, s);
  if (e != cudaSuccess) return e;
  const dim3 grid(slices, p.B);
  cls_keys<<<grid, kThreads, 0, s>>>(p);
  cls_setup<<<p.B, 32, 0, s>>>(p);
  *launches = 2;
  for (int pass = 0; pass < 8; ++pass) {
    cls_hist<<<grid, kThreads, 0, s>>>(p, pass);
    cls_select<<<p.B, 96, 0, s>>>(p);
    *launches += 2;
  }
  cls_tie_count<<<grid, kThreads, 0, s>>>(p);
  cls_tie_scan<<<p.B, 32, 0, s>>>(p);
  cls_assign<<<grid, kThreads, 0, s>>>(p);
  *launches += 3;
  return cudaGetLastError();
}

}  // namespace tkv
