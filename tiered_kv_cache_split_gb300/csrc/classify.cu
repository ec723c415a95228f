// Tier reassignment of "Not All Thoughts Need HBM" (Methodology 1, 4) as a
// segmented radix select: one CTA per sequence.
//
// Candidates are the positions that are neither protected (prompt, sinks,
// recent window) nor already evicted. Ranked by (score descending, position
// ascending), the first max(n0 - |P|, 0) go to T0, the next n1 to T1, the next
// n2 to T2 and the rest to T3. Instead of sorting, the kernel finds the three
// boundary elements of that order: each score becomes a 64-bit key whose
// ascending order is descending score (-0 folded onto +0), an 8-bit-digit
// most-significant-first radix select narrows the key of each boundary rank in
// 8 passes (three histograms per pass, warp-aggregated), and one ordered scan
// resolves ties at each boundary key by position. Every candidate then compares
// (key, position) against the three boundaries. The result is exact: the same
// tiers as a stable sort, bit for bit.
#include <cuda_runtime.h>

#include "tkv_internal.h"

namespace tkv {
namespace {

constexpr int kThreads = 1024;
constexpr unsigned long long kNone = ~0ull;

__device__ __forceinline__ unsigned long long desc_key(double s) {
  if (s == 0.0) s = 0.0;  // -0 and +0 tie
  const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(s));
  const unsigned long long ord = (bits >> 63) ? ~bits : (bits | (1ull << 63));
  return ~ord;  // ascending key = descending score
}

__device__ long long block_sum(long long v, long long* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  if (lane == 0) red[w] = v;
  __syncthreads();
  long long t = 0;
  if (threadIdx.x < 32) {
    t = threadIdx.x < (kThreads / 32) ? red[threadIdx.x] : 0;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
    if (threadIdx.x == 0) red[32] = t;
  }
  __syncthreads();
  t = red[32];
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(kThreads) classify_kernel(const __grid_constant__ ClassifyParams p) {
  const int b = blockIdx.x;
  const int64_t N = p.N[b];
  const double* s = p.s + b * p.stride;
  const uint8_t* old = p.old_tier + b * p.stride;
  uint8_t* nt = p.new_tier + b * p.stride;
  unsigned long long* keys = p.keys + b * p.stride;
  const int64_t plen = p.prompt_len[b] > p.n_sink ? p.prompt_len[b] : p.n_sink;
  const int64_t rstart = N - p.recent_window > 0 ? N - p.recent_window : 0;

  __shared__ long long red[33];
  __shared__ int hist[3][256];
  __shared__ unsigned long long s_prefix[3];
  __shared__ long long s_rem[3];
  __shared__ int s_done[3];
  __shared__ long long s_tpos[3];
  __shared__ long long s_scan[3][kThreads / 32];

  // 1. keys; count candidates and protected positions
  long long ncand = 0, nprot = 0;
  for (int64_t i = threadIdx.x; i < N; i += kThreads) {
    const bool prot = i < plen || i >= rstart;
    const bool cand = !prot && old[i] != 3;
    keys[i] = cand ? desc_key(s[i]) : kNone;
    ncand += cand;
    nprot += prot;
  }
  ncand = block_sum(ncand, red);
  nprot = block_sum(nprot, red);

  const long long a0 = p.n0[b] - nprot > 0 ? p.n0[b] - nprot : 0;
  if (threadIdx.x < 3) {
    const long long r = threadIdx.x == 0 ? a0 : threadIdx.x == 1 ? a0 + p.n1[b] : a0 + p.n1[b] + p.n2[b];
    s_rem[threadIdx.x] = r;
    s_done[threadIdx.x] = r >= ncand;  // boundary past the end: every candidate is before it
    s_prefix[threadIdx.x] = 0;
    s_tpos[threadIdx.x] = -1;
  }
  __syncthreads();

  // 2. radix select of the three boundary keys, 8 bits per pass, MSB first
  const int lane = threadIdx.x & 31;
  const int64_t nround = (N + kThreads - 1) / kThreads * kThreads;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int i = threadIdx.x; i < 3 * 256; i += kThreads) (&hist[0][0])[i] = 0;
    __syncthreads();
    unsigned long long pre[3];
    int done[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      pre[j] = s_prefix[j];
      done[j] = s_done[j];
    }
    for (int64_t i = threadIdx.x; i < nround; i += kThreads) {
      const unsigned long long key = i < N ? keys[i] : kNone;
      const int digit = static_cast<int>((key >> shift) & 0xffu);
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const bool take = key != kNone && !done[j] && (pass == 0 || (key >> (shift + 8)) == pre[j]);
        const unsigned grp = __match_any_sync(0xffffffffu, take ? digit : 256 + lane);
        if (take && lane == __ffs(grp) - 1) atomicAdd(&hist[j][digit], __popc(grp));
      }
    }
    __syncthreads();
    if (threadIdx.x < 3) {
      const int j = threadIdx.x;
      if (!s_done[j]) {
        long long rem = s_rem[j], cum = 0;
        int d = 0;
        for (; d < 256; ++d) {
          if (rem < cum + hist[j][d]) break;
          cum += hist[j][d];
        }
        s_prefix[j] = (s_prefix[j] << 8) | static_cast<unsigned long long>(d & 0xff);
        s_rem[j] = rem - cum;
      }
    }
    __syncthreads();
  }

  // 3. ties at each boundary key: the s_rem[j]-th tie in position order
  {
    const int64_t span = (N + kThreads - 1) / kThreads;
    const int64_t lo = static_cast<int64_t>(threadIdx.x) * span;
    const int64_t hi = lo + span < N ? lo + span : N;
    long long cnt[3] = {0, 0, 0};
    for (int64_t i = lo; i < hi; ++i) {
      const unsigned long long key = keys[i];
#pragma unroll
      for (int j = 0; j < 3; ++j) cnt[j] += (key != kNone && key == s_prefix[j]);
    }
    // block exclusive scan of the three counts (in thread order = position order)
    const int w = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      long long incl = cnt[j];
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, m);
        if (lane >= m) incl += t;
      }
      if (lane == 31) s_scan[j][w] = incl;
      cnt[j] = incl - cnt[j];  // exclusive within the warp
    }
    __syncthreads();
    if (threadIdx.x < 3) {
      long long run = 0;
      for (int ww = 0; ww < kThreads / 32; ++ww) {
        const long long t = s_scan[threadIdx.x][ww];
        s_scan[threadIdx.x][ww] = run;
        run += t;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      if (s_done[j]) continue;
      long long before = cnt[j] + s_scan[j][w];
      const long long want = s_rem[j];
      for (int64_t i = lo; i < hi; ++i) {
        const unsigned long long key = keys[i];
        if (key != kNone && key == s_prefix[j]) {
          if (before == want) s_tpos[j] = i;
          ++before;
        }
      }
    }
    __syncthreads();
  }

  // 4. assign
  unsigned long long K[3];
  long long P[3];
  int done[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    K[j] = s_prefix[j];
    P[j] = s_tpos[j];
    done[j] = s_done[j];
  }
  for (int64_t i = threadIdx.x; i < N; i += kThreads) {
    const bool prot = i < plen || i >= rstart;
    uint8_t t;
    if (prot) {
      t = 0;
    } else if (old[i] == 3) {
      t = 3;
    } else {
      const unsigned long long key = keys[i];
      t = 3;
#pragma unroll
      for (int j = 2; j >= 0; --j) {
        const bool before = done[j] || key < K[j] || (key == K[j] && i < P[j]);
        if (before) t = static_cast<uint8_t>(j);
      }
    }
    nt[i] = t;
  }
}

}  // namespace

cudaError_t launch_classify(const ClassifyParams& p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  classify_kernel<<<p.B, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tkv
