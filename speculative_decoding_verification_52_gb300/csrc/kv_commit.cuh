// kv_commit.cuh -- commit on accept for the KV cache: the drafts' entries are
// written to a scratch buffer by the verification pass, and only the accepted
// ones are appended to the cache, so a rejection leaves the cache at the
// accepted length ("Speculative decoding: draft, verify, repeat", KV rollback:
// scratch buffer, commit on acceptance, discard on reject).
//
// One CTA per (sequence, appended entry): the sequence's request is checked
// (slots inside the scratch buffer, no overflow of the cache) by every CTA of
// the sequence, then the entry is copied with 16-byte vectors when the entry
// size and both buffers allow it, else byte by byte.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int KV_THREADS = 256;

struct KvCommitArgs {
  unsigned char* cache;          // [B, Lmax, E]
  const int32_t* lengths;        // [B]
  const unsigned char* scratch;  // [B, N, E]
  const int32_t* path;           // [B, W] or null (slots 0, 1, ...)
  const int32_t* count;          // [B]
  int B, Lmax, N, W, J;          // J: entries per sequence handled by the grid (W, or N without a path)
  unsigned long long E;          // entry bytes
  int32_t* new_lengths;          // [B]
  bool vec;                      // 16-byte copies
};

__device__ __forceinline__ int kv_slot(const KvCommitArgs& a, int b, int j) {
  return a.path ? a.path[static_cast<long long>(b) * a.W + j] : j;
}

__global__ void __launch_bounds__(KV_THREADS) kv_commit_kernel(const KvCommitArgs a) {
  const long long pairs = static_cast<long long>(a.B) * a.J;
  for (long long p = blockIdx.x; p < pairs; p += gridDim.x) {
    const int b = static_cast<int>(p / a.J), j = static_cast<int>(p - static_cast<long long>(b) * a.J);
    const int n = a.count[b], L = a.lengths[b];
    if (n < 0) {
      if (j == 0 && threadIdx.x == 0) a.new_lengths[b] = L;
      continue;
    }
    bool ok = L >= 0 && static_cast<long long>(L) + n <= a.Lmax && (a.path == nullptr || n <= a.W);
    for (int k = threadIdx.x; ok && k < n; k += KV_THREADS) {
      const int s = kv_slot(a, b, k);
      if (s < 0 || s >= a.N) ok = false;
    }
    ok = __syncthreads_and(ok);
    if (j == 0 && threadIdx.x == 0) a.new_lengths[b] = ok ? L + n : -1;
    if (!ok || j >= n) continue;
    const int s = kv_slot(a, b, j);
    const unsigned char* src = a.scratch + (static_cast<unsigned long long>(b) * a.N + s) * a.E;
    unsigned char* dst = a.cache + (static_cast<unsigned long long>(b) * a.Lmax + L + j) * a.E;
    if (a.vec) {
      // four loads in flight per thread before their stores
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      const unsigned long long nv = a.E / 16;
      unsigned long long k = threadIdx.x;
      for (; k + 3 * KV_THREADS < nv; k += 4 * KV_THREADS) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcs(s4 + k + u * KV_THREADS);
#pragma unroll
        for (int u = 0; u < 4; ++u) d4[k + u * KV_THREADS] = v[u];
      }
      for (; k < nv; k += KV_THREADS) d4[k] = __ldcs(s4 + k);
    } else {
      for (unsigned long long k = threadIdx.x; k < a.E; k += KV_THREADS) dst[k] = src[k];
    }
  }
}

}  // namespace sv
