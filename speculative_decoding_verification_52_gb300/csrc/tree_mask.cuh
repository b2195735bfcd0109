// tree_mask.cuh -- the tree attention mask: every node of a candidate tree
// attends only to its ancestors and itself ("Speculative decoding and EAGLE",
// section "Tree attention verification"; "Speculative Decoding: from idea to
// SOTA", section 6).
//
// One CTA per sequence (grid-stride over sequences): the sequence's parent
// array is staged in shared memory and checked (parents[0] = -1,
// 0 <= parents[i] < i); then each thread builds the masks of its rows, one at a
// time, in a private shared-memory row of NW = ceil(N/32) words by walking from
// the node up to the root, and writes the row out (the rows of consecutive
// threads are consecutive in memory, so the stores coalesce).  Rows of up to 16
// words take tree_mask_run_kernel (one store per word run of the walk, vector
// stores out); longer rows the general tree_mask_kernel.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int TM_THREADS = 128;
constexpr int TM_MAX_N = 1024;

__global__ void __launch_bounds__(TM_THREADS) tree_mask_kernel(const int32_t* __restrict__ parents, int B, int N,
                                                               uint32_t* __restrict__ out, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char tm_smem[];
  const int NW = (N + 31) / 32;
  int* par = reinterpret_cast<int*>(tm_smem);
  uint32_t* rowbuf = reinterpret_cast<uint32_t*>(par + N) + threadIdx.x * NW;
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    const int32_t* pb = parents + static_cast<long long>(b) * N;
    bool ok = true;
    for (int i = threadIdx.x; i < N; i += TM_THREADS) {
      const int p = pb[i];
      par[i] = p;
      ok &= (i == 0) ? (p == -1) : (p >= 0 && p < i);
    }
    ok = __syncthreads_and(ok);
    uint32_t* ob = out + static_cast<long long>(b) * N * NW;
    for (int i = threadIdx.x; i < N; i += TM_THREADS) {
      for (int w = 0; w < NW; ++w) rowbuf[w] = 0u;
      if (ok) {
        // parents[node] < node on a valid tree, so the walk ends at the root
        for (int node = i; node >= 0; node = par[node]) rowbuf[node >> 5] |= 1u << (node & 31);
      }
      uint32_t* orow = ob + static_cast<long long>(i) * NW;
      for (int w = 0; w < NW; ++w) orow[w] = rowbuf[w];
    }
    if (threadIdx.x == 0) status[b] = ok ? 0 : -1;
    __syncthreads();   // par is reused by the next sequence
  }
}

// The walk visits its nodes in decreasing order (parents[i] < i), so the words
// of the row are visited in non-increasing order and each word's bits form one
// run of the walk: the run's bits gather in one register and are stored once,
// into the thread's row in shared memory (zeroed first), when the walk moves to
// a lower word.  A step costs a shift, an OR and a compare instead of a select
// over every word of the row; the row then goes out with vector stores.
template <int NWT>
__global__ void __launch_bounds__(TM_THREADS) tree_mask_run_kernel(const int32_t* __restrict__ parents, int B, int N,
                                                                   uint32_t* __restrict__ out,
                                                                   int32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char tm_smem[];
  int* par = reinterpret_cast<int*>(tm_smem);
  uint32_t* row = reinterpret_cast<uint32_t*>(tm_smem + ((static_cast<size_t>(N) * sizeof(int) + 15) & ~size_t(15))) +
                  threadIdx.x * NWT;
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    const int32_t* pb = parents + static_cast<long long>(b) * N;
    bool ok = true;
    for (int i = threadIdx.x; i < N; i += TM_THREADS) {
      const int p = pb[i];
      par[i] = p;
      ok &= (i == 0) ? (p == -1) : (p >= 0 && p < i);
    }
    ok = __syncthreads_and(ok);
    const int NW = (N + 31) / 32;   // the row stride; NW <= NWT
    uint32_t* ob = out + static_cast<long long>(b) * N * NW;
    for (int i = threadIdx.x; i < N; i += TM_THREADS) {
      if constexpr (NWT % 4 == 0) {
#pragma unroll
        for (int w = 0; w < NWT; w += 4) reinterpret_cast<uint4*>(row)[w / 4] = make_uint4(0u, 0u, 0u, 0u);
      } else {
#pragma unroll
        for (int w = 0; w < NWT; ++w) row[w] = 0u;
      }
      if (ok) {
        int cw = i >> 5;
        uint32_t run = 0u;
        for (int node = i; node >= 0; node = par[node]) {
          const int wn = node >> 5;
          if (wn != cw) {
            row[cw] = run;
            cw = wn;
            run = 0u;
          }
          run |= 1u << (node & 31);
        }
        row[cw] = run;
      }
      uint32_t* orow = ob + static_cast<long long>(i) * NW;
      if (NW == NWT && NWT % 4 == 0) {
#pragma unroll
        for (int w = 0; w < NWT; w += 4)
          reinterpret_cast<uint4*>(orow)[w / 4] = reinterpret_cast<const uint4*>(row)[w / 4];
      } else {
#pragma unroll
        for (int w = 0; w < NWT; ++w)
          if (w < NW) orow[w] = row[w];
      }
    }
    if (threadIdx.x == 0) status[b] = ok ? 0 : -1;
    __syncthreads();   // par is reused by the next sequence
  }
}

}  // namespace sv
