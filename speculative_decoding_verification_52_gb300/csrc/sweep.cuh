// sweep.cuh -- the vocabulary sweep: one streaming pass over every logit row of
// the batch, producing per-slice partial reductions.
//
// Stats mode computes the temperature-softmax normaliser of each row (the
// pages compute softmax(logits / temperature) for every draft and every target
// position -- "Speculative decoding and EAGLE", section "Make it"; target rows
// over K+1 positions, "The concept", step 2).  Argmax mode computes the
// first-index argmax the greedy rules use ("The exactness rule", greedy case;
// "Tree attention verification").
//
// Work decomposition: rows are cut into S slices of L elements; a unit is one
// (row, slice).  A persistent grid of (SMs x resident CTAs) walks the units
// round-robin.  In each CTA one producer thread streams unit bytes into a ring
// of shared-memory stages with 1-D bulk async copies (cp.async.bulk, completion
// counted on an mbarrier per stage); eight consumer warps read each stage from
// shared memory with 16-byte loads, fold it into per-thread accumulators, hand
// the stage back through an "empty" mbarrier, and reduce the unit across the
// CTA at its end.  Every mbarrier wait is time-bounded; on a timeout the CTA
// writes poison partials (which the finishing kernels report as -2) and drains
// its in-flight copies before exiting.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int SW_CW = 8;                        // consumer warps per CTA
constexpr int SW_CT = SW_CW * 32;               // consumer threads
constexpr int SW_THREADS = SW_CT + 32;          // + one producer warp
constexpr int SW_STAGE = 16384;                 // bytes per ring stage
constexpr int SW_NSTAGE = 4;                    // ring depth
constexpr int SW_SMEM = SW_NSTAGE * SW_STAGE + 2 * SW_NSTAGE * 8 + 2 * SW_CW * 8 + 16;

enum { MODE_STATS = 0, MODE_ARGMAX = 1 };

struct SweepArgs {
  const unsigned char* seg0;   // rows [0, rows0): element type TA
  const unsigned char* seg1;   // rows [rows0, ...): element type TB
  long long rows0;
  long long units;             // total rows * S
  int S;                       // slices per row
  int L;                       // slice length in elements (multiple of 8)
  int V;
  float c;                     // log2(e) / temperature (stats mode)
  float2* part;                // [units] partials
  unsigned long long timeout_ns;
};

struct Unit {
  const unsigned char* src;
  uint32_t bytes;
  int e0;
  bool seg1;
};

template <class TA, class TB>
__device__ __forceinline__ Unit sweep_unit(const SweepArgs& a, long long u) {
  const long long r = u / a.S;
  const int j = static_cast<int>(u - r * a.S);
  const int e0 = j * a.L;
  const int e1 = min(a.V, e0 + a.L);
  Unit d;
  d.e0 = e0;
  if (r < a.rows0) {
    d.src = a.seg0 + (r * a.V + e0) * static_cast<long long>(TA::esz);
    d.bytes = static_cast<uint32_t>((e1 - e0) * TA::esz);
    d.seg1 = false;
  } else {
    d.src = a.seg1 + ((r - a.rows0) * a.V + e0) * static_cast<long long>(TB::esz);
    d.bytes = static_cast<uint32_t>((e1 - e0) * TB::esz);
    d.seg1 = true;
  }
  return d;
}

template <int MODE>
struct AccOf;
template <>
struct AccOf<MODE_STATS> { using type = StatsAcc; };
template <>
struct AccOf<MODE_ARGMAX> { using type = ArgmaxAcc; };

template <class T, int MODE, class Acc>
__device__ __forceinline__ void consume_stage(const uint4* buf, int nvec, int ctid, int elem_base, float c,
                                              Acc& acc) {
#pragma unroll 4
  for (int v = ctid; v < nvec; v += SW_CT) {
    const uint4 q = buf[v];
    float x[T::vpe];
    T::unpack(q, x);
    if constexpr (MODE == MODE_STATS) {
      acc.template add<T::vpe>(x, c);
    } else {
      acc.template add<T::vpe>(x, elem_base + v * T::vpe);
    }
  }
}

template <class TA, class TB, int MODE>
__global__ void __launch_bounds__(SW_THREADS, 1) sweep_tma_kernel(const SweepArgs a) {
  using Acc = typename AccOf<MODE>::type;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SW_NSTAGE * SW_STAGE);
  uint64_t* empty = full + SW_NSTAGE;
  float2* red = reinterpret_cast<float2*>(empty + SW_NSTAGE);        // [2][SW_CW]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 2 * SW_CW);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < SW_NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], SW_CW);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer: one thread issues the bulk copies ----------
    if (lane != 0) return;
    int stage = 0;
    uint32_t phase = 0;
    int last_parity[SW_NSTAGE];
#pragma unroll
    for (int s = 0; s < SW_NSTAGE; ++s) last_parity[s] = -1;
    bool ok = true;
    for (long long u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
      const Unit d = sweep_unit<TA, TB>(a, u);
      for (uint32_t off = 0; off < d.bytes; off += SW_STAGE) {
        const uint32_t n = min(static_cast<uint32_t>(SW_STAGE), d.bytes - off);
        if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1u, a.timeout_ns)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], n);
        bulk_g2s(smem + stage * SW_STAGE, d.src + off, n, &full[stage]);
        last_parity[stage] = static_cast<int>(phase);
        if (++stage == SW_NSTAGE) { stage = 0; phase ^= 1u; }
      }
    }
    // drain: do not leave while a copy may still land in this CTA's memory
#pragma unroll
    for (int s = 0; s < SW_NSTAGE; ++s)
      if (last_parity[s] >= 0) mbar_wait(&full[s], static_cast<uint32_t>(last_parity[s]), a.timeout_ns);
    return;
  }

  // ---------------- consumers ------------------------------------------------
  const int ctid = threadIdx.x - 32, cw = warp - 1;
  int stage = 0;
  uint32_t phase = 0;
  int rb = 0;
  bool dead = false;
  for (long long u = blockIdx.x; u < a.units; u += gridDim.x) {
    const Unit d = sweep_unit<TA, TB>(a, u);
    Acc acc;
    acc.init();
    for (uint32_t off = 0; off < d.bytes; off += SW_STAGE) {
      const uint32_t n = min(static_cast<uint32_t>(SW_STAGE), d.bytes - off);
      if (!dead && *abort_flag) dead = true;
      if (!dead && !mbar_wait(&full[stage], phase, a.timeout_ns)) {
        dead = true;
        *abort_flag = 1;
      }
      if (!dead) {
        const uint4* buf = reinterpret_cast<const uint4*>(smem + stage * SW_STAGE);
        const int nvec = static_cast<int>(n >> 4);
        if (d.seg1) {
          consume_stage<TB, MODE>(buf, nvec, ctid, d.e0 + static_cast<int>(off / TB::esz), a.c, acc);
        } else {
          consume_stage<TA, MODE>(buf, nvec, ctid, d.e0 + static_cast<int>(off / TA::esz), a.c, acc);
        }
      }
      __syncwarp();
      if (lane == 0 && !dead) mbar_arrive(&empty[stage]);
      if (++stage == SW_NSTAGE) { stage = 0; phase ^= 1u; }
    }
    // unit reduction across the consumer warps
    if constexpr (MODE == MODE_STATS) {
      acc.warp_reduce(a.c);
    } else {
      acc.finalize();
      acc.warp_reduce();
    }
    if (lane == 0) red[rb * SW_CW + cw] = acc.pack();
    named_bar_sync(1, SW_CT);
    if (cw == 0) {
      Acc t;
      t.init();
      if (lane < SW_CW) t.unpack(red[rb * SW_CW + lane]);
      if constexpr (MODE == MODE_STATS) {
        t.warp_reduce(a.c);
      } else {
        t.warp_reduce();
      }
      if (lane == 0) a.part[u] = (*abort_flag) ? Acc::poison() : t.pack();
    }
    rb ^= 1;
  }
}

// Scalar fallback for rows that are not 16-byte aligned (V * elem_size not a
// multiple of 16, or unaligned base pointers): one CTA per unit, plain loads.
constexpr int SS_THREADS = 256;

template <class TA, class TB, int MODE>
__global__ void __launch_bounds__(SS_THREADS) sweep_scalar_kernel(const SweepArgs a) {
  using Acc = typename AccOf<MODE>::type;
  __shared__ float2 red[SS_THREADS / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long long u = blockIdx.x; u < a.units; u += gridDim.x) {
    const long long r = u / a.S;
    const int j = static_cast<int>(u - r * a.S);
    const int e0 = j * a.L, e1 = min(a.V, e0 + a.L);
    Acc acc;
    acc.init();
    for (int e = e0 + threadIdx.x; e < e1; e += SS_THREADS) {
      float x[1];
      x[0] = (r < a.rows0) ? TA::load(a.seg0, r * a.V + e) : TB::load(a.seg1, (r - a.rows0) * a.V + e);
      if constexpr (MODE == MODE_STATS) {
        acc.template add<1>(x, a.c);
      } else {
        acc.template add<1>(x, e);
      }
    }
    if constexpr (MODE == MODE_STATS) {
      acc.warp_reduce(a.c);
    } else {
      acc.finalize();
      acc.warp_reduce();
    }
    if (lane == 0) red[warp] = acc.pack();
    __syncthreads();
    if (warp == 0) {
      Acc t;
      t.init();
      if (lane < SS_THREADS / 32) t.unpack(red[lane]);
      if constexpr (MODE == MODE_STATS) {
        t.warp_reduce(a.c);
      } else {
        t.warp_reduce();
      }
      if (lane == 0) a.part[u] = t.pack();
    }
    __syncthreads();
  }
}

}  // namespace sv
