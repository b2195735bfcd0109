// common.cuh -- device helpers shared by the verification kernels (sm_103a):
// inline PTX for mbarriers, 1-D bulk async copies (the TMA engine), the
// hardware exp2 approximation, element types, and the two per-row reductions
// the sweep computes (online softmax normaliser, first-index argmax).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kIdxNone = 0x7fffffff;   // argmax index before any element is seen
constexpr int kIdxPoison = -2;         // argmax partial written after a wait timed out

// ---------------------------------------------------------------------------
// element types: bf16 is carried as raw uint16 bits, widened exactly to fp32
// ---------------------------------------------------------------------------
struct F32T {
  static constexpr int esz = 4;
  static constexpr int vpe = 4;   // elements per 16-byte vector
  __device__ static __forceinline__ float load(const unsigned char* base, long long i) {
    return reinterpret_cast<const float*>(base)[i];
  }
  __device__ static __forceinline__ void unpack(const uint4& q, float* x) {
    x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
  }
};

struct BF16T {
  static constexpr int esz = 2;
  static constexpr int vpe = 8;
  __device__ static __forceinline__ float load(const unsigned char* base, long long i) {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(base)[i]) << 16);
  }
  __device__ static __forceinline__ void unpack(const uint4& q, float* x) {
    x[0] = __uint_as_float(q.x << 16); x[1] = __uint_as_float(q.x & 0xffff0000u);
    x[2] = __uint_as_float(q.y << 16); x[3] = __uint_as_float(q.y & 0xffff0000u);
    x[4] = __uint_as_float(q.z << 16); x[5] = __uint_as_float(q.z & 0xffff0000u);
    x[6] = __uint_as_float(q.w << 16); x[7] = __uint_as_float(q.w & 0xffff0000u);
  }
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// try_wait with a suspend-time hint: a waiting warp is parked by the hardware
// (up to ~1 ms) instead of spinning, so it does not steal issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Bounded:
// gives up (returns false) after `timeout_ns` of wall time or 2^24 polls,
// whichever comes first, so a logic error cannot hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < (1u << 24); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > timeout_ns) return false;
  }
  return false;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// fire-and-forget add with release semantics: prior writes of this thread are
// visible before the increment is
__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// packed fp32 pairs (sm_100 family): one instruction for two lanes of math
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the two bf16 halves of a 32-bit word widened to an fp32 pair (exact)
__device__ __forceinline__ unsigned long long bf16x2_to_f2(uint32_t w) {
  return (static_cast<unsigned long long>(w & 0xffff0000u) << 32) | static_cast<unsigned long long>(w << 16);
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One-dimensional bulk copy global -> shared on the async (TMA) engine; the
// byte count is credited to `bar` when the data has landed.  Both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// orders this thread's generic-proxy view of global memory before its later
// bulk-copy (async proxy) reads
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Online softmax normaliser of one row piece at temperature T.
// Keeps m = max element seen and s = sum_i 2^(z_i * c - fl(m * c)), c =
// log2(e)/T, where fl(m * c) is the fp32-rounded product.  Because every term
// of a piece is taken relative to the same rounded offset fl(m * c), pieces
// merge exactly by 2^(fl(m1*c) - fl(m*c)), and the finishing code can rebuild
// the row sum relative to any offset in double precision.
// A NaN element turns s into NaN; +inf makes s NaN too (inf - inf); a piece of
// only -inf elements keeps m = -inf, s = 0.
// ---------------------------------------------------------------------------
struct StatsAcc {
  float m, nA, s;   // nA = -fl(m * c)  (0 while m == -inf)
  __device__ __forceinline__ void init() { m = kNegInf; nA = 0.f; s = 0.f; }

  template <int N>
  __device__ __forceinline__ void add(const float* x, float c) {
    float vm = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) vm = fmaxf(vm, x[i]);
    if (vm > m) {
      const float An = __fmul_rn(vm, c);
      s = (m == kNegInf) ? 0.f : s * ex2_approx(__fadd_rn(-nA, -An));
      m = vm;
      nA = -An;
    }
    float e[N];
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = ex2_approx(__fmaf_rn(x[i], c, nA));
#pragma unroll
    for (int w = 1; w < N; w <<= 1)
#pragma unroll
      for (int i = 0; i + w < N; i += 2 * w) e[i] += e[i + w];
    s += e[0];
  }

  // merge another piece (m2, s2)
  __device__ __forceinline__ void merge(float m2, float s2, float c) {
    const float M = fmaxf(m, m2);
    if (M == kNegInf) return;
    const float AM = __fmul_rn(M, c);
    const float t1 = (m == kNegInf) ? 0.f : s * ex2_approx(__fsub_rn(__fmul_rn(m, c), AM));
    const float t2 = (m2 == kNegInf) ? 0.f : s2 * ex2_approx(__fsub_rn(__fmul_rn(m2, c), AM));
    s = t1 + t2;
    m = M;
    nA = -AM;
  }

  // warp-wide merge: the max first, then each lane rescales its sum once to
  // the common offset fl(M*c) and the sums are added
  __device__ __forceinline__ void warp_reduce(float c) {
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == kNegInf) return;   // every lane empty: s == 0 everywhere
    const float AM = __fmul_rn(M, c);
    float t = (m == kNegInf) ? 0.f : s * ex2_approx(__fsub_rn(__fmul_rn(m, c), AM));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    m = M;
    s = t;
    nA = -AM;
  }
  __device__ __forceinline__ float2 pack() const { return make_float2(m, s); }
  __device__ __forceinline__ void unpack(float2 p) { m = p.x; s = p.y; }
  __device__ static __forceinline__ float2 poison() { return make_float2(__int_as_float(0x7fc00000), -1.f); }
};

// ---------------------------------------------------------------------------
// First-index argmax of one row piece (NaN anywhere poisons the value).
// Elements are visited in increasing index order per thread, so a strict '>'
// keeps the lowest index; merges break value ties by the smaller index.
// ---------------------------------------------------------------------------
struct ArgmaxAcc {
  float best;
  int idx;
  bool nan;
  __device__ __forceinline__ void init() { best = kNegInf; idx = kIdxNone; nan = false; }

  template <int N>
  __device__ __forceinline__ void add(const float* x, int base) {
    float vm = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) vm = fmax_nan(vm, x[i]);
    if (vm > best || idx == kIdxNone || vm != vm) {
      if (vm != vm) {
        nan = true;
      } else if (vm > best || idx == kIdxNone) {
        int f = N - 1;
#pragma unroll
        for (int i = N - 1; i >= 0; --i)
          if (x[i] == vm) f = i;
        best = vm;
        idx = base + f;
      }
    }
  }

  __device__ __forceinline__ void merge(float v2, int i2) {
    if (best != best) return;
    if (v2 != v2) { best = v2; return; }
    if (v2 > best || (v2 == best && i2 < idx)) { best = v2; idx = i2; }
  }
  __device__ __forceinline__ void finalize() {
    if (nan) best = __int_as_float(0x7fc00000);
  }
  __device__ __forceinline__ void warp_reduce() {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
      merge(v2, i2);
    }
  }
  __device__ __forceinline__ float2 pack() const { return make_float2(best, __int_as_float(idx)); }
  __device__ __forceinline__ void unpack(float2 p) { best = p.x; idx = __float_as_int(p.y); nan = false; }
  __device__ static __forceinline__ float2 poison() {
    return make_float2(__int_as_float(0x7fc00000), __int_as_float(kIdxPoison));
  }
};

}  // namespace sv
