// row_stats.cuh -- per-position acceptance statistics of a draft against its
// target: alpha = sum_v min(p, q), KL(q || p) and TV = 1/2 sum_v |p - q|.
//
// "Speculative decoding: draft, verify, repeat", step 4 (acceptance rate
// against the divergence between the draft and the verifier) and "Speculative
// Decoding: from idea to SOTA", section 3 (a draft token is accepted with
// probability min(1, p/q), so position t is accepted with probability
// sum_v q(v) min(1, p(v)/q(v)) = sum_v min(p(v), q(v))).
//
// One thread-block cluster per (sequence, position) pair.  Each CTA of the
// cluster holds one vocabulary slice of the target row and of the draft row in
// shared memory, landed by two bulk async copies, so HBM is read exactly once.
// Three passes over shared memory follow, each closed by one exchange through
// distributed shared memory (every CTA stores its partial into a slot of every
// peer, then a cluster barrier):
//   A. row maxima M_p, M_q (NaN propagates; +inf, NaN or an all -inf row mark
//      the pair invalid);
//   B. S_p = sum 2^(z c - fl(M_p c)), S_q likewise, D = sum e_q (y - z), with
//      c = log2(e) / T (draft probabilities: S_p and the validity of q only);
//   C. alpha = sum 2^min(u_p, u_q) with u = x c - fl(M c) - log2 S, i.e. the
//      log2 of p and q: min(2^a, 2^b) = 2^min(a, b) costs one exp per pair.
//      With draft probabilities: alpha = sum min(p, q), TV = 1/2 sum |p - q|,
//      KL = sum_{q>0} q (ln q - ln p).
// For logits, KL(q || p) = sum q (ln q - ln p) has the closed form
//   ln2 * (c D / S_q - fl(M_q c) + fl(M_p c)) - ln S_q + ln S_p
// (sum q = 1), and TV = 1 - alpha (|p - q| = p + q - 2 min(p, q), both sums 1).
#pragma once

#include "common.cuh"

namespace sv {

constexpr int RS_THREADS = 256;
constexpr int RS_MAX_CLUSTER = 8;
constexpr int RS_TARGET_SMEM = 64 * 1024;    // slice bytes aimed at (3 CTAs per SM)
constexpr int RS_MAX_SMEM = 200 * 1024;      // largest slice pair one CTA may hold
constexpr float RS_TIMEOUT_MARK = -2.f;      // all three outputs after a wait ran out

struct RowStatsArgs {
  const unsigned char* target;   // [B, K+1, V]
  const unsigned char* draft;    // [B, K, V]
  int B, K, V;
  int L;        // slice length per CTA (elements, multiple of 16)
  int CS;       // CTAs per cluster = ceil(V / L)
  int vec;      // rows may be landed by bulk copies
  float c;      // log2(e) / T
  float* alpha; // [B, K]
  float* kl;
  float* tv;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// store v into the same shared-memory slot of CTA `peer` of this cluster
__device__ __forceinline__ void st_peer_f32(float* local_slot, uint32_t peer, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local_slot)), "r"(peer));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// 8 consecutive elements of a shared-memory slice, widened to fp32
template <class T>
__device__ __forceinline__ void rs_ld8(const unsigned char* s, int g, float* x);
template <>
__device__ __forceinline__ void rs_ld8<BF16T>(const unsigned char* s, int g, float* x) {
  BF16T::unpack(*reinterpret_cast<const uint4*>(s + static_cast<size_t>(g) * 16), x);
}
template <>
__device__ __forceinline__ void rs_ld8<F32T>(const unsigned char* s, int g, float* x) {
  const uint4* p = reinterpret_cast<const uint4*>(s + static_cast<size_t>(g) * 32);
  F32T::unpack(p[0], x);
  F32T::unpack(p[1], x + 4);
}

// fill value of padding elements: -inf for logits (no mass), 0 for probabilities
template <class T>
__device__ __forceinline__ void rs_pad(unsigned char* s, int i, bool zero) {
  if (T::esz == 2)
    reinterpret_cast<uint16_t*>(s)[i] = zero ? 0 : 0xff80u;
  else
    reinterpret_cast<uint32_t*>(s)[i] = zero ? 0u : 0xff800000u;
}

// block-wide reduction of up to 4 values (op: 0 = sum, 1 = NaN-propagating max);
// every thread receives the result.  Each call site has its own scratch
// array, so no barrier is needed before the scratch is written.
template <int N>
__device__ __forceinline__ void rs_block_reduce(float* v, const int* op, float (*red)[RS_THREADS / 32]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < N; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float w = __shfl_xor_sync(0xffffffffu, v[k], o);
      v[k] = op[k] ? fmax_nan(v[k], w) : v[k] + w;
    }
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < N; ++k) red[k][warp] = v[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float r = red[k][0];
#pragma unroll
    for (int w = 1; w < RS_THREADS / 32; ++w) r = op[k] ? fmax_nan(r, red[k][w]) : r + red[k][w];
    v[k] = r;
  }
}

// publish this CTA's N values into slot[rank] of every peer, then meet at a
// cluster barrier; afterwards slots[k][0..CS) hold every CTA's values
template <int N>
__device__ __forceinline__ void rs_exchange(const float* v, float (*slots)[RS_MAX_CLUSTER], uint32_t rank,
                                            uint32_t CS) {
  if (threadIdx.x < CS)
#pragma unroll
    for (int k = 0; k < N; ++k) st_peer_f32(&slots[k][rank], threadIdx.x, v[k]);
  cluster_sync_all();
}

template <class TP, class TQ, bool PROBS>
__global__ void __launch_bounds__(RS_THREADS) row_stats_kernel(RowStatsArgs a) {
  extern __shared__ __align__(128) unsigned char rs_smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ float red[3][4][RS_THREADS / 32];   // one scratch array per pass
  __shared__ float xa[2][RS_MAX_CLUSTER];   // pass A: M_p, M_q
  __shared__ float xb[4][RS_MAX_CLUSTER];   // pass B: S_p, S_q, D (or bad q), timeout
  __shared__ float xc[3][RS_MAX_CLUSTER];   // pass C: alpha, (probs) tv, kl
  __shared__ int s_timeout;

  const uint32_t CS = static_cast<uint32_t>(a.CS);
  // bf16 target and draft logits: packed bf16x2 / f32x2 arithmetic
  constexpr bool kPackedBF16 = TP::esz == 2 && TQ::esz == 2 && !PROBS;
  const uint32_t rank = cluster_rank();
  const long long pos = blockIdx.x / CS;   // (sequence, position) pair of this cluster
  const int b = static_cast<int>(pos / a.K), t = static_cast<int>(pos % a.K);
  const int start = static_cast<int>(rank) * a.L;
  const int n = max(0, min(a.L, a.V - start));
  const int ng = (n + 7) >> 3;   // groups of 8 (the last one padded)

  unsigned char* sp = rs_smem;
  unsigned char* sq = rs_smem + static_cast<size_t>(a.L) * TP::esz;
  const unsigned char* gp =
      a.target + ((static_cast<long long>(b) * (a.K + 1) + t) * a.V + start) * static_cast<long long>(TP::esz);
  const unsigned char* gq =
      a.draft + ((static_cast<long long>(b) * a.K + t) * a.V + start) * static_cast<long long>(TQ::esz);

  // ---- land the slices -------------------------------------------------------
  if (threadIdx.x == 0) {
    s_timeout = 0;
    if (a.vec) {
      mbar_init(&bar, 1);
      mbar_fence_init();
    }
  }
  __syncthreads();
  // every CTA of the cluster must be running before any of them stores into a
  // peer's shared memory: arrive now, wait just before the first exchange
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  bool timed_out = false;
  if (a.vec) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(n) * (TP::esz + TQ::esz));
      if (n > 0) {
        bulk_g2s(sp, gp, static_cast<uint32_t>(n) * TP::esz, &bar);
        bulk_g2s(sq, gq, static_cast<uint32_t>(n) * TQ::esz, &bar);
      }
    }
    if (!mbar_wait(&bar, 0, 1000000000ull)) {
      timed_out = true;
      s_timeout = 1;
    }
  } else {
    for (int i = threadIdx.x; i < n; i += RS_THREADS) {
      if (TP::esz == 2) reinterpret_cast<uint16_t*>(sp)[i] = reinterpret_cast<const uint16_t*>(gp)[i];
      else reinterpret_cast<uint32_t*>(sp)[i] = reinterpret_cast<const uint32_t*>(gp)[i];
      if (TQ::esz == 2) reinterpret_cast<uint16_t*>(sq)[i] = reinterpret_cast<const uint16_t*>(gq)[i];
      else reinterpret_cast<uint32_t*>(sq)[i] = reinterpret_cast<const uint32_t*>(gq)[i];
    }
  }
  // pad the last group (disjoint from the bulk-copied bytes)
  if (threadIdx.x < ng * 8 - n) {
    rs_pad<TP>(sp, n + threadIdx.x, false);
    rs_pad<TQ>(sq, n + threadIdx.x, PROBS);
  }
  __syncthreads();

  // ---- pass A: row maxima ----------------------------------------------------
  float mx[2] = {kNegInf, kNegInf};
  {
    if constexpr (kPackedBF16) {
      // NaN-propagating packed maxima of the raw bf16 words, halves combined once
      uint32_t mp = 0xff80ff80u, mq = 0xff80ff80u;
      for (int g = threadIdx.x; g < ng; g += RS_THREADS) {
        const uint4 a4 = reinterpret_cast<const uint4*>(sp)[g], b4 = reinterpret_cast<const uint4*>(sq)[g];
        mp = bf16x2_max_nan(mp, bf16x2_max_nan(bf16x2_max_nan(a4.x, a4.y), bf16x2_max_nan(a4.z, a4.w)));
        mq = bf16x2_max_nan(mq, bf16x2_max_nan(bf16x2_max_nan(b4.x, b4.y), bf16x2_max_nan(b4.z, b4.w)));
      }
      mx[0] = fmax_nan(__uint_as_float(mp << 16), __uint_as_float(mp & 0xffff0000u));
      mx[1] = fmax_nan(__uint_as_float(mq << 16), __uint_as_float(mq & 0xffff0000u));
    } else {
      float zp[8], zq[8];
      for (int g = threadIdx.x; g < ng; g += RS_THREADS) {
        rs_ld8<TP>(sp, g, zp);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[0] = fmax_nan(mx[0], zp[i]);
        if (!PROBS) {
          rs_ld8<TQ>(sq, g, zq);
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[1] = fmax_nan(mx[1], zq[i]);
        }
      }
    }
  }
  {
    const int op[2] = {1, 1};
    rs_block_reduce<2>(mx, op, red[0]);
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  rs_exchange<2>(mx, xa, rank, CS);
  float Mp = xa[0][0], Mq = xa[1][0];
  for (uint32_t r = 1; r < CS; ++r) {
    Mp = fmax_nan(Mp, xa[0][r]);
    Mq = fmax_nan(Mq, xa[1][r]);
  }
  const float c = a.c;
  const float Ap = __fmul_rn(Mp, c), Aq = __fmul_rn(Mq, c);
  // a row is usable iff its maximum is finite (NaN, +inf, or no finite entry: not)
  const bool rows_ok = isfinite(Mp) && (PROBS || isfinite(Mq));
  const float kp = rows_ok ? -Ap : 0.f, kq = rows_ok ? -Aq : 0.f;

  // ---- pass B: normalisers ---------------------------------------------------
  float vb[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (kPackedBF16) {
    // per pair of elements: both exponents by one packed fma each, two ex2
    // per row, D += e_q (y - z) with y - z >= -FLT_MAX (a -inf draft logit has
    // e_q = 0 and must add nothing)
    const unsigned long long c2 = f2_pack(c, c), kp2 = f2_pack(kp, kp), kq2 = f2_pack(kq, kq);
    const unsigned long long m1 = f2_pack(-1.f, -1.f);
    unsigned long long sp2 = f2_pack(0.f, 0.f), sq2 = sp2, d2 = sp2;
    for (int g = threadIdx.x; g < ng; g += RS_THREADS) {
      const uint4 a4 = reinterpret_cast<const uint4*>(sp)[g], b4 = reinterpret_cast<const uint4*>(sq)[g];
      const uint32_t wz[4] = {a4.x, a4.y, a4.z, a4.w}, wy[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const unsigned long long z2 = bf16x2_to_f2(wz[i]), y2 = bf16x2_to_f2(wy[i]);
        float a0, a1, b0, b1, t0, t1;
        f2_unpack(f2_fma(z2, c2, kp2), a0, a1);
        f2_unpack(f2_fma(y2, c2, kq2), b0, b1);
        const unsigned long long ep2 = f2_pack(ex2_approx(a0), ex2_approx(a1));
        const unsigned long long eq2 = f2_pack(ex2_approx(b0), ex2_approx(b1));
        sp2 = f2_add(sp2, ep2);
        sq2 = f2_add(sq2, eq2);
        f2_unpack(f2_fma(z2, m1, y2), t0, t1);
        d2 = f2_fma(eq2, f2_pack(fmaxf(t0, -3.402823466e38f), fmaxf(t1, -3.402823466e38f)), d2);
      }
    }
    float x0, x1;
    f2_unpack(sp2, x0, x1);
    vb[0] = x0 + x1;
    f2_unpack(sq2, x0, x1);
    vb[1] = x0 + x1;
    f2_unpack(d2, x0, x1);
    vb[2] = x0 + x1;
  } else {
    float zp[8], zq[8];
    for (int g = threadIdx.x; g < ng; g += RS_THREADS) {
      rs_ld8<TP>(sp, g, zp);
      rs_ld8<TQ>(sq, g, zq);
      float e[8], f[8], d[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) e[i] = ex2_approx(__fmaf_rn(zp[i], c, kp));
      if (!PROBS) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          f[i] = ex2_approx(__fmaf_rn(zq[i], c, kq));
          d[i] = f[i] > 0.f ? f[i] * (zq[i] - zp[i]) : 0.f;
        }
      } else {
        bool bad = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) bad |= !(zq[i] >= 0.f);   // NaN or negative
        vb[1] = bad ? 1.f : vb[1];
      }
      // tree within the group, then one add per group
#pragma unroll
      for (int w = 1; w < 8; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < 8; i += 2 * w) {
          e[i] += e[i + w];
          if (!PROBS) {
            f[i] += f[i + w];
            d[i] += d[i + w];
          }
        }
      vb[0] += e[0];
      if (!PROBS) {
        vb[1] += f[0];
        vb[2] += d[0];
      }
    }
  }
  vb[3] = static_cast<float>(s_timeout);
  {
    const int op[4] = {0, PROBS ? 1 : 0, 0, 1};
    rs_block_reduce<4>(vb, op, red[1]);
  }
  rs_exchange<4>(vb, xb, rank, CS);
  float Sp = 0.f, Sq = 0.f, Dq = 0.f, badq = 0.f, tmo = 0.f;
  for (uint32_t r = 0; r < CS; ++r) {
    Sp += xb[0][r];
    if (PROBS) badq = fmaxf(badq, xb[1][r]);
    else Sq += xb[1][r];
    Dq += xb[2][r];
    tmo = fmaxf(tmo, xb[3][r]);
  }
  const float lSp = __log2f(Sp), lSq = PROBS ? 0.f : __log2f(Sq);
  const float up = kp - lSp, uq = kq - lSq;   // log2 p = z c + up, log2 q = y c + uq

  // ---- pass C: alpha (and, for probabilities, TV and KL) ----------------------
  float vc[3] = {0.f, 0.f, 0.f};
  if constexpr (kPackedBF16) {
    const unsigned long long c2 = f2_pack(c, c), up2 = f2_pack(up, up), uq2 = f2_pack(uq, uq);
    unsigned long long al2 = f2_pack(0.f, 0.f);
    for (int g = threadIdx.x; g < ng; g += RS_THREADS) {
      const uint4 a4 = reinterpret_cast<const uint4*>(sp)[g], b4 = reinterpret_cast<const uint4*>(sq)[g];
      const uint32_t wz[4] = {a4.x, a4.y, a4.z, a4.w}, wy[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a0, a1, b0, b1;
        f2_unpack(f2_fma(bf16x2_to_f2(wz[i]), c2, up2), a0, a1);
        f2_unpack(f2_fma(bf16x2_to_f2(wy[i]), c2, uq2), b0, b1);
        al2 = f2_add(al2, f2_pack(ex2_approx(fminf(a0, b0)), ex2_approx(fminf(a1, b1))));
      }
    }
    float x0, x1;
    f2_unpack(al2, x0, x1);
    vc[0] = x0 + x1;
  } else {
    float zp[8], zq[8];
    for (int g = threadIdx.x; g < ng; g += RS_THREADS) {
      rs_ld8<TP>(sp, g, zp);
      rs_ld8<TQ>(sq, g, zq);
      float m[8], ad[8], k[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float lp = __fmaf_rn(zp[i], c, up);
        if (!PROBS) {
          m[i] = ex2_approx(fminf(lp, __fmaf_rn(zq[i], c, uq)));
        } else {
          const float p = ex2_approx(lp), q = zq[i];
          m[i] = fminf(p, q);
          ad[i] = fabsf(p - q);
          // q ln(q/p) = q (log2 q - log2 p) ln 2; q == 0 contributes nothing
          float lq;
          asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lq) : "f"(q));
          // subnormal q (flushed by lg2) contributes below 1e-36: skipped
          k[i] = q >= 1.17549435e-38f ? q * (lq - lp) : 0.f;
        }
      }
#pragma unroll
      for (int w = 1; w < 8; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < 8; i += 2 * w) {
          m[i] += m[i + w];
          if (PROBS) {
            ad[i] += ad[i + w];
            k[i] += k[i + w];
          }
        }
      vc[0] += m[0];
      if (PROBS) {
        vc[1] += ad[0];
        vc[2] += k[0];
      }
    }
  }
  {
    const int op[3] = {0, 0, 0};
    rs_block_reduce<3>(vc, op, red[2]);
  }
  // only rank 0 needs the totals: publish to it alone (it is alive until the
  // barrier below completes, and no CTA touches a peer after that barrier)
  if (threadIdx.x == 0)
#pragma unroll
    for (int k = 0; k < 3; ++k) st_peer_f32(&xc[k][rank], 0, vc[k]);
  cluster_sync_all();

  if (rank == 0 && threadIdx.x == 0) {
    float al = 0.f, tvs = 0.f, kls = 0.f;
    for (uint32_t r = 0; r < CS; ++r) {
      al += xc[0][r];
      tvs += xc[1][r];
      kls += xc[2][r];
    }
    float o_alpha, o_kl, o_tv;
    if (tmo > 0.f) {
      o_alpha = o_kl = o_tv = RS_TIMEOUT_MARK;
    } else if (!rows_ok || badq > 0.f || !(Sp > 0.f) || (!PROBS && !(Sq > 0.f))) {
      o_alpha = o_kl = o_tv = __int_as_float(0x7fc00000);
    } else if (!PROBS) {
      o_alpha = al;
      o_tv = 1.f - al;
      // ln2 (c D / S_q - fl(M_q c) + fl(M_p c) - log2 S_q + log2 S_p), combined in double
      const double l2 = 0.69314718055994530942;
      o_kl = static_cast<float>(l2 * (static_cast<double>(c) * Dq / Sq - static_cast<double>(Aq) +
                                      static_cast<double>(Ap) - log2(static_cast<double>(Sq)) +
                                      log2(static_cast<double>(Sp))));
    } else {
      o_alpha = al;
      o_tv = 0.5f * tvs;
      o_kl = 0.69314718f * kls;
    }
    a.alpha[pos] = o_alpha;
    a.kl[pos] = o_kl;
    a.tv[pos] = o_tv;
  }
  // a copy that outlived its wait must land before this CTA's shared memory goes away
  if (timed_out && threadIdx.x == 0) mbar_wait(&bar, 0, 1000000000ull);
}

}  // namespace sv
