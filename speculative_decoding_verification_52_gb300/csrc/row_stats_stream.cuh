// row_stats_stream.cuh -- the acceptance statistics of row_stats.cuh (alpha =
// sum_v min(p, q), KL(q || p) and TV per drafted position, "Speculative
// decoding: draft, verify, repeat", step 4) for draft logits whose rows can be
// streamed by bulk copies, without any exchange between CTAs.
//
// A persistent CTA (one per SM) takes position pairs (b, t) round-robin and
// reads each pair's target row t and draft row t twice, in chunks of E
// elements (RT_VPT 16-byte vectors per consumer thread and row) through a ring of
// RT_NS shared-memory stages filled by bulk async copies:
//   pass 1 (chunks in increasing order): per thread, online normalisers of
//     both rows (m, sum 2^(x c - fl(m c)), rescaled when m rises) and
//     D = sum e_q (y - z) relative to the draft offset, merged across the
//     CTA into M_p, S_p, M_q, S_q, D;
//   pass 2 (chunks in decreasing order, so the most recently read bytes come
//     first and are still in L2): alpha = sum 2^min(u_p, u_q) with
//     u = x c - fl(M c) - log2 S, the log2 of p and q (one exp per pair).
// KL(q || p) = ln2 (c D / S_q - fl(M_q c) + fl(M_p c) - log2 S_q + log2 S_p)
// and TV = 1 - alpha, as in row_stats.cuh.  A row is usable iff its maximum
// is finite and its sum positive (NaN anywhere makes the sum NaN; +inf makes
// the maximum infinite; an all -inf row has no finite maximum).
// The producer runs ahead into the next pair's first pass while the
// consumers finish the current pair's second pass.  Every wait is bounded;
// after a timeout every later wait of the CTA is skipped and its remaining
// pairs are marked RS_TIMEOUT_MARK.
#pragma once

#include "row_stats.cuh"

namespace sv {

constexpr int RT_CW = 16;                    // consumer warps
constexpr int RT_CT = RT_CW * 32;
constexpr int RT_THREADS = RT_CT + 32;       // + producer warp
constexpr int RT_VPT = 4;                    // 16-byte vectors per consumer thread, row and chunk
constexpr int RT_STAGE = 2 * RT_VPT * 16 * RT_CT;   // a chunk of the target row, then the same elements of the draft row
constexpr int RT_NS = 3;                     // ring stages (192 KB: one CTA per SM)
constexpr unsigned long long RT_WAIT_NS = 1000000000ull;

struct RtShared {
  uint64_t full[RT_NS];
  uint64_t empty[RT_NS];
  float red1[5][RT_CW];   // pass 1 per warp: M_p, S_p, M_q, S_q, D
  float red2[RT_CW];      // pass 2 per warp: alpha
  int abort;
};

__device__ __forceinline__ bool rt_aborted(const RtShared& sh) {
  return *reinterpret_cast<const volatile int*>(&sh.abort) != 0;
}

// The element count of a chunk: RT_VPT 16-byte vectors per consumer thread and row.
template <class T>
__device__ __forceinline__ constexpr int rt_chunk() {
  return RT_VPT * RT_CT * T::vpe;
}

// online normaliser of one row: m, s relative to fl(m c), with nA = -fl(m c)
// (0 while m == -inf); returns the factor the partial sums are rescaled by
__device__ __forceinline__ float rt_raise(float vm, float c, float& m, float& nA) {
  if (!(vm > m)) return 1.f;
  const float An = __fmul_rn(vm, c);
  const float f = (m == kNegInf) ? 0.f : ex2_approx(__fadd_rn(-nA, -An));
  m = vm;
  nA = -An;
  return f;
}

// the maximum of a thread's vectors of one row (fp32; NaN is skipped: it
// reaches the sums instead); bf16 words are reduced packed, then unpacked once
template <class T>
__device__ __forceinline__ float rt_vmax(const uint4 (&q)[RT_VPT]) {
  if constexpr (T::esz == 2) {
    uint32_t mx = bf16x2_max(bf16x2_max(q[0].x, q[0].y), bf16x2_max(q[0].z, q[0].w));
#pragma unroll
    for (int u = 1; u < RT_VPT; ++u)
      mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(q[u].x, q[u].y), bf16x2_max(q[u].z, q[u].w)));
    return fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
  } else {
    float m = kNegInf;
#pragma unroll
    for (int u = 0; u < RT_VPT; ++u)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(q[u].x), __uint_as_float(q[u].y)),
                         fmaxf(__uint_as_float(q[u].z), __uint_as_float(q[u].w))));
    return m;
  }
}

// the 32-bit words of a vector as fp32 pairs (two elements each for bf16; one
// pair per two words for fp32)
template <class T>
__device__ __forceinline__ unsigned long long rt_pair(const uint4& q, int i) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  if constexpr (T::esz == 2) return bf16x2_to_f2(w[i]);
  else return f2_pack(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}

template <class T>
__global__ void __launch_bounds__(RT_THREADS, 1) row_stats_stream_kernel(RowStatsArgs a) {
  extern __shared__ __align__(128) unsigned char rt_ring[];   // RT_NS * RT_STAGE bytes
  __shared__ RtShared sh;
  constexpr int E = rt_chunk<T>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int V = a.V, K = a.K;
  const int nch = (V + E - 1) / E;
  const long long npairs = static_cast<long long>(a.B) * K;
  if (threadIdx.x == 0) {
    for (int s = 0; s < RT_NS; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], RT_CW);
    }
    sh.abort = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == RT_CW) {
    // ---- producer ------------------------------------------------------------
    if (lane != 0) return;
    int stage = 0;
    uint32_t phase = 0;
    int last_parity[RT_NS];
#pragma unroll
    for (int s = 0; s < RT_NS; ++s) last_parity[s] = -1;
    bool ok = true;
    for (long long pr = blockIdx.x; pr < npairs && ok; pr += gridDim.x) {
      const long long b = pr / K, t = pr % K;
      const unsigned char* tp = a.target + (b * (K + 1) + t) * static_cast<long long>(V) * T::esz;
      const unsigned char* dp = a.draft + (b * K + t) * static_cast<long long>(V) * T::esz;
      for (int k = 0; k < 2 * nch && ok; ++k) {
        const int ch = k < nch ? k : 2 * nch - 1 - k;
        if (rt_aborted(sh) || !mbar_wait(&sh.empty[stage], phase ^ 1u, RT_WAIT_NS)) {
          *reinterpret_cast<volatile int*>(&sh.abort) = 1;
          ok = false;
          break;
        }
        const long long e0 = static_cast<long long>(ch) * E;
        const uint32_t bytes = static_cast<uint32_t>(min(static_cast<long long>(E), V - e0) * T::esz);
        mbar_arrive_expect_tx(&sh.full[stage], 2 * bytes);
        bulk_g2s(rt_ring + stage * RT_STAGE, tp + e0 * T::esz, bytes, &sh.full[stage]);
        bulk_g2s(rt_ring + stage * RT_STAGE + RT_STAGE / 2, dp + e0 * T::esz, bytes, &sh.full[stage]);
        last_parity[stage] = static_cast<int>(phase);
        if (++stage == RT_NS) { stage = 0; phase ^= 1u; }
      }
    }
    // do not leave while a copy may still land in this CTA's shared memory
#pragma unroll
    for (int s = 0; s < RT_NS; ++s)
      if (last_parity[s] >= 0) mbar_wait(&sh.full[s], static_cast<uint32_t>(last_parity[s]), RT_WAIT_NS);
    return;
  }

  // ---- consumers (16 warps) ---------------------------------------------------
  const int ctid = threadIdx.x;
  const float c = a.c;
  const unsigned long long c2 = f2_pack(c, c), m1 = f2_pack(-1.f, -1.f);
  const uint32_t ninf = T::esz == 2 ? 0xff80ff80u : __float_as_uint(kNegInf);
  const uint4 ninf4 = make_uint4(ninf, ninf, ninf, ninf);
  int stage = 0;
  uint32_t phase = 0;
  bool tmo = false;   // a wait of this warp ran out, or another's did (warp-uniform)
  // the next chunk's two vectors of this thread, or -inf past the row's end
  auto take = [&](int ch, uint4 (&zt)[RT_VPT], uint4 (&yt)[RT_VPT]) {
    if (!tmo) {   // warp-uniform: the warp consumes the stage, or none of it does
      const bool bad = __any_sync(0xffffffffu, rt_aborted(sh) || !mbar_wait(&sh.full[stage], phase, RT_WAIT_NS));
      if (bad) {
        *reinterpret_cast<volatile int*>(&sh.abort) = 1;
        tmo = true;
      }
    }
    const int nv = static_cast<int>(min(static_cast<long long>(E), V - static_cast<long long>(ch) * E)) / T::vpe;
    const uint4* tb = reinterpret_cast<const uint4*>(rt_ring + stage * RT_STAGE);
    const uint4* db = reinterpret_cast<const uint4*>(rt_ring + stage * RT_STAGE + RT_STAGE / 2);
    // (after a timeout the stage's bytes are garbage; the pair is marked anyway)
    if (nv == E / T::vpe) {   // a full chunk (all but a row's last): no bounds to test
#pragma unroll
      for (int u = 0; u < RT_VPT; ++u) {
        zt[u] = tb[ctid + u * RT_CT];
        yt[u] = db[ctid + u * RT_CT];
      }
    } else {
#pragma unroll
      for (int u = 0; u < RT_VPT; ++u) {
        const int v = ctid + u * RT_CT;
        zt[u] = v < nv ? tb[v] : ninf4;
        yt[u] = v < nv ? db[v] : ninf4;
      }
    }
    __syncwarp();
    if (lane == 0 && !tmo) mbar_arrive(&sh.empty[stage]);
    if (++stage == RT_NS) { stage = 0; phase ^= 1u; }
  };

  for (long long pr = blockIdx.x; pr < npairs; pr += gridDim.x) {
    // ---- pass 1: online normalisers and D ------------------------------------
    float mp = kNegInf, np = 0.f, mq = kNegInf, nq = 0.f;
    unsigned long long sp2 = f2_pack(0.f, 0.f), sq2 = sp2, d2 = sp2;
    for (int ch = 0; ch < nch; ++ch) {
      uint4 zt[RT_VPT], yt[RT_VPT];
      take(ch, zt, yt);
      const float vp = rt_vmax<T>(zt), vq = rt_vmax<T>(yt);
      const float fp = rt_raise(vp, c, mp, np);
      const float fq = rt_raise(vq, c, mq, nq);
      if (fp != 1.f) sp2 = f2_fma(sp2, f2_pack(fp, fp), f2_pack(0.f, 0.f));
      if (fq != 1.f) {
        const unsigned long long fq2 = f2_pack(fq, fq), z0 = f2_pack(0.f, 0.f);
        sq2 = f2_fma(sq2, fq2, z0);
        d2 = f2_fma(d2, fq2, z0);
      }
      const unsigned long long kp2 = f2_pack(np, np), kq2 = f2_pack(nq, nq);
#pragma unroll
      for (int j = 0; j < RT_VPT * T::vpe / 2; ++j) {
        const int u = j / (T::vpe / 2), i = j % (T::vpe / 2);
        const unsigned long long z2 = rt_pair<T>(zt[u], i), y2 = rt_pair<T>(yt[u], i);
        float a0, a1, b0, b1, t0, t1;
        f2_unpack(f2_fma(z2, c2, kp2), a0, a1);
        f2_unpack(f2_fma(y2, c2, kq2), b0, b1);
        const unsigned long long ep2 = f2_pack(ex2_approx(a0), ex2_approx(a1));
        const unsigned long long eq2 = f2_pack(ex2_approx(b0), ex2_approx(b1));
        sp2 = f2_add(sp2, ep2);
        sq2 = f2_add(sq2, eq2);
        // y - z >= -FLT_MAX: a -inf draft logit has e_q = 0 and adds nothing
        f2_unpack(f2_fma(z2, m1, y2), t0, t1);
        d2 = f2_fma(eq2, f2_pack(fmaxf(t0, -3.402823466e38f), fmaxf(t1, -3.402823466e38f)), d2);
      }
    }
    float sp, sq, dq;
    {
      float x0, x1;
      f2_unpack(sp2, x0, x1);
      sp = x0 + x1;
      f2_unpack(sq2, x0, x1);
      sq = x0 + x1;
      f2_unpack(d2, x0, x1);
      dq = x0 + x1;
    }
    // merge: the warp's maxima, each lane's sums rescaled to them, summed;
    // then the warps' through shared memory (every consumer thread merges)
    float Mp = mp, Mq = mq;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Mp = fmaxf(Mp, __shfl_xor_sync(0xffffffffu, Mp, o));
      Mq = fmaxf(Mq, __shfl_xor_sync(0xffffffffu, Mq, o));
    }
    {
      const float gp = (mp == kNegInf) ? 0.f : ex2_approx(__fsub_rn(-np, __fmul_rn(Mp, c)));
      const float gq = (mq == kNegInf) ? 0.f : ex2_approx(__fsub_rn(-nq, __fmul_rn(Mq, c)));
      sp *= gp;
      sq *= gq;
      dq *= gq;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sp += __shfl_xor_sync(0xffffffffu, sp, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      dq += __shfl_xor_sync(0xffffffffu, dq, o);
    }
    if (lane == 0) {
      sh.red1[0][warp] = Mp;
      sh.red1[1][warp] = sp;
      sh.red1[2][warp] = Mq;
      sh.red1[3][warp] = sq;
      sh.red1[4][warp] = dq;
    }
    named_bar_sync(1, RT_CT);
    tmo = rt_aborted(sh);   // (read by the whole warp after the barrier: warp-uniform)
    Mp = sh.red1[0][0];
    Mq = sh.red1[2][0];
#pragma unroll
    for (int w = 1; w < RT_CW; ++w) {
      Mp = fmaxf(Mp, sh.red1[0][w]);
      Mq = fmaxf(Mq, sh.red1[2][w]);
    }
    const float Ap = __fmul_rn(Mp, c), Aq = __fmul_rn(Mq, c);
    float Sp = 0.f, Sq = 0.f, Dq = 0.f;
#pragma unroll
    for (int w = 0; w < RT_CW; ++w) {
      const float wp = sh.red1[0][w], wq = sh.red1[2][w];
      const float gp = (wp == kNegInf) ? 0.f : ex2_approx(__fsub_rn(__fmul_rn(wp, c), Ap));
      const float gq = (wq == kNegInf) ? 0.f : ex2_approx(__fsub_rn(__fmul_rn(wq, c), Aq));
      Sp += sh.red1[1][w] * gp;
      Sq += sh.red1[3][w] * gq;
      Dq += sh.red1[4][w] * gq;
    }
    const bool rows_ok = isfinite(Mp) && isfinite(Mq);
    const float kp = rows_ok ? -Ap : 0.f, kq = rows_ok ? -Aq : 0.f;
    const float up = kp - __log2f(Sp), uq = kq - __log2f(Sq);   // log2 p = z c + up, log2 q = y c + uq

    // ---- pass 2: alpha ---------------------------------------------------------
    const unsigned long long up2 = f2_pack(up, up), uq2 = f2_pack(uq, uq);
    unsigned long long al2 = f2_pack(0.f, 0.f);
    for (int ch = nch - 1; ch >= 0; --ch) {
      uint4 zt[RT_VPT], yt[RT_VPT];
      take(ch, zt, yt);
#pragma unroll
      for (int j = 0; j < RT_VPT * T::vpe / 2; ++j) {
        const int u = j / (T::vpe / 2), i = j % (T::vpe / 2);
        float a0, a1, b0, b1;
        f2_unpack(f2_fma(rt_pair<T>(zt[u], i), c2, up2), a0, a1);
        f2_unpack(f2_fma(rt_pair<T>(yt[u], i), c2, uq2), b0, b1);
        al2 = f2_add(al2, f2_pack(ex2_approx(fminf(a0, b0)), ex2_approx(fminf(a1, b1))));
      }
    }
    float al;
    {
      float x0, x1;
      f2_unpack(al2, x0, x1);
      al = x0 + x1;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) al += __shfl_xor_sync(0xffffffffu, al, o);
    if (lane == 0) sh.red2[warp] = al;
    named_bar_sync(1, RT_CT);
    tmo = rt_aborted(sh);
    if (ctid == 0) {
      float alpha = 0.f;
#pragma unroll
      for (int w = 0; w < RT_CW; ++w) alpha += sh.red2[w];
      float o_alpha, o_kl, o_tv;
      if (tmo) {
        o_alpha = o_kl = o_tv = RS_TIMEOUT_MARK;
      } else if (!rows_ok || !(Sp > 0.f) || !(Sq > 0.f)) {
        o_alpha = o_kl = o_tv = __int_as_float(0x7fc00000);
      } else {
        o_alpha = alpha;
        o_tv = 1.f - alpha;
        // ln2 (c D / S_q - fl(M_q c) + fl(M_p c) - log2 S_q + log2 S_p), combined in double
        const double l2 = 0.69314718055994530942;
        o_kl = static_cast<float>(l2 * (static_cast<double>(c) * Dq / Sq - static_cast<double>(Aq) +
                                        static_cast<double>(Ap) - log2(static_cast<double>(Sq)) +
                                        log2(static_cast<double>(Sp))));
      }
      a.alpha[pr] = o_alpha;
      a.kl[pr] = o_kl;
      a.tv[pr] = o_tv;
    }
  }
}

}  // namespace sv
