// fused.cuh -- the whole sampling-mode verification step in one persistent
// kernel ("Speculative decoding and EAGLE", sections "The concept" and "The
// exactness rule"; "Speculative decoding: draft, verify, repeat", steps 1-3;
// "Speculative Decoding: from idea to SOTA", section 3).
//
// Work items, handed out dynamically (global atomic counters) to a grid of
// SMs x 3 CTAs:
//   sweep unit    (sequence b, row r, slice j): softmax-normaliser partial
//                 (max m, sum 2^(z*c - fl(m*c))) of one slice of one target or
//                 draft row.  Units are numbered sequence-major, so a sequence's
//                 units run at about the same time.
//   residual unit (sequence b, slice j): sum over one slice of the stopping
//                 row pair of w = max(0, p - q) (or p alone for the bonus row).
// Whichever CTA completes the last sweep unit of a sequence runs the accept
// scan for it (merging the partials in double precision), writes the accepted
// prefix, and publishes the sequence's residual units in a queue; producers
// take queued residual units before new sweep units, so the stopping rows are
// re-read while they are still in L2.  Whichever CTA completes the last
// residual unit of a sequence runs the inverse-CDF pick: it finds the slice
// holding u*R from the slice sums, re-reads that slice, and locates the token
// with a block-wide prefix scan.
//
// Inside a CTA: one producer thread streams each work item's bytes into a
// 4-stage ring of 16 KB shared-memory stages with 1-D bulk async copies
// (cp.async.bulk, completion on an mbarrier per stage) and writes a small
// descriptor per stage; eight consumer warps do the arithmetic.  Every wait
// (stage barriers, the consumer-group barrier, queue polling) is bounded in
// time; a timeout sets an error word and the last CTA to leave marks every
// sequence -2.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace sv {

constexpr int FU_CW = 8;
constexpr int FU_CT = FU_CW * 32;
constexpr int FU_THREADS = FU_CT + 32;
constexpr int FU_STAGE = 16384;
constexpr int FU_NSTAGE = 4;
constexpr int FU_MAX_ROWS = 2 * 31 + 1;
constexpr int FU_MAX_SR = 64;

enum : int { KIND_STOP = -1, KIND_SWEEP = 0, KIND_RESID = 1 };
enum : int { FL_FIRST = 1, FL_LAST = 2, FL_DRAFT = 4, FL_HASQ = 8 };

struct SeqInfo {          // per sequence, written by the accept scan
  int status, tstar;
  float AP, AQ;           // fl(row max * c) of the stopping target / draft rows
  float iSp, iSq;         // 1 / row sums (relative to AP / AQ); iSq = 1 for probabilities
  float u1;               // uniform of the replacement / bonus draw
  float pad;
};

struct FuCtl {            // zeroed before every call
  unsigned next;          // sweep units claimed
  unsigned rnext;         // residual units claimed
  unsigned rres;          // residual units reserved by finished scans
  unsigned err;           // a wait timed out
  unsigned done;          // CTAs that have left
  unsigned pad[3];
};

struct StageDesc {
  int kind, b, unit, e0, n, flags, status, tstar;
  float AP, AQ, iSp, iSq;
};

struct FusedArgs {
  const unsigned char* target;   // [B, K+1, V]
  const unsigned char* draft;    // [B, K, V] logits, or f32 probabilities
  const int32_t* tokens;         // [B, K]
  const float* uni;              // [B, K+1, 2]
  int B, K, V, RB;               // RB: sweep rows per sequence (2K+1 logits, K+1 probabilities)
  int S, L;                      // sweep slices per row and their length (elements)
  int Sr, Lr, RE;                // residual slices per row, their length, elements per stage
  unsigned U;                    // sweep units = B * RB * S
  float c;                       // log2(e) / T
  FuCtl* ctl;
  unsigned* cnt1;                // [B] sweep units completed
  unsigned* cnt2;                // [B] residual units completed
  unsigned* queue;               // [B * Sr] residual units: b * FU_MAX_SR + j + 1
  SeqInfo* info;                 // [B]
  double* rsum;                  // [B * Sr] residual slice sums
  float2* part;                  // [U] sweep partials
  int32_t* out_tokens;           // [B, K+1]
  int32_t* num_accepted;         // [B]
  int debug_b, debug_t;
  float* debug_row;
  float* debug_mass;
  unsigned long long timeout_ns;
};

struct FuShared {
  uint64_t full[FU_NSTAGE];
  uint64_t empty[FU_NSTAGE];
  uint64_t gbar;                 // consumer-group barrier (one arrival per consumer warp)
  StageDesc desc[FU_NSTAGE];
  float2 red2[FU_CW];
  double redd[FU_CW];
  double wsum[FU_CW];
  int flag_last;
  int abort;
  int pick, lastpos;
  // accept scan
  float rowA[FU_MAX_ROWS];
  double rowS[FU_MAX_ROWS];
  int rowState[FU_MAX_ROWS];
  float gp[32], gq[32], u0[32];
  int xt[32];
  // pick
  double sl[FU_MAX_SR];
  double base, target, R;
  int jstar, mode;
  SeqInfo inf;
};

__device__ __forceinline__ bool fu_aborted(const FuShared& sh) {
  return *reinterpret_cast<const volatile int*>(&sh.abort) != 0;
}
__device__ __forceinline__ void fu_set_abort(FuShared& sh) { *reinterpret_cast<volatile int*>(&sh.abort) = 1; }

// element loaders for 8 consecutive elements (16 B of bf16, 32 B of f32)
template <class T>
__device__ __forceinline__ void load8(const unsigned char* p, float* x);
template <>
__device__ __forceinline__ void load8<BF16T>(const unsigned char* p, float* x) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  BF16T::unpack(q, x);
}
template <>
__device__ __forceinline__ void load8<F32T>(const unsigned char* p, float* x) {
  const uint4 q0 = reinterpret_cast<const uint4*>(p)[0];
  const uint4 q1 = reinterpret_cast<const uint4*>(p)[1];
  F32T::unpack(q0, x);
  F32T::unpack(q1, x + 4);
}
template <class T>
__device__ __forceinline__ void load8_global(const unsigned char* p, float* x) {
  if constexpr (T::esz == 2) {
    const uint4 q = __ldcg(reinterpret_cast<const uint4*>(p));
    BF16T::unpack(q, x);
  } else {
    const uint4 q0 = __ldcg(reinterpret_cast<const uint4*>(p));
    const uint4 q1 = __ldcg(reinterpret_cast<const uint4*>(p) + 1);
    F32T::unpack(q0, x);
    F32T::unpack(q1, x + 4);
  }
}

// residual weight of one element, identical arithmetic in the slice sums and
// in the pick (so both see the same fp32 values)
__device__ __forceinline__ float resid_w(float zp, float zq, float c, float nAP, float nAQ, float iSp, float iSq,
                                         bool has_q, bool probs) {
  const float wp = __fmul_rn(ex2_approx(__fmaf_rn(zp, c, nAP)), iSp);
  if (!has_q) return wp;
  const float eq = probs ? zq : ex2_approx(__fmaf_rn(zq, c, nAQ));
  return fmaxf(0.f, __fmaf_rn(-eq, iSq, wp));
}

// ---------------------------------------------------------------------------
// consumer arithmetic on one ring stage
// ---------------------------------------------------------------------------
// softmax-normaliser partial over a sweep stage of bf16 elements: the stage
// max first (packed bf16x2 max), one rescale at most, then exp2 and sums on
// packed fp32 pairs
__device__ __forceinline__ void stats_stage_bf16(const uint4* buf, int nvec, int ctid, float c, StatsAcc& acc) {
  uint4 q[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int v = ctid + k * FU_CT;
    q[k] = v < nvec ? buf[v] : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  }
  uint32_t mx = bf16x2_max(bf16x2_max(q[0].x, q[0].y), bf16x2_max(q[0].z, q[0].w));
#pragma unroll
  for (int k = 1; k < 4; ++k)
    mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(q[k].x, q[k].y), bf16x2_max(q[k].z, q[k].w)));
  const float vm = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
  if (vm > acc.m) {
    const float An = __fmul_rn(vm, c);
    acc.s = (acc.m == kNegInf) ? 0.f : acc.s * ex2_approx(__fadd_rn(-acc.nA, -An));
    acc.m = vm;
    acc.nA = -An;
  }
  const unsigned long long c2 = f2_pack(c, c), n2 = f2_pack(acc.nA, acc.nA);
  unsigned long long s2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float a0, a1;
      f2_unpack(f2_fma(bf16x2_to_f2(w[i]), c2, n2), a0, a1);
      s2 = f2_add(s2, f2_pack(ex2_approx(a0), ex2_approx(a1)));
    }
  }
  float s0, s1;
  f2_unpack(s2, s0, s1);
  acc.s += s0 + s1;
}

__device__ __forceinline__ void stats_stage_f32(const uint4* buf, int nvec, int ctid, float c, StatsAcc& acc) {
  uint4 q[4];
  const uint32_t ni = __float_as_uint(kNegInf);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int v = ctid + k * FU_CT;
    q[k] = v < nvec ? buf[v] : make_uint4(ni, ni, ni, ni);
  }
  float vm = kNegInf;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    vm = fmaxf(vm, fmaxf(fmaxf(__uint_as_float(q[k].x), __uint_as_float(q[k].y)),
                         fmaxf(__uint_as_float(q[k].z), __uint_as_float(q[k].w))));
  if (vm > acc.m) {
    const float An = __fmul_rn(vm, c);
    acc.s = (acc.m == kNegInf) ? 0.f : acc.s * ex2_approx(__fadd_rn(-acc.nA, -An));
    acc.m = vm;
    acc.nA = -An;
  }
  const unsigned long long c2 = f2_pack(c, c), n2 = f2_pack(acc.nA, acc.nA);
  unsigned long long s2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a0, a1, a2, a3;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(q[k].x), __uint_as_float(q[k].y)), c2, n2), a0, a1);
    f2_unpack(f2_fma(f2_pack(__uint_as_float(q[k].z), __uint_as_float(q[k].w)), c2, n2), a2, a3);
    s2 = f2_add(s2, f2_pack(ex2_approx(a0), ex2_approx(a1)));
    s2 = f2_add(s2, f2_pack(ex2_approx(a2), ex2_approx(a3)));
  }
  float s0, s1;
  f2_unpack(s2, s0, s1);
  acc.s += s0 + s1;
}

template <class T>
__device__ __forceinline__ void stats_stage(const uint4* buf, int nvec, int ctid, float c, StatsAcc& acc) {
  if constexpr (T::esz == 2) stats_stage_bf16(buf, nvec, ctid, c, acc);
  else stats_stage_f32(buf, nvec, ctid, c, acc);
}

// residual partial sum over one stage: P chunk at buf, Q chunk at buf + RE*esz_P
template <class TP, class TQ, bool PROBS>
__device__ __forceinline__ float resid_stage(const unsigned char* buf, const StageDesc& d, int RE, int ctid, float c) {
  constexpr int QE = PROBS ? 4 : TQ::esz;
  const bool has_q = d.flags & FL_HASQ;
  const unsigned char* qb = buf + RE * TP::esz;
  float acc = 0.f;
  for (int g = ctid; g < d.n / 8; g += FU_CT) {
    float zp[8], zq[8];
    load8<TP>(buf + g * 8 * TP::esz, zp);
    if (has_q) {
      if constexpr (PROBS || QE == 4) load8<F32T>(qb + g * 8 * 4, zq);
      else load8<BF16T>(qb + g * 8 * 2, zq);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      acc += resid_w(zp[i], has_q ? zq[i] : 0.f, c, -d.AP, -d.AQ, d.iSp, d.iSq, has_q, PROBS);
  }
  return acc;
}

// ---------------------------------------------------------------------------
// consumer-group barrier on an mbarrier (bounded wait)
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool group_sync(FuShared& sh, uint32_t& gphase, uint64_t timeout) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.gbar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&sh.gbar, gphase, timeout));
  gphase ^= 1u;
  if (!ok) fu_set_abort(sh);
  return __all_sync(0xffffffffu, ok && !fu_aborted(sh));
}

// ---------------------------------------------------------------------------
// accept scan of sequence b (all consumer threads)
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS>
__device__ bool finish_scan(const FusedArgs& a, FuShared& sh, int b, int ctid, uint32_t& gphase) {
  const int K = a.K, W = K + 1, V = a.V;
  if (ctid < a.RB) {
    // merge the S slice partials of row ctid (double precision, offsets fl(m*c))
    const float2* part = a.part + (static_cast<long long>(b) * a.RB + ctid) * a.S;
    float M = kNegInf;
    bool poison = false;
    for (int j = 0; j < a.S; ++j) {
      const float2 p = __ldcg(part + j);
      if (p.x != p.x) poison = true;
      else M = fmaxf(M, p.x);
    }
    int st = 0;
    double Sr = 0.0;
    float AM = 0.f;
    if (poison) st = 2;
    else if (M == kNegInf) st = 1;
    else {
      AM = __fmul_rn(M, a.c);
      for (int j = 0; j < a.S; ++j) {
        const float2 p = __ldcg(part + j);
        if (p.x == kNegInf) continue;
        Sr += static_cast<double>(p.y) * exp2(static_cast<double>(__fmul_rn(p.x, a.c)) - static_cast<double>(AM));
      }
      st = (isfinite(Sr) && Sr > 0.0) ? 0 : 1;
    }
    sh.rowA[ctid] = AM;
    sh.rowS[ctid] = Sr;
    sh.rowState[ctid] = st;
  } else if (ctid >= 64 && ctid < 64 + K) {
    const int t = ctid - 64;
    const int x = a.tokens[static_cast<long long>(b) * K + t];
    sh.xt[t] = x;
    if (x >= 0 && x < V) {
      sh.gp[t] = TP::load(a.target, (static_cast<long long>(b) * W + t) * V + x);
      const long long oq = (static_cast<long long>(b) * K + t) * V + x;
      sh.gq[t] = PROBS ? F32T::load(a.draft, oq) : TQ::load(a.draft, oq);
    }
    sh.u0[t] = a.uni[(static_cast<long long>(b) * W + t) * 2];
  }
  if (!group_sync(sh, gphase, a.timeout_ns)) return false;
  if (ctid == 0) {
    int status = 0, tstar = K;
    for (int t = 0; t < K; ++t)
      if (sh.xt[t] < 0 || sh.xt[t] >= V) status = -1;
    const bool forced = (b == a.debug_b);
    const double cd = static_cast<double>(a.c);
    for (int t = 0; status == 0 && !forced && t < K; ++t) {
      if (sh.rowState[t] != 0) { status = sh.rowState[t] == 2 ? -2 : -1; break; }
      const double pa = exp2(static_cast<double>(sh.gp[t]) * cd - static_cast<double>(sh.rowA[t])) / sh.rowS[t];
      double qc;
      if (PROBS) {
        const float qv = sh.gq[t];
        if (qv != qv || qv < 0.f) { status = -1; break; }
        qc = static_cast<double>(qv);
      } else {
        const int r = W + t;
        if (sh.rowState[r] != 0) { status = sh.rowState[r] == 2 ? -2 : -1; break; }
        qc = exp2(static_cast<double>(sh.gq[t]) * cd - static_cast<double>(sh.rowA[r])) / sh.rowS[r];
      }
      const bool accept = (qc == 0.0) || (static_cast<double>(sh.u0[t]) < pa / qc);
      if (!accept) { tstar = t; break; }
    }
    if (forced) tstar = a.debug_t;
    if (status == 0 && sh.rowState[tstar] != 0) status = sh.rowState[tstar] == 2 ? -2 : -1;
    if (status == 0 && tstar < K && !PROBS && sh.rowState[W + tstar] != 0)
      status = sh.rowState[W + tstar] == 2 ? -2 : -1;
    SeqInfo inf;
    inf.status = status;
    inf.tstar = tstar;
    inf.AP = sh.rowA[tstar];
    inf.iSp = static_cast<float>(1.0 / sh.rowS[tstar]);
    const bool has_q = tstar < K;
    inf.AQ = (has_q && !PROBS) ? sh.rowA[W + tstar] : 0.f;
    inf.iSq = (has_q && !PROBS) ? static_cast<float>(1.0 / sh.rowS[W + tstar]) : 1.f;
    inf.u1 = a.uni[(static_cast<long long>(b) * W + tstar) * 2 + 1];
    inf.pad = 0.f;
    int32_t* out = a.out_tokens + static_cast<long long>(b) * W;
    for (int j = 0; j < W; ++j) out[j] = (status == 0 && j < tstar) ? sh.xt[j] : -1;
    a.num_accepted[b] = status == 0 ? tstar : status;
    a.info[b] = inf;
    __threadfence();
    const unsigned k0 = atomicAdd(&a.ctl->rres, static_cast<unsigned>(a.Sr));
    for (int j = 0; j < a.Sr; ++j) st_release_u32(a.queue + k0 + j, static_cast<unsigned>(b * FU_MAX_SR + j + 1));
  }
  return group_sync(sh, gphase, a.timeout_ns);
}

// ---------------------------------------------------------------------------
// inverse-CDF pick of sequence b (all consumer threads)
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS>
__device__ bool finish_pick(const FusedArgs& a, FuShared& sh, int b, int ctid, uint32_t& gphase) {
  constexpr int QE = PROBS ? 4 : TQ::esz;
  const int K = a.K, W = K + 1, V = a.V;
  const int lane = ctid & 31, warp = ctid >> 5;
  if (ctid == 0) {
    SeqInfo inf;
    const int* src = reinterpret_cast<const int*>(a.info + b);
    int* dst = reinterpret_cast<int*>(&inf);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = __ldcg(src + i);
    sh.inf = inf;
  }
  if (ctid < a.Sr) sh.sl[ctid] = __ldcg(a.rsum + static_cast<long long>(b) * a.Sr + ctid);
  if (!group_sync(sh, gphase, a.timeout_ns)) return false;
  const SeqInfo inf = sh.inf;
  if (inf.status != 0) return true;   // outputs already written by the scan
  const bool has_q0 = inf.tstar < K;
  const unsigned char* prow = a.target + (static_cast<long long>(b) * W + inf.tstar) * V * TP::esz;
  const unsigned char* qrow = has_q0 ? a.draft + (static_cast<long long>(b) * K + inf.tstar) * V * QE : nullptr;
  const float c = a.c;

  // residual mass zero: recompute the slice sums for w = p (rare)
  bool has_q = has_q0;
  for (int pass = 0; pass < 2; ++pass) {
    if (ctid == 0) {
      double R = 0.0;
      for (int j = 0; j < a.Sr; ++j) R += sh.sl[j];
      sh.R = R;
      sh.mode = (R > 0.0 || !has_q) ? 0 : 1;
      const double target = static_cast<double>(inf.u1) * R;
      int js = -1, jlast = -1;
      double pre = 0.0, base = 0.0;
      for (int j = 0; j < a.Sr; ++j) {
        if (sh.sl[j] > 0.0) {
          jlast = j;
          if (js < 0 && pre + sh.sl[j] > target) { js = j; base = pre; }
        }
        pre += sh.sl[j];
      }
      if (js < 0) {  // rounding: fall back to the last slice with mass
        js = jlast;
        base = 0.0;
        for (int j = 0; j < jlast; ++j) base += sh.sl[j];
      }
      sh.jstar = js;
      sh.base = base;
      sh.target = target;
      sh.pick = 0x7fffffff;
      sh.lastpos = -1;
    }
    if (!group_sync(sh, gphase, a.timeout_ns)) return false;
    if (sh.mode == 0) break;
    has_q = false;
    for (int j = 0; j < a.Sr; ++j) {
      const int e0 = j * a.Lr, e1 = min(V, e0 + a.Lr);
      float acc = 0.f;
      for (int g = e0 / 8 + ctid; g < e1 / 8; g += FU_CT) {
        float zp[8];
        load8_global<TP>(prow + static_cast<long long>(g) * 8 * TP::esz, zp);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc += resid_w(zp[i], 0.f, c, -inf.AP, 0.f, inf.iSp, 1.f, false, PROBS);
      }
      double v = static_cast<double>(acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) sh.wsum[warp] = v;
      if (!group_sync(sh, gphase, a.timeout_ns)) return false;
      if (ctid == 0) {
        double t = 0.0;
        for (int w = 0; w < FU_CW; ++w) t += sh.wsum[w];
        sh.sl[j] = t;
      }
      if (!group_sync(sh, gphase, a.timeout_ns)) return false;
    }
  }
  const int js = sh.jstar;
  int pick = -1;
  if (js >= 0) {
    const int e0 = js * a.Lr;
    const int n = min(V, e0 + a.Lr) - e0;
    int seg = (n + FU_CT - 1) / FU_CT;
    seg = (seg + 7) / 8 * 8;
    const int k0 = min(n, ctid * seg), k1 = min(n, k0 + seg);
    float Tt = 0.f;
    int lastpos = -1;
    for (int k = k0; k < k1; k += 8) {
      float zp[8], zq[8];
      load8_global<TP>(prow + static_cast<long long>(e0 + k) * TP::esz, zp);
      if (has_q) load8_global<typename std::conditional<QE == 4, F32T, BF16T>::type>(
          qrow + static_cast<long long>(e0 + k) * QE, zq);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float w = resid_w(zp[i], has_q ? zq[i] : 0.f, c, -inf.AP, -inf.AQ, inf.iSp, inf.iSq, has_q, PROBS);
        Tt += w;
        if (w > 0.f) lastpos = e0 + k + i;
      }
    }
    double x = static_cast<double>(Tt);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sh.wsum[warp] = x;
    int lp = lastpos;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
    if (lane == 0 && lp >= 0) atomicMax(&sh.lastpos, lp);
    if (!group_sync(sh, gphase, a.timeout_ns)) return false;
    double wex = 0.0;
    for (int w = 0; w < warp; ++w) wex += sh.wsum[w];
    const double base = sh.base + wex + (x - static_cast<double>(Tt));
    const double target = sh.target;
    if (Tt > 0.f && base <= target && base + static_cast<double>(Tt) > target) {
      float run = 0.f;
      for (int k = k0; k < k1; k += 8) {
        float zp[8], zq[8];
        load8_global<TP>(prow + static_cast<long long>(e0 + k) * TP::esz, zp);
        if (has_q) load8_global<typename std::conditional<QE == 4, F32T, BF16T>::type>(
            qrow + static_cast<long long>(e0 + k) * QE, zq);
        int found = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float w = resid_w(zp[i], has_q ? zq[i] : 0.f, c, -inf.AP, -inf.AQ, inf.iSp, inf.iSq, has_q, PROBS);
          run += w;
          if (found < 0 && base + static_cast<double>(run) > target) found = i;
        }
        if (found >= 0) {
          atomicMin(&sh.pick, e0 + k + found);
          break;
        }
      }
    }
    if (!group_sync(sh, gphase, a.timeout_ns)) return false;
    pick = (sh.pick != 0x7fffffff) ? sh.pick : sh.lastpos;
  }
  if (ctid == 0) a.out_tokens[static_cast<long long>(b) * W + inf.tstar] = pick;
  if (b == a.debug_b && sh.R > 0.0) {
    const double R = sh.R;
    for (int g = ctid; g < V / 8; g += FU_CT) {
      float zp[8], zq[8];
      load8_global<TP>(prow + static_cast<long long>(g) * 8 * TP::esz, zp);
      if (has_q) load8_global<typename std::conditional<QE == 4, F32T, BF16T>::type>(
          qrow + static_cast<long long>(g) * 8 * QE, zq);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float w = resid_w(zp[i], has_q ? zq[i] : 0.f, c, -inf.AP, -inf.AQ, inf.iSp, inf.iSq, has_q, PROBS);
        a.debug_row[g * 8 + i] = static_cast<float>(static_cast<double>(w) / R);
      }
    }
    if (ctid == 0) *a.debug_mass = static_cast<float>(R);
  }
  return group_sync(sh, gphase, a.timeout_ns);
}

// ---------------------------------------------------------------------------
// producer (one thread)
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS>
__device__ void fu_producer(const FusedArgs& a, unsigned char* ring, FuShared& sh) {
  constexpr int QE = PROBS ? 4 : TQ::esz;
  int stage = 0;
  uint32_t phase = 0;
  int last_parity[FU_NSTAGE];
#pragma unroll
  for (int s = 0; s < FU_NSTAGE; ++s) last_parity[s] = -1;
  const unsigned RU = static_cast<unsigned>(a.B) * static_cast<unsigned>(a.Sr);
  const unsigned per_seq = static_cast<unsigned>(a.RB) * static_cast<unsigned>(a.S);
  const int W = a.K + 1;
  bool sweep_done = false;

  auto next_stage = [&]() -> bool {
    if (fu_aborted(sh)) return false;
    if (!mbar_wait(&sh.empty[stage], phase ^ 1u, a.timeout_ns)) {
      fu_set_abort(sh);
      atomicOr(&a.ctl->err, 1u);
      return false;
    }
    return true;
  };
  auto advance = [&]() {
    if (++stage == FU_NSTAGE) { stage = 0; phase ^= 1u; }
  };

  bool ok = true;
  while (ok) {
    // 1. a queued residual unit, if one is ready
    long long rid = -1;
    unsigned rn = *reinterpret_cast<volatile unsigned*>(&a.ctl->rnext);
    unsigned rr = *reinterpret_cast<volatile unsigned*>(&a.ctl->rres);
    for (int tries = 0; tries < 8 && rn < rr; ++tries) {
      const unsigned prev = atomicCAS(&a.ctl->rnext, rn, rn + 1);
      if (prev == rn) { rid = rn; break; }
      rn = prev;
      rr = *reinterpret_cast<volatile unsigned*>(&a.ctl->rres);
    }
    // 2. otherwise a sweep unit
    long long uid = -1;
    if (rid < 0 && !sweep_done) {
      const unsigned u = atomicAdd(&a.ctl->next, 1u);
      if (u < a.U) uid = u;
      else sweep_done = true;
    }
    // 3. sweep exhausted: the next residual unit, waiting for it if needed
    if (rid < 0 && uid < 0) {
      const unsigned r = atomicAdd(&a.ctl->rnext, 1u);
      if (r >= RU) break;
      rid = r;
    }
    if (uid >= 0) {
      const unsigned u = static_cast<unsigned>(uid);
      const int b = static_cast<int>(u / per_seq);
      const unsigned rem = u - static_cast<unsigned>(b) * per_seq;
      const int row = static_cast<int>(rem / a.S);
      const int j = static_cast<int>(rem - static_cast<unsigned>(row) * a.S);
      const bool is_draft = row >= W;
      const int esz = is_draft ? QE : TP::esz;
      const unsigned char* src =
          is_draft ? a.draft + ((static_cast<long long>(b) * a.K + (row - W)) * a.V) * esz
                   : a.target + ((static_cast<long long>(b) * W + row) * a.V) * esz;
      const int e0 = j * a.L, e1 = min(a.V, e0 + a.L);
      const uint32_t bytes = static_cast<uint32_t>((e1 - e0) * esz);
      for (uint32_t off = 0; off < bytes; off += FU_STAGE) {
        const uint32_t n = min(static_cast<uint32_t>(FU_STAGE), bytes - off);
        if (!next_stage()) { ok = false; break; }
        StageDesc& d = sh.desc[stage];
        d.kind = KIND_SWEEP;
        d.b = b;
        d.unit = static_cast<int>(u);
        d.e0 = e0 + static_cast<int>(off) / esz;
        d.n = static_cast<int>(n);   // bytes for sweep stages
        d.flags = (off == 0 ? FL_FIRST : 0) | (off + n >= bytes ? FL_LAST : 0) | (is_draft ? FL_DRAFT : 0);
        mbar_arrive_expect_tx(&sh.full[stage], n);
        bulk_g2s(ring + stage * FU_STAGE, src + e0 * esz + off, n, &sh.full[stage]);
        last_parity[stage] = static_cast<int>(phase);
        advance();
      }
      continue;
    }
    // residual unit rid: wait for its queue entry (written by a finished scan)
    unsigned ent = ld_acquire_u32(a.queue + rid);
    if (ent == 0) {
      const uint64_t t0 = global_ns();
      while ((ent = ld_acquire_u32(a.queue + rid)) == 0) {
        if (fu_aborted(sh) || global_ns() - t0 > a.timeout_ns) break;
        __nanosleep(256);
      }
      if (ent == 0) {
        fu_set_abort(sh);
        atomicOr(&a.ctl->err, 2u);
        break;
      }
    }
    const int b = static_cast<int>((ent - 1) / FU_MAX_SR);
    const int j = static_cast<int>((ent - 1) % FU_MAX_SR);
    SeqInfo inf;
    {
      const int* src = reinterpret_cast<const int*>(a.info + b);
      int* dst = reinterpret_cast<int*>(&inf);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = __ldcg(src + i);
    }
    if (inf.status != 0) {
      if (!next_stage()) break;
      StageDesc& d = sh.desc[stage];
      d.kind = KIND_RESID;
      d.b = b;
      d.unit = j;
      d.e0 = 0;
      d.n = 0;
      d.flags = FL_FIRST | FL_LAST;
      d.status = inf.status;
      mbar_arrive(&sh.full[stage]);
      // the stage was released, so its previous copy has landed: nothing to drain
      last_parity[stage] = -1;
      advance();
      continue;
    }
    const bool has_q = inf.tstar < a.K;
    const unsigned char* prow = a.target + ((static_cast<long long>(b) * W + inf.tstar) * a.V) * TP::esz;
    const unsigned char* qrow = has_q ? a.draft + ((static_cast<long long>(b) * a.K + inf.tstar) * a.V) * QE : nullptr;
    const int e0 = j * a.Lr, e1 = min(a.V, e0 + a.Lr);
    for (int e = e0; e < e1; e += a.RE) {
      const int n = min(a.RE, e1 - e);
      if (!next_stage()) { ok = false; break; }
      StageDesc& d = sh.desc[stage];
      d.kind = KIND_RESID;
      d.b = b;
      d.unit = j;
      d.e0 = e;
      d.n = n;   // elements for residual stages
      d.flags = (e == e0 ? FL_FIRST : 0) | (e + n >= e1 ? FL_LAST : 0) | (has_q ? FL_HASQ : 0);
      d.status = 0;
      d.tstar = inf.tstar;
      d.AP = inf.AP;
      d.AQ = inf.AQ;
      d.iSp = inf.iSp;
      d.iSq = inf.iSq;
      const uint32_t bp = static_cast<uint32_t>(n * TP::esz), bq = has_q ? static_cast<uint32_t>(n * QE) : 0u;
      mbar_arrive_expect_tx(&sh.full[stage], bp + bq);
      unsigned char* dst = ring + stage * FU_STAGE;
      bulk_g2s(dst, prow + static_cast<long long>(e) * TP::esz, bp, &sh.full[stage]);
      if (has_q) bulk_g2s(dst + a.RE * TP::esz, qrow + static_cast<long long>(e) * QE, bq, &sh.full[stage]);
      last_parity[stage] = static_cast<int>(phase);
      advance();
    }
  }
  // stop marker for the consumers
  if (next_stage()) {
    sh.desc[stage].kind = KIND_STOP;
    mbar_arrive(&sh.full[stage]);
    last_parity[stage] = -1;
  }
  // Do not leave while a copy may still land in this CTA's shared memory.  A
  // stage's recorded parity is that of its last copy; any later arrival on the
  // stage (which would flip the phase again) clears the record, so a wait here
  // can only be for a copy that has not been consumed yet (abort path).
#pragma unroll
  for (int s = 0; s < FU_NSTAGE; ++s)
    if (last_parity[s] >= 0 && !mbar_wait(&sh.full[s], static_cast<uint32_t>(last_parity[s]), a.timeout_ns))
      atomicOr(&a.ctl->err, 8u);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
constexpr size_t fu_smem_bytes() { return FU_NSTAGE * FU_STAGE + sizeof(FuShared) + 128; }

template <class TP, class TQ, bool PROBS>
__global__ void __launch_bounds__(FU_THREADS, 3) fused_sample_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) unsigned char fu_smem[];
  unsigned char* ring = fu_smem;
  FuShared& sh = *reinterpret_cast<FuShared*>(fu_smem + FU_NSTAGE * FU_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < FU_NSTAGE; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], FU_CW);
    }
    mbar_init(&sh.gbar, FU_CW);
    sh.abort = 0;
    sh.pick = 0x7fffffff;
    sh.lastpos = -1;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) fu_producer<TP, TQ, PROBS>(a, ring, sh);
  } else {
    const int ctid = threadIdx.x - 32, cw = warp - 1;
    int stage = 0;
    uint32_t phase = 0, gphase = 0;
    StatsAcc sacc;
    sacc.init();
    float racc = 0.f;
    const unsigned per_seq = static_cast<unsigned>(a.RB) * static_cast<unsigned>(a.S);
    for (;;) {
      if (__any_sync(0xffffffffu, fu_aborted(sh))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(&sh.full[stage], phase, a.timeout_ns))) {
        fu_set_abort(sh);
        atomicOr(&a.ctl->err, 4u);
        break;
      }
      const StageDesc d = sh.desc[stage];
      if (d.kind == KIND_STOP) break;
      if (d.flags & FL_FIRST) {
        sacc.init();
        racc = 0.f;
      }
      const unsigned char* buf = ring + stage * FU_STAGE;
      if (d.kind == KIND_SWEEP) {
        if (d.flags & FL_DRAFT) {
          if constexpr (!PROBS) stats_stage<TQ>(reinterpret_cast<const uint4*>(buf), d.n >> 4, ctid, a.c, sacc);
        } else {
          stats_stage<TP>(reinterpret_cast<const uint4*>(buf), d.n >> 4, ctid, a.c, sacc);
        }
      } else if (d.n > 0) {
        racc += resid_stage<TP, TQ, PROBS>(buf, d, a.RE, ctid, a.c);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[stage]);
      if (++stage == FU_NSTAGE) { stage = 0; phase ^= 1u; }
      if (!(d.flags & FL_LAST)) continue;

      // ---- end of a work unit: reduce across the consumer warps ----------
      if (d.kind == KIND_SWEEP) {
        sacc.warp_reduce(a.c);
        if (lane == 0) sh.red2[cw] = sacc.pack();
      } else {
        double v = static_cast<double>(racc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sh.redd[cw] = v;
      }
      if (!group_sync(sh, gphase, a.timeout_ns)) break;
      if (cw == 0) {
        if (d.kind == KIND_SWEEP) {
          StatsAcc t;
          t.init();
          if (lane < FU_CW) t.unpack(sh.red2[lane]);
          t.warp_reduce(a.c);
          if (lane == 0) {
            a.part[d.unit] = t.pack();
            __threadfence();
            const unsigned old = atomicAdd(&a.cnt1[d.b], 1u);
            sh.flag_last = (old + 1u == per_seq);
            if (sh.flag_last) __threadfence();
          }
        } else if (lane == 0) {
          double tot = 0.0;
          for (int w = 0; w < FU_CW; ++w) tot += sh.redd[w];
          a.rsum[static_cast<long long>(d.b) * a.Sr + d.unit] = d.n > 0 ? tot : 0.0;
          __threadfence();
          const unsigned old = atomicAdd(&a.cnt2[d.b], 1u);
          sh.flag_last = (old + 1u == static_cast<unsigned>(a.Sr));
          if (sh.flag_last) __threadfence();
        }
      }
      if (!group_sync(sh, gphase, a.timeout_ns)) break;
      if (__shfl_sync(0xffffffffu, sh.flag_last, 0)) {
        const bool ok = d.kind == KIND_SWEEP ? finish_scan<TP, TQ, PROBS>(a, sh, d.b, ctid, gphase)
                                             : finish_pick<TP, TQ, PROBS>(a, sh, d.b, ctid, gphase);
        if (!ok) break;
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned left = atomicAdd(&a.ctl->done, 1u);
    if (left + 1u == gridDim.x) {
      __threadfence();
      if (ld_acquire_u32(&a.ctl->err) != 0u) {
        const int W = a.K + 1;
        for (long long i = 0; i < static_cast<long long>(a.B) * W; ++i) a.out_tokens[i] = -1;
        for (int b = 0; b < a.B; ++b) a.num_accepted[b] = -2;
      }
    }
  }
}

}  // namespace sv
