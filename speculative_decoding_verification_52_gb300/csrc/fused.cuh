// fused.cuh -- the whole sampling-mode verification step in one persistent
// kernel ("Speculative decoding and EAGLE", sections "The concept" and "The
// exactness rule"; "Speculative decoding: draft, verify, repeat", steps 1-3;
// "Speculative Decoding: from idea to SOTA", section 3).
//
// Work items (sweep units claimed from one counter in unit order; residual
// units dealt round-robin to the CTAs):
//   sweep unit    (sequence b, row r, slice j): softmax-normaliser partials
//                 (max m, sum 2^(z*c - fl(m*c))) of one slice of one target or
//                 draft row, numbered sequence-major so the batch is swept in
//                 roughly sequence order.
//   residual unit (sequence b, slice j): the residual weights w = max(0, p - q)
//                 (p alone for the bonus row) of one slice of the stopping row
//                 pair, summed per block of 256 elements.  A producer takes its
//                 next residual unit as soon as sequence b is ready (its accept
//                 scan is done), ahead of its next sweep unit, so a finished
//                 sequence's draw does not wait behind the rest of the sweep.
// Roles inside a CTA:
//   producer   (1 thread) streams work-item bytes into a ring of FU_NSTAGE 16 KB
//              shared-memory stages with 1-D bulk async copies (cp.async.bulk,
//              completion counted on an mbarrier per stage) and writes a small
//              descriptor per stage.
//   consumers  (FU_CW warps) each reduce their share of every stage.  At the
//              end of a work item every warp leaves its partial in shared
//              memory and the warps count themselves there; the last one hands
//              a sweep unit to the merger warp, or adds a residual unit to the
//              sequence's counter with a fire-and-forget release reduction.
//   merger     (1 warp) clears this CTA's share of the control block before the
//              grid barrier; then merges the warp partials of completed sweep
//              units, stores each unit's partial and adds it to the sequence's
//              counter (release), off the consumers' path, and polls the
//              readiness word of the sequence the producer wants residual units
//              of.
//   finisher   (1 warp) owns a fixed set of sequences: the accept scan of b runs
//              on CTA b mod grid, the pick of b on CTA (b + grid/2) mod grid.
//              It polls those sequences' counters; the scan merges the partials
//              (warp-parallel), tests all positions at once (one lane each),
//              writes the accepted prefix and marks the sequence ready; the
//              pick finds the 256-element block holding u*R from the block
//              sums, re-reads that block, and locates the token with a
//              warp-wide prefix scan.
// The fixed roles above (owner CTAs of scans and picks, residual units dealt
// round-robin) need every CTA of the grid resident at once.  The kernel is
// therefore launched cooperatively: a grid that cannot be resident fails at
// launch instead of leaving resident CTAs waiting on CTAs that never start.
// The kernel clears its own control block (each CTA a share) and meets at one
// bounded grid barrier, so a call needs no memset; each producer's first
// FU_STATIC_UNITS sweep units need no claim and stream while the barrier
// completes.
// Every wait (stage barriers, the grid barrier, readiness and counter polling)
// is bounded in time; a timeout sets an error word, and the last CTA to leave
// then marks every sequence -2.
#pragma once

#include <cooperative_groups.h>

#include <type_traits>

#include "common.cuh"

namespace sv {

constexpr int FU_CW = 8;                          // consumer warps (4 vectors each per stage)
constexpr int FU_CT = FU_CW * 32;
constexpr int FU_THREADS = FU_CT + 96;            // + producer, merger and finisher warps
constexpr int FU_MERGE_WARP = FU_CW + 1;
constexpr int FU_FIN_WARP = FU_CW + 2;
constexpr int FU_STAGE = 16384;
constexpr int FU_VPT = (FU_STAGE / 16 + FU_CT - 1) / FU_CT;   // 16-byte vectors per consumer thread per stage
static_assert((FU_VPT - 1) * FU_CT <= FU_STAGE / 16, "a full stage covers every consumer thread's first FU_VPT-1 vectors");
constexpr int FU_NSTAGE = 4;
constexpr int FU_CTAS_PER_SM = 3;
constexpr int FU_MAX_GRID = 1024;                 // persistent grid cap
constexpr int FU_BLK = 256;                       // residual block (elements)
// Per-sequence flags (units swept, residual units done, ready) share one
// block of FU_FLAG_STRIDE words, so different sequences' polled words sit in
// different 32-byte sectors.
constexpr int FU_FLAG_STRIDE = 8;
constexpr int FU_IDLE_NS = 256;                   // finisher's sleep between idle polls
constexpr int FU_WSLOTS = 16;                     // sweep units whose warp partials await their merge
constexpr int FU_STATIC_UNITS = 3;                // sweep units per CTA taken without a claim (blockIdx + k * grid)

enum : int { KIND_STOP = -1, KIND_SWEEP = 0, KIND_RESID = 1 };
enum : int { FL_FIRST = 1, FL_LAST = 2, FL_DRAFT = 4, FL_HASQ = 8 };

struct SeqInfo {          // per sequence, written by the accept scan
  float AP, AQ;           // fl(row max * c) of the stopping target / draft rows
  float iSp, iSq;         // 1 / row sums (relative to AP / AQ); iSq = 1 for probabilities
  int status, tstar;
  float u1;               // uniform of the replacement / bonus draw
  float pad;
};
static_assert(sizeof(SeqInfo) == 32, "SeqInfo: the residual scales are its first 16 bytes");

// The readiness word of a sequence, written (release) by its accept scan:
// bit 31 set, bit 8 = the sequence is invalid, bits 0-7 = the stopping position.
__device__ __forceinline__ unsigned fu_ready_word(int status, int tstar) {
  return 0x80000000u | (status != 0 ? 0x100u : 0u) | static_cast<unsigned>(tstar);
}

struct FuCtl {            // cleared by the kernel before its grid barrier (32 bytes reserved)
  unsigned err;           // a wait timed out
  unsigned done;          // CTAs that have left
  unsigned claim;         // sweep units claimed by the producers beyond the static ones, in unit order
};
static_assert(sizeof(FuCtl) <= 32, "control block must fit its 32-byte slot");

struct StageDesc {
  int kind, b, unit, e0, n, flags, slot, pad;   // slot: partial slot of a sweep unit
};

struct FusedArgs {
  const unsigned char* target;   // [B, K+1, V]
  const unsigned char* draft;    // [B, K, V] logits, or f32 probabilities
  const int32_t* tokens;         // [B, K]
  const float* uni;              // [B, K+1, 2]
  int B, K, V, RB;               // RB: sweep rows per sequence (2K+1 logits, K+1 probabilities)
  int S, L;                      // sweep slices per row and their length (elements)
  int Sr, Lr, RE;                // residual slices per row, their length, elements per stage
  int NB;                        // residual blocks per row = ceil(V / 256)
  unsigned U;                    // sweep units = B * RB * S
  float c;                       // log2(e) / T
  unsigned zero_words;           // 16-byte words of [ctl | flags] the kernel clears
  FuCtl* ctl;
  unsigned* flags;               // [B * FU_FLAG_STRIDE]: per sequence, words 0 (sweep units completed),
                                 // 1 (residual units completed), 2 (1 once the accept scan wrote SeqInfo)
  SeqInfo* info;                 // [B]
  float* bsum;                   // [B * NB] residual block sums
  float4* part;                  // [U] sweep-unit partials (m, hi, lo, 0): sum = hi + lo relative to fl(m*c)
  int32_t* out_tokens;           // [B, K+1]
  int32_t* num_accepted;         // [B]
  int debug_b, debug_t;
  int debug_stall_b;             // test hook: this sequence's scan waits for a unit that never comes (-1: off)
  float* debug_row;
  float* debug_mass;
  unsigned long long timeout_ns;
};

struct FuShared {
  uint64_t full[FU_NSTAGE];
  uint64_t empty[FU_NSTAGE];
  StageDesc desc[FU_NSTAGE];
  int unit_cnt[FU_NSTAGE];       // consumer warps done with the work item ending in this stage
  float4 stage_info[FU_NSTAGE];  // residual stages: the sequence's (AP, AQ, iSp, iSq), copied in with the data
  float2 wpart[FU_WSLOTS][FU_CW];   // warp partials of completed sweep units, merged by the merger warp
  int slot_unit[FU_WSLOTS];      // unit id + 1 once its partials are complete; 0 = free
  int units_issued;              // sweep units the producer issued (-1 while it is running)
  unsigned res_word;             // readiness word of sequence res_have
  int res_want;                  // sequence of the producer's next residual unit (-1: none)
  int res_have;                  // sequence whose readiness word is in res_word (-1: none)
  int grid_ready;                // the control block is cleared on every CTA (set by the merger warp)
  float4 scan_scratch[32];       // the finisher's per-lane row shares during an accept scan
  int abort;
};

__device__ __forceinline__ unsigned* fu_cnt1(const FusedArgs& a, int b) { return a.flags + b * FU_FLAG_STRIDE; }
__device__ __forceinline__ unsigned* fu_cnt2(const FusedArgs& a, int b) { return a.flags + b * FU_FLAG_STRIDE + 1; }
__device__ __forceinline__ unsigned* fu_ready(const FusedArgs& a, int b) { return a.flags + b * FU_FLAG_STRIDE + 2; }

__device__ __forceinline__ bool fu_aborted(const FuShared& sh) {
  return *reinterpret_cast<const volatile int*>(&sh.abort) != 0;
}
__device__ __forceinline__ void fu_fail(FuShared& sh, FuCtl* ctl, unsigned bit) {
  *reinterpret_cast<volatile int*>(&sh.abort) = 1;
  atomicOr(&ctl->err, bit);
}

// Wait (bounded) until the merger warp has seen the grid barrier pass, i.e.
// every CTA has cleared its share of the control block.
__device__ __forceinline__ bool fu_wait_grid(FuShared& sh, unsigned long long timeout_ns) {
  if (*reinterpret_cast<volatile int*>(&sh.grid_ready) != 0) return true;
  const uint64_t t0 = global_ns();
  while (*reinterpret_cast<volatile int*>(&sh.grid_ready) == 0) {
    if (fu_aborted(sh) || global_ns() - t0 > timeout_ns) return false;
    __nanosleep(64);
  }
  return true;
}

// One grid-wide barrier on the barrier word the driver provides to
// cooperative launches (its flip-bit protocol: CTA 0 adds 2^31 - (G - 1), the
// others 1, so bit 31 flips once all G have arrived).  Called by one thread
// per CTA; gives up after timeout_ns and returns false.
__device__ __forceinline__ bool fu_grid_barrier(unsigned long long timeout_ns) {
  namespace cg = cooperative_groups;
  cg::details::grid_workspace* ws = cg::details::get_grid_workspace();
  if (ws == nullptr) return false;   // not a cooperative launch
  unsigned* bar = &ws->barrier;
  const unsigned nb = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1u) : 1u;
  unsigned old;
  asm volatile("atom.add.release.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(bar), "r"(nb) : "memory");
  const uint64_t t0 = global_ns();
  for (;;) {
    if (((old ^ ld_acquire_u32(bar)) & 0x80000000u) != 0u) return true;
    if (global_ns() - t0 > timeout_ns) return false;
    __nanosleep(128);
  }
}

// element loaders for 8 consecutive elements (16 B of bf16, 32 B of f32)
template <class T>
__device__ __forceinline__ void load8_smem(const unsigned char* p, float* x) {
  if constexpr (T::esz == 2) {
    BF16T::unpack(*reinterpret_cast<const uint4*>(p), x);
  } else {
    F32T::unpack(reinterpret_cast<const uint4*>(p)[0], x);
    F32T::unpack(reinterpret_cast<const uint4*>(p)[1], x + 4);
  }
}
template <class T>
__device__ __forceinline__ void load8_global(const unsigned char* p, float* x) {
  if constexpr (T::esz == 2) {
    BF16T::unpack(__ldcg(reinterpret_cast<const uint4*>(p)), x);
  } else {
    F32T::unpack(__ldcg(reinterpret_cast<const uint4*>(p)), x);
    F32T::unpack(__ldcg(reinterpret_cast<const uint4*>(p) + 1), x + 4);
  }
}

// residual weight of one element; the block sums and the pick use exactly this
// arithmetic (and the same 8-element sequential sums), so both see the same
// fp32 values
__device__ __forceinline__ float resid_w(float zp, float zq, float c, float nAP, float nAQ, float iSp, float iSq,
                                         bool has_q, bool probs) {
  const float wp = __fmul_rn(ex2_approx(__fmaf_rn(zp, c, nAP)), iSp);
  if (!has_q) return wp;
  const float eq = probs ? zq : ex2_approx(__fmaf_rn(zq, c, nAQ));
  return fmaxf(0.f, __fmaf_rn(-eq, iSq, wp));
}

// error-free sum of two floats: (s, e) with s + e == a + b exactly (Knuth)
__device__ __forceinline__ float2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return make_float2(s, e);
}

// Float-float numbers (hi + lo, |lo| <= ulp(hi)/2): ~48 significant bits on
// the fp32 pipes.  The finishing warps sum, scan and compare in this form;
// GB300's fp64 rate is a small fraction of its fp32 rate, and these steps sit
// on the latency path at the end of every launch.
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_norm(float hi, float lo) {   // |hi| >= |lo|
  const float s = __fadd_rn(hi, lo);
  return FF{s, __fsub_rn(lo, __fsub_rn(s, hi))};
}
__device__ __forceinline__ FF ff_add_f(FF a, float b) {
  const float2 t = two_sum(a.hi, b);
  return ff_norm(t.x, __fadd_rn(t.y, a.lo));
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float2 t = two_sum(a.hi, b.hi);
  return ff_norm(t.x, __fadd_rn(t.y, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ FF ff_sub(FF a, FF b) { return ff_add(a, FF{-b.hi, -b.lo}); }
__device__ __forceinline__ FF ff_mul_f(FF a, float b) {
  const float p = __fmul_rn(a.hi, b);
  const float e = __fmaf_rn(a.hi, b, -p);   // the product's rounding error, exactly
  return ff_norm(p, __fmaf_rn(a.lo, b, e));
}
// a > b
__device__ __forceinline__ bool ff_gt(FF a, FF b) {
  return __fadd_rn(__fsub_rn(a.hi, b.hi), __fsub_rn(a.lo, b.lo)) > 0.f;
}
__device__ __forceinline__ float ff_to_f(FF a) { return __fadd_rn(a.hi, a.lo); }
__device__ __forceinline__ FF ff_shfl_xor(FF a, int o) {
  return FF{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ FF ff_shfl_up(FF a, int o) {
  return FF{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ FF ff_shfl(FF a, int l) {
  return FF{__shfl_sync(0xffffffffu, a.hi, l), __shfl_sync(0xffffffffu, a.lo, l)};
}

// 2^(z*c - A) for an fp32 logit z, c = log2(e)/T and A = fl(M*c): the exponent
// is formed exactly as a float-float (the product's error by fma, the
// difference by two-sum), then the accurate fp32 exp2f of its leading part is
// corrected to first order for the remainder (~1e-7 relative accuracy)
__device__ __forceinline__ float exp2_arg_ff(float z, float c, float A) {
  const float p = __fmul_rn(z, c);
  const float pe = __fmaf_rn(z, c, -p);
  const float2 x = two_sum(p, -A);
  const float r = __fadd_rn(x.y, pe);
  return __fmul_rn(exp2f(x.x), __fmaf_rn(r, 0.69314718f, 1.f));
}

// ---------------------------------------------------------------------------
// consumer arithmetic on one ring stage
// ---------------------------------------------------------------------------
// softmax-normaliser partial over a sweep stage of bf16 elements: the stage
// max first (packed bf16x2 max), one rescale at most, then exp2 and sums on
// packed fp32 pairs
__device__ __forceinline__ void stats_stage_bf16(const uint4* buf, int nvec, int ctid, float c, StatsAcc& acc) {
  uint4 q[FU_VPT];
  if (nvec == FU_STAGE / 16) {   // a full stage: only the last vector may lie past its end
#pragma unroll
    for (int k = 0; k < FU_VPT; ++k) {
      const int v = ctid + k * FU_CT;
      q[k] = (k + 1 < FU_VPT || v < FU_STAGE / 16) ? buf[v]
                                                    : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    }
  } else {
#pragma unroll
    for (int k = 0; k < FU_VPT; ++k) {
      const int v = ctid + k * FU_CT;
      q[k] = v < nvec ? buf[v] : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    }
  }
  uint32_t mx = bf16x2_max(bf16x2_max(q[0].x, q[0].y), bf16x2_max(q[0].z, q[0].w));
#pragma unroll
  for (int k = 1; k < FU_VPT; ++k)
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
  for (int k = 0; k < FU_VPT; ++k) {
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
  uint4 q[FU_VPT];
  const uint32_t ni = __float_as_uint(kNegInf);
#pragma unroll
  for (int k = 0; k < FU_VPT; ++k) {
    const int v = ctid + k * FU_CT;
    q[k] = v < nvec ? buf[v] : make_uint4(ni, ni, ni, ni);
  }
  float vm = kNegInf;
#pragma unroll
  for (int k = 0; k < FU_VPT; ++k)
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
  for (int k = 0; k < FU_VPT; ++k) {
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

// Residual weights of one stage (P chunk at buf, Q chunk at buf + RE*esz_P),
// summed per 256-element block: warp cw covers elements [256*(8k + cw), +256)
// of the stage in its k-th pass (lane l: 8 consecutive elements), so each
// block sum is one warp reduction of the lanes' sequential 8-element sums.
template <class TP, class TQ, bool PROBS>
__device__ __forceinline__ void resid_stage(const unsigned char* buf, const StageDesc& d, float4 sc, int RE, int cw,
                                            int lane, float c, float* bsum_row) {
  using QT = typename std::conditional<PROBS, F32T, TQ>::type;
  const bool has_q = d.flags & FL_HASQ;
  const unsigned char* qb = buf + RE * TP::esz;
  const int ngroups = d.n / 8;
  for (int k = 0; k * FU_CT * 8 < RE; ++k) {
    const int g0 = FU_CT * k + 32 * cw;   // first 8-element group of this warp's block
    if (g0 >= ngroups) break;
    const int g = g0 + lane;
    float s = 0.f;
    if (g < ngroups) {
      float zp[8], zq[8];
      load8_smem<TP>(buf + g * 8 * TP::esz, zp);
      if (has_q) load8_smem<QT>(qb + g * 8 * QT::esz, zq);
#pragma unroll
      for (int i = 0; i < 8; ++i) s += resid_w(zp[i], has_q ? zq[i] : 0.f, c, -sc.x, -sc.y, sc.z, sc.w, has_q, PROBS);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) bsum_row[(d.e0 + g0 * 8) / FU_BLK] = s;
  }
}

// ---------------------------------------------------------------------------
// finisher: accept scan of sequence b (one warp)
// ---------------------------------------------------------------------------
template <class T>
__device__ __forceinline__ T row_get(const T (&v)[2], int r) {   // row r lives in lane r & 31, slot r >> 5
  const T v0 = __shfl_sync(0xffffffffu, v[0], r & 31);
  const T v1 = __shfl_sync(0xffffffffu, v[1], r & 31);
  return r < 32 ? v0 : v1;
}
__device__ __forceinline__ FF row_get_ff(const FF (&v)[2], int r) {
  const FF v0 = ff_shfl(v[0], r & 31);
  const FF v1 = ff_shfl(v[1], r & 31);
  return r < 32 ? v0 : v1;
}

// Inputs of position `lane` of sequence b that do not depend on the sweep:
// the drafted token, its target and draft logits (or draft probability) and
// the accept and draw uniforms.  The finisher loads them while it waits for the
// sequence's sweep to complete.
struct ScanInputs {
  int x;
  float zp, zq, u0, u1;   // u1: the replacement-draw uniform of position `lane` (lanes 0..K)
};

template <class TP, class TQ, bool PROBS>
__device__ __forceinline__ ScanInputs scan_inputs(const FusedArgs& a, int b, int lane) {
  const int K = a.K, W = K + 1, V = a.V;
  ScanInputs in{-1, 0.f, 0.f, 0.f, 0.f};
  if (lane < W) in.u1 = a.uni[(static_cast<long long>(b) * W + lane) * 2 + 1];
  if (lane < K) {
    in.x = a.tokens[static_cast<long long>(b) * K + lane];
    in.u0 = a.uni[(static_cast<long long>(b) * W + lane) * 2];
    if (in.x >= 0 && in.x < V) {
      const long long oq = (static_cast<long long>(b) * K + lane) * V + in.x;
      in.zp = TP::load(a.target, (static_cast<long long>(b) * W + lane) * V + in.x);
      in.zq = PROBS ? F32T::load(a.draft, oq) : TQ::load(a.draft, oq);
    }
  }
  return in;
}

// Merge the 8 warp partials (m, s) of a sweep unit into one float-float
// partial (M, hi, lo): sum = hi + lo relative to fl(M*c).  Lanes 0-7 hold one
// partial each (the others (-inf, 0)); the whole warp calls it.
__device__ __forceinline__ float4 merge_unit(float2 p, int lane, float c) {
  const bool nan = __any_sync(0xffffffffu, p.x != p.x);
  float M = p.x;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float hi = 0.f, lo = 0.f;
  if (!nan && M != kNegInf && p.x != kNegInf) {
    // fl(m*c) - fl(M*c) is exact in fp32 whenever the factor is not negligible
    const float f = exp2f(__fmul_rn(p.x, c) - __fmul_rn(M, c));
    hi = p.y * f;
    lo = fmaf(p.y, f, -hi);   // the product's rounding error, exactly
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    const float2 t = two_sum(hi, h2);
    hi = t.x;
    lo = lo + (l2 + t.y);
  }
  return make_float4(nan ? __int_as_float(0x7fc00000) : M, hi, lo, 0.f);
}

// Online float-float accumulation of normaliser partials (m, hi, lo): the
// running maximum M and the sum hi + lo relative to fl(M*c).  A NaN partial
// poisons the accumulation; partials of only -inf elements add nothing.
struct RowAcc {
  float M, hi, lo;
  bool bad;
};
__device__ __forceinline__ void row_acc_add(RowAcc& s, float4 u, float c) {
  if (u.x != u.x) {
    s.bad = true;
    return;
  }
  if (u.x == kNegInf) return;
  if (u.x > s.M) {
    if (s.M != kNegInf) {
      const float f = exp2f(__fmul_rn(s.M, c) - __fmul_rn(u.x, c));
      const float h = s.hi * f;
      s.lo = fmaf(s.hi, f, -h) + s.lo * f;
      s.hi = h;
    }
    s.M = u.x;
  }
  const float f = exp2f(__fmul_rn(u.x, c) - __fmul_rn(s.M, c));
  const float h = u.y * f;
  const float2 t = two_sum(s.hi, h);
  s.hi = t.x;
  s.lo += t.y + fmaf(u.y, f, -h) + u.z * f;
}

// The row's scale, sum and state (0 valid, 1 invalid: no finite entry or a
// non-positive or infinite sum, 2 poisoned) from its accumulation.
__device__ __forceinline__ void row_acc_result(const RowAcc& s, float c, float& A, FF& S, int& st) {
  const FF acc = ff_norm(s.hi, s.lo);
  A = (s.bad || s.M == kNegInf) ? 0.f : __fmul_rn(s.M, c);
  S = acc;
  st = s.bad ? 2 : (s.M == kNegInf ? 1 : ((isfinite(acc.hi) && acc.hi > 0.f) ? 0 : 1));
}

// Accumulate the unit partials j0, j0 + step, ... of one row (one lane).
__device__ __forceinline__ RowAcc merge_share(const float4* up, int j0, int step, int S, float c) {
  RowAcc s{kNegInf, 0.f, 0.f, false};
#pragma unroll 4
  for (int j = j0; j < S; j += step) row_acc_add(s, __ldcg(up + j), c);
  return s;
}

// Merge the unit partials of every row of sequence b.  Small batches split
// rows into many slices (one ring stage each), so with at most 16 rows of more
// than 4 slices each row gets lpr = min(32 / rows, S) lanes that accumulate a
// strided share of its slices; the shares meet in the scratch in shared
// memory, where lane r combines row r's.  Otherwise lane r merges rows r and
// r + 32 alone.  Row r lands in slot r >> 5 of lane r & 31.  (The kernel's
// sweep rate proved sensitive to the size of this rarely run code, so both
// forms share one accumulation routine.)
__device__ __forceinline__ void merge_rows(const FusedArgs& a, int b, int lane, float4* scratch, float (&Ar)[2],
                                           FF (&Sr)[2], int (&st)[2]) {
  const int RB = a.RB, S = a.S;
  const float c = a.c;
  const int lpr = (RB <= 16 && S > 4) ? max(1, min(32 / RB, S)) : 1;
  if (lpr == 1) {
    for (int r = lane; r < RB; r += 32) {
      const RowAcc s = merge_share(a.part + (static_cast<long long>(b) * RB + r) * S, 0, 1, S, c);
      row_acc_result(s, c, Ar[r >> 5], Sr[r >> 5], st[r >> 5]);
    }
    return;
  }
  const int r = lane / lpr;
  RowAcc s{kNegInf, 0.f, 0.f, false};
  if (r < RB) s = merge_share(a.part + (static_cast<long long>(b) * RB + r) * S, lane - r * lpr, lpr, S, c);
  // a poisoned share travels as a NaN maximum
  scratch[lane] = make_float4(s.bad ? __int_as_float(0x7fc00000) : s.M, s.hi, s.lo, 0.f);
  __syncwarp();
  if (lane < RB) {
    RowAcc t{kNegInf, 0.f, 0.f, false};
    for (int k = 0; k < lpr; ++k) row_acc_add(t, scratch[lane * lpr + k], c);
    row_acc_result(t, c, Ar[0], Sr[0], st[0]);
  }
  __syncwarp();
}

template <class TP, class TQ, bool PROBS>
__device__ void finish_scan(const FusedArgs& a, int b, int lane, const ScanInputs& in, float4* scratch) {
  const int K = a.K, W = K + 1, V = a.V;
  const int x = in.x;
  const float u0 = in.u0;
  float Ar[2] = {0.f, 0.f};
  FF Sr[2] = {FF{0.f, 0.f}, FF{0.f, 0.f}};
  int st[2] = {1, 1};
  // lane r merges row r (and row r + 32 when there are more than 32 rows)
  merge_rows(a, b, lane, scratch, Ar, Sr, st);

  // lane t tests position t
  const int t = lane;
  const int rp = t < W ? t : 0;
  const int rq = (t < K && !PROBS) ? W + t : 0;
  const float At = row_get(Ar, rp), Aq = row_get(Ar, rq);
  const FF St = row_get_ff(Sr, rp), Sq = row_get_ff(Sr, rq);
  const int stt = row_get(st, rp), stq = row_get(st, rq);
  bool tok_bad = false, acc_t = true;
  int row_bad = 0;   // rows read at position t: 0 ok, 1 invalid, 2 poisoned
  if (t < K) {
    tok_bad = x < 0 || x >= V;
    row_bad = stt;
    if (!PROBS && row_bad == 0) row_bad = stq;
    if (!tok_bad && row_bad == 0) {
      // accept iff q(x) == 0 or u < p(x)/q(x), with p(x) = ep / St and q(x) = eq / Sq:
      // u * St * eq < ep * Sq, no division (float-float products)
      const float zpf = in.zp, zqf = in.zq;
      const float ep = exp2_arg_ff(zpf, a.c, At);
      float eq;
      FF Sqq;
      if (PROBS) {
        if (zqf != zqf || zqf < 0.f) row_bad = 1;
        eq = zqf;
        Sqq = FF{1.f, 0.f};
      } else {
        eq = exp2_arg_ff(zqf, a.c, Aq);
        Sqq = Sq;
      }
      acc_t = (eq == 0.f) || ff_gt(ff_mul_f(Sqq, ep), ff_mul_f(ff_mul_f(St, u0), eq));
    }
  }
  const unsigned badtok = __ballot_sync(0xffffffffu, t < K && tok_bad);
  // the scan stops at the first rejection or at the first position whose rows are bad
  const unsigned stop = __ballot_sync(0xffffffffu, t < K && (row_bad != 0 || !acc_t));
  int tstar = stop ? (__ffs(stop) - 1) : K;
  const int rb_at = __shfl_sync(0xffffffffu, row_bad, tstar & 31);
  int status = badtok ? -1 : 0;
  if (b == a.debug_b) {
    tstar = a.debug_t;
  } else if (status == 0 && tstar < K && rb_at != 0) {
    status = rb_at == 2 ? -2 : -1;
  }
  // the replacement draw reads the stopping rows
  const int sp_state = row_get(st, tstar);
  if (status == 0 && sp_state != 0) status = sp_state == 2 ? -2 : -1;
  const bool has_q = tstar < K && !PROBS;
  const int sq_state = row_get(st, has_q ? W + tstar : 0);
  if (status == 0 && has_q && sq_state != 0) status = sq_state == 2 ? -2 : -1;
  const float Ap = row_get(Ar, tstar);
  const FF Sp = row_get_ff(Sr, tstar);
  const float Aq2 = row_get(Ar, has_q ? W + tstar : 0);
  const FF Sq2 = row_get_ff(Sr, has_q ? W + tstar : 0);

  const float u1 = __shfl_sync(0xffffffffu, in.u1, tstar);
  // accepted prefix (slot tstar is written by the pick), -1 padding
  int32_t* out = a.out_tokens + static_cast<long long>(b) * W;
  const int x_all = x;
  for (int j = lane; j < W; j += 32) {
    const int xj = (j < 32) ? x_all : a.tokens[static_cast<long long>(b) * K + j];
    out[j] = (status == 0 && j < tstar) ? xj : -1;
  }
  if (lane == 0) {
    a.num_accepted[b] = status == 0 ? tstar : status;
    SeqInfo inf;
    inf.status = status;
    inf.tstar = tstar;
    inf.AP = Ap;
    inf.AQ = has_q ? Aq2 : 0.f;
    inf.iSp = __frcp_rn(ff_to_f(Sp));   // scales of the residual weights: fp32 suffices
    inf.iSq = has_q ? __frcp_rn(ff_to_f(Sq2)) : 1.f;
    inf.u1 = u1;
    inf.pad = 0.f;
    a.info[b] = inf;
  }
  // the warp's writes are ordered before lane 0's release by the warp barrier
  __syncwarp();
  if (lane == 0) st_release_u32(fu_ready(a, b), fu_ready_word(status, tstar));
}

// ---------------------------------------------------------------------------
// finisher: inverse-CDF pick of sequence b (one warp)
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS>
__device__ void finish_pick(const FusedArgs& a, int b, int lane) {
  using QT = typename std::conditional<PROBS, F32T, TQ>::type;
  const int K = a.K, W = K + 1, V = a.V, NB = a.NB;
  const int nbl = (NB + 31) / 32;               // blocks per lane (contiguous)
  const int bl0 = min(NB, lane * nbl), bl1 = min(NB, bl0 + nbl);
  float* brow = a.bsum + static_cast<long long>(b) * NB;
  // the sequence's info and this lane's block sums in one round of loads
  SeqInfo inf;
  {
    const int* src = reinterpret_cast<const int*>(a.info + b);
    int* dst = reinterpret_cast<int*>(&inf);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = __ldcg(src + i);
  }
  constexpr int kRegBlocks = 16;   // block sums kept in registers per lane (V <= 131072)
  float bv[kRegBlocks];
#pragma unroll
  for (int k = 0; k < kRegBlocks; ++k) bv[k] = (bl0 + k < bl1) ? __ldcg(brow + bl0 + k) : 0.f;
  FF lsum{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kRegBlocks; ++k) lsum = ff_add_f(lsum, bv[k]);
  for (int k = bl0 + kRegBlocks; k < bl1; ++k) lsum = ff_add_f(lsum, __ldcg(brow + k));
  if (inf.status != 0) return;   // outputs already written by the scan
  const unsigned char* prow = a.target + (static_cast<long long>(b) * W + inf.tstar) * V * TP::esz;
  const unsigned char* qrow =
      inf.tstar < K ? a.draft + (static_cast<long long>(b) * K + inf.tstar) * V * QT::esz : nullptr;
  bool has_q = inf.tstar < K;
  const float c = a.c;

  auto weights8 = [&](int e, float* w) {   // w of the 8 elements at e (e % 8 == 0)
    float zp[8], zq[8];
    load8_global<TP>(prow + static_cast<long long>(e) * TP::esz, zp);
    if (has_q) load8_global<QT>(qrow + static_cast<long long>(e) * QT::esz, zq);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = resid_w(zp[i], has_q ? zq[i] : 0.f, c, -inf.AP, -inf.AQ, inf.iSp, inf.iSq, has_q, PROBS);
  };

  FF R{0.f, 0.f};
  for (int pass = 0; pass < 2; ++pass) {
    if (pass > 0) {
      lsum = FF{0.f, 0.f};
#pragma unroll
      for (int k = 0; k < kRegBlocks; ++k) {
        bv[k] = (bl0 + k < bl1) ? __ldcg(brow + bl0 + k) : 0.f;
        lsum = ff_add_f(lsum, bv[k]);
      }
      for (int k = bl0 + kRegBlocks; k < bl1; ++k) lsum = ff_add_f(lsum, __ldcg(brow + k));
    }
    R = lsum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) R = ff_add(R, ff_shfl_xor(R, o));
    if (R.hi > 0.f || !has_q) break;
    // residual mass zero: draw from p_t instead (rebuild the block sums; rare)
    has_q = false;
    for (int blk = 0; blk < NB; ++blk) {
      const int e = blk * FU_BLK + 8 * lane;
      float s = 0.f;
      if (e < V) {
        float w[8];
        weights8(e, w);
#pragma unroll
        for (int i = 0; i < 8; ++i) s += w[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) brow[blk] = s;
    }
    __syncwarp();
    __threadfence_block();
  }
  const FF target = ff_mul_f(R, inf.u1);
  // exclusive prefix of the lanes' block ranges, then the block holding the target
  FF incl = lsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF y = ff_shfl_up(incl, o);
    if (lane >= o) incl = ff_add(incl, y);
  }
  int jb = -1, jlast = -1;
  FF jbase{0.f, 0.f}, lastbase{0.f, 0.f};
  {
    FF run = ff_shfl_up(incl, 1);
    if (lane == 0) run = FF{0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kRegBlocks; ++k) {
      const float v = bv[k];
      const FF nxt = ff_add_f(run, v);
      if (v > 0.f) {
        jlast = bl0 + k;
        lastbase = run;
        if (jb < 0 && ff_gt(nxt, target)) { jb = bl0 + k; jbase = run; }
      }
      run = nxt;
    }
    for (int k = bl0 + kRegBlocks; k < bl1; ++k) {
      const float v = __ldcg(brow + k);
      const FF nxt = ff_add_f(run, v);
      if (v > 0.f) {
        jlast = k;
        lastbase = run;
        if (jb < 0 && ff_gt(nxt, target)) { jb = k; jbase = run; }
      }
      run = nxt;
    }
  }
  const unsigned hit = __ballot_sync(0xffffffffu, jb >= 0);
  const unsigned pos = __ballot_sync(0xffffffffu, jlast >= 0);
  int src_lane;
  bool exact = true;
  if (hit) src_lane = __ffs(hit) - 1;
  else if (pos) { src_lane = 31 - __clz(pos); exact = false; }   // rounding: last block with mass
  else src_lane = -1;
  int pick = -1;
  if (src_lane >= 0) {
    const int blk = __shfl_sync(0xffffffffu, exact ? jb : jlast, src_lane);
    const FF bb = ff_shfl(exact ? jbase : lastbase, src_lane);
    // re-read the block: lane l holds elements blk*256 + 8l .. +8
    const int e = blk * FU_BLK + 8 * lane;
    float w[8];
    float s = 0.f;
    if (e < V) {
      weights8(e, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) s += w[i];
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = 0.f;
    }
    FF x2{s, 0.f};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const FF y = ff_shfl_up(x2, o);
      if (lane >= o) x2 = ff_add(x2, y);
    }
    FF ex = ff_shfl_up(x2, 1);
    if (lane == 0) ex = FF{0.f, 0.f};
    const FF lb = ff_add(bb, ex);
    int cand = 0x7fffffff, lastpos = -1;
    if (s > 0.f && !ff_gt(lb, target) && ff_gt(ff_add_f(lb, s), target)) {
      // the lane holding the target: search its 8 weights against the
      // remaining mass (in fp32; the lane's own sum is exact enough here)
      const float rem = ff_to_f(ff_sub(target, lb));
      float run = 0.f;
      int lastw = -1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        run += w[i];
        if (cand == 0x7fffffff && run > rem) cand = e + i;
        if (w[i] > 0.f) lastw = e + i;
      }
      if (cand == 0x7fffffff) cand = lastw;   // rounding at the lane's end: its last element with weight
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (w[i] > 0.f) lastpos = e + i;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
      lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
    }
    pick = cand != 0x7fffffff ? cand : lastpos;
  }
  if (lane == 0) a.out_tokens[static_cast<long long>(b) * W + inf.tstar] = pick;
  if (b == a.debug_b && R.hi > 0.f) {
    for (int e = 8 * lane; e < V; e += 256) {
      float w[8];
      weights8(e, w);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        a.debug_row[e + i] =
            static_cast<float>(static_cast<double>(w[i]) / (static_cast<double>(R.hi) + static_cast<double>(R.lo)));
    }
    if (lane == 0) *a.debug_mass = ff_to_f(R);
  }
}

// ---------------------------------------------------------------------------
// producer (one thread)
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS>
__device__ void fu_producer(const FusedArgs& a, unsigned char* ring, FuShared& sh) {
  using QT = typename std::conditional<PROBS, F32T, TQ>::type;
  int stage = 0;
  uint32_t phase = 0;
  int last_parity[FU_NSTAGE];
#pragma unroll
  for (int s = 0; s < FU_NSTAGE; ++s) last_parity[s] = -1;
  const unsigned RU = static_cast<unsigned>(a.B) * static_cast<unsigned>(a.Sr);
  const unsigned per_seq = static_cast<unsigned>(a.RB) * static_cast<unsigned>(a.S);
  const int W = a.K + 1;
  const unsigned G = gridDim.x;
  unsigned next_res = blockIdx.x;
  // The finisher warp watches the readiness of the sequence of this CTA's next
  // residual unit and hands its readiness word (stopping position, validity)
  // over in shared memory, so the producer never waits on a global load: it
  // only reads sh.res_have / sh.res_word.
  auto want_next = [&]() {
    *reinterpret_cast<volatile int*>(&sh.res_want) = next_res < RU ? static_cast<int>(next_res / a.Sr) : -1;
  };
  auto res_is_ready = [&]() -> bool {
    return next_res < RU && *reinterpret_cast<volatile int*>(&sh.res_have) == static_cast<int>(next_res / a.Sr);
  };
  want_next();

  auto next_stage = [&]() -> bool {
    if (fu_aborted(sh)) return false;
    if (!mbar_wait(&sh.empty[stage], phase ^ 1u, a.timeout_ns)) {
      fu_fail(sh, a.ctl, 1u);
      return false;
    }
    return true;
  };
  auto advance = [&]() {
    if (++stage == FU_NSTAGE) { stage = 0; phase ^= 1u; }
  };

  // The next residual unit rid = b * Sr + j (its sequence is ready).  Its
  // stages may go between two stages of a sweep unit: the consumers keep their
  // sweep accumulators across them.  The sequence's residual scales (the first
  // 16 bytes of its SeqInfo) are copied into each stage's info slot by the
  // bulk-copy engine together with the row data.
  auto issue_resid = [&]() -> bool {
    const long long rid = next_res;
    next_res += G;
    const int b = static_cast<int>(rid / a.Sr);
    const int j = static_cast<int>(rid - static_cast<long long>(b) * a.Sr);
    __threadfence_block();   // the finisher stored res_word before res_have
    const unsigned word = *reinterpret_cast<volatile unsigned*>(&sh.res_word);
    want_next();
    const int tstar = static_cast<int>(word & 0xffu);
    if (word & 0x100u) {
      // invalid sequence: a data-less stage, so the arrival is still counted
      if (!next_stage()) return false;
      StageDesc& d = sh.desc[stage];
      d.kind = KIND_RESID;
      d.b = b;
      d.unit = j;
      d.e0 = 0;
      d.n = 0;
      d.flags = FL_FIRST | FL_LAST;
      mbar_arrive(&sh.full[stage]);
      last_parity[stage] = -1;   // the stage was released: its previous copy has landed
      advance();
      return true;
    }
    // The scan's SeqInfo stores are ordered before its release of the
    // readiness word, which the finisher acquired before handing it over; the
    // proxy fence orders the bulk-copy engine's reads after that.
    fence_proxy_async_global();
    const bool has_q = tstar < a.K;
    const unsigned char* prow = a.target + ((static_cast<long long>(b) * W + tstar) * a.V) * TP::esz;
    const unsigned char* qrow =
        has_q ? a.draft + ((static_cast<long long>(b) * a.K + tstar) * a.V) * QT::esz : nullptr;
    const int e0 = j * a.Lr, e1 = min(a.V, e0 + a.Lr);
    for (int e = e0; e < e1; e += a.RE) {
      const int n = min(a.RE, e1 - e);
      if (!next_stage()) return false;
      StageDesc& d = sh.desc[stage];
      d.kind = KIND_RESID;
      d.b = b;
      d.unit = j;
      d.e0 = e;
      d.n = n;   // elements for residual stages
      d.flags = (e == e0 ? FL_FIRST : 0) | (e + n >= e1 ? FL_LAST : 0) | (has_q ? FL_HASQ : 0);
      const uint32_t bp = static_cast<uint32_t>(n * TP::esz), bq = has_q ? static_cast<uint32_t>(n * QT::esz) : 0u;
      mbar_arrive_expect_tx(&sh.full[stage], bp + bq + 16u);
      unsigned char* dst = ring + stage * FU_STAGE;
      bulk_g2s(dst, prow + static_cast<long long>(e) * TP::esz, bp, &sh.full[stage]);
      if (has_q) bulk_g2s(dst + a.RE * TP::esz, qrow + static_cast<long long>(e) * QT::esz, bq, &sh.full[stage]);
      bulk_g2s(&sh.stage_info[stage], a.info + b, 16u, &sh.full[stage]);
      last_parity[stage] = static_cast<int>(phase);
      advance();
    }
    return true;
  };

  // Sweep units take partial slots in turn; a slot is free again once the
  // finisher warp has read (and then merges) the partials left in it.
  int unit_seq = 0;

  // Sweep units: this CTA's FU_STATIC_UNITS static units (blockIdx + k * grid)
  // first, then units claimed from one counter in unit order (sequence-major),
  // one claim ahead so its latency is hidden.  The first claim is issued once
  // the grid barrier has passed (the counter is cleared by then).  The loop
  // acquires one ring stage at a time and then decides what fills it: the
  // next residual unit if its sequence is ready, else the next stage of the
  // current sweep unit.
  int static_taken = 0;
  bool claiming = false, sweep_open = true;
  unsigned next_claim = 0;
  bool ok = true;
  // current sweep unit and its partial slot
  bool have = false;
  unsigned u = 0;
  int slot = 0;
  int b = 0, e0 = 0, esz = 0;
  bool is_draft = false;
  const unsigned char* src = nullptr;
  uint32_t bytes = 0, off = 0;
  while (ok) {
    if (!next_stage()) break;
    if (!claiming && *reinterpret_cast<volatile int*>(&sh.grid_ready) != 0) {
      next_claim = atomicAdd(&a.ctl->claim, 1u);
      claiming = true;
    }
    if (res_is_ready()) {
      ok = issue_resid();
      continue;
    }
    if (!have) {
      long long uid = -1;
      while (static_taken < FU_STATIC_UNITS && uid < 0) {
        const long long cand = static_cast<long long>(blockIdx.x) + static_cast<long long>(static_taken) * G;
        ++static_taken;
        if (cand < static_cast<long long>(a.U)) uid = cand;
      }
      if (uid < 0 && sweep_open) {
        if (!claiming) {
          if (!fu_wait_grid(sh, a.timeout_ns)) {
            if (!fu_aborted(sh)) fu_fail(sh, a.ctl, 256u);
            break;
          }
          next_claim = atomicAdd(&a.ctl->claim, 1u);
          claiming = true;
        }
        const long long cand = static_cast<long long>(FU_STATIC_UNITS) * G + next_claim;
        if (cand < static_cast<long long>(a.U)) {
          uid = cand;
          next_claim = atomicAdd(&a.ctl->claim, 1u);
        } else {
          sweep_open = false;
        }
      }
      if (uid < 0) {
        // no sweep work left: the remaining residual units, as their sequences become ready
        if (next_res >= RU) break;
        const uint64_t t0 = global_ns();
        bool rdy = false;
        while (!(rdy = res_is_ready())) {
          if (fu_aborted(sh) || global_ns() - t0 > a.timeout_ns) break;
          __nanosleep(100);
        }
        if (!rdy) {
          fu_fail(sh, a.ctl, 2u);
          break;
        }
        ok = issue_resid();
        continue;
      }
      u = static_cast<unsigned>(uid);
      b = static_cast<int>(u / per_seq);
      const unsigned rem = u - static_cast<unsigned>(b) * per_seq;
      const int row = static_cast<int>(rem / a.S);
      const int j = static_cast<int>(rem - static_cast<unsigned>(row) * a.S);
      is_draft = row >= W;
      esz = is_draft ? QT::esz : TP::esz;
      src = is_draft ? a.draft + ((static_cast<long long>(b) * a.K + (row - W)) * a.V) * esz
                     : a.target + ((static_cast<long long>(b) * W + row) * a.V) * esz;
      e0 = j * a.L;
      bytes = static_cast<uint32_t>((min(a.V, e0 + a.L) - e0) * esz);
      off = 0;
      have = true;
      slot = unit_seq % FU_WSLOTS;
      ++unit_seq;
      // the slot's previous unit (FU_WSLOTS units back) must have been read
      if (*reinterpret_cast<volatile int*>(&sh.slot_unit[slot]) != 0) {
        const uint64_t t0 = global_ns();
        while (*reinterpret_cast<volatile int*>(&sh.slot_unit[slot]) != 0) {
          if (fu_aborted(sh) || global_ns() - t0 > a.timeout_ns) {
            fu_fail(sh, a.ctl, 16u);
            ok = false;
            break;
          }
          __nanosleep(64);
        }
        if (!ok) break;
      }
    }
    const uint32_t n = min(static_cast<uint32_t>(FU_STAGE), bytes - off);
    StageDesc& d = sh.desc[stage];
    d.kind = KIND_SWEEP;
    d.b = b;
    d.unit = static_cast<int>(u);
    d.e0 = e0 + static_cast<int>(off) / esz;
    d.n = static_cast<int>(n);   // bytes for sweep stages
    d.flags = (off == 0 ? FL_FIRST : 0) | (off + n >= bytes ? FL_LAST : 0) | (is_draft ? FL_DRAFT : 0);
    d.slot = slot;
    mbar_arrive_expect_tx(&sh.full[stage], n);
    bulk_g2s(ring + stage * FU_STAGE, src + static_cast<long long>(e0) * esz + off, n, &sh.full[stage]);
    last_parity[stage] = static_cast<int>(phase);
    advance();
    off += n;
    if (off >= bytes) have = false;
  }
  // the finisher may leave once it has merged this many units (a unit claimed
  // but never issued is not counted)
  *reinterpret_cast<volatile int*>(&sh.units_issued) = have && off == 0 ? unit_seq - 1 : unit_seq;
  *reinterpret_cast<volatile int*>(&sh.res_want) = -1;
  // stop marker for the consumers
  if (next_stage()) {
    sh.desc[stage].kind = KIND_STOP;
    mbar_arrive(&sh.full[stage]);
    last_parity[stage] = -1;
  }
  // Do not leave while a copy may still land in this CTA's shared memory.  A
  // stage's recorded parity is that of its last copy; any later arrival on the
  // stage (which would flip the phase again) clears the record, so a wait here
  // is only for a copy that has not been consumed (abort path).
#pragma unroll
  for (int s = 0; s < FU_NSTAGE; ++s)
    if (last_parity[s] >= 0 && !mbar_wait(&sh.full[s], static_cast<uint32_t>(last_parity[s]), a.timeout_ns))
      atomicOr(&a.ctl->err, 8u);
}

// ---------------------------------------------------------------------------
// consumers (eight warps)
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS>
__device__ void fu_consumer(const FusedArgs& a, unsigned char* ring, FuShared& sh, int cw, int lane) {
  const int ctid = cw * 32 + lane;
  int stage = 0;
  uint32_t phase = 0;
  StatsAcc sacc;
  sacc.init();
  for (;;) {
    if (__any_sync(0xffffffffu, fu_aborted(sh))) break;
    if (!__all_sync(0xffffffffu, mbar_wait(&sh.full[stage], phase, a.timeout_ns))) {
      fu_fail(sh, a.ctl, 4u);
      break;
    }
    const StageDesc d = sh.desc[stage];
    if (d.kind == KIND_STOP) break;
    if (d.kind == KIND_SWEEP && (d.flags & FL_FIRST)) sacc.init();
    const int cur = stage;
    const unsigned char* buf = ring + stage * FU_STAGE;
    if (d.kind == KIND_SWEEP) {
      if (d.flags & FL_DRAFT) {
        if constexpr (!PROBS) stats_stage<TQ>(reinterpret_cast<const uint4*>(buf), d.n >> 4, ctid, a.c, sacc);
      } else {
        stats_stage<TP>(reinterpret_cast<const uint4*>(buf), d.n >> 4, ctid, a.c, sacc);
      }
    } else if (d.n > 0) {
      resid_stage<TP, TQ, PROBS>(buf, d, sh.stage_info[cur], a.RE, cw, lane, a.c,
                                 a.bsum + static_cast<long long>(d.b) * a.NB);
    }
    if (++stage == FU_NSTAGE) { stage = 0; phase ^= 1u; }
    if (!(d.flags & FL_LAST)) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[cur]);
      continue;
    }
    // End of a work item: every warp leaves its partial in shared memory (a
    // sweep unit's slot) and counts itself there.  The last one releases the
    // stage and hands the unit on: a sweep unit to the finisher warp, which
    // merges the partials and adds the unit to the sequence's counter off the
    // consumers' path; a residual unit straight to its counter
    // (fire-and-forget, release ordered).
    if (d.kind == KIND_SWEEP) sacc.warp_reduce(a.c);
    else __syncwarp();
    int prev = 0;
    if (lane == 0) {
      if (d.kind == KIND_SWEEP) sh.wpart[d.slot][cw] = sacc.pack();
      __threadfence_block();
      prev = atomicAdd(&sh.unit_cnt[cur], 1);
    }
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev == FU_CW - 1 && lane == 0) {
      sh.unit_cnt[cur] = 0;   // the slot's next item starts only after this warp releases it
      // the other warps' partials are ordered before their increments, which
      // this warp observed; its block fence orders the hand-over after them
      __threadfence_block();
      if (d.kind == KIND_SWEEP) {
        *reinterpret_cast<volatile int*>(&sh.slot_unit[d.slot]) = d.unit + 1;
        mbar_arrive(&sh.empty[cur]);
      } else {
        // the stage first: the release reduction waits until the block sums
        // are visible device-wide, and the ring should not wait with it
        mbar_arrive(&sh.empty[cur]);
        red_release_add_u32(fu_cnt2(a, d.b), 1u);
      }
    } else if (lane == 0) {
      mbar_arrive(&sh.empty[cur]);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// merger (one warp): merges the warp partials of this CTA's completed sweep
// units and hands the readiness word of the producer's next residual sequence
// over, off the consumers' and the producer's paths
// ---------------------------------------------------------------------------
__device__ void fu_merger(const FusedArgs& a, FuShared& sh, int lane) {
  // clear this CTA's share of the control block, then the grid barrier
  {
    uint4* z = reinterpret_cast<uint4*>(a.ctl);
    for (unsigned i = blockIdx.x * 32u + static_cast<unsigned>(lane); i < a.zero_words; i += gridDim.x * 32u)
      z[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    __threadfence();
    // If the barrier gives up, a CTA that had not yet cleared its share could
    // still clear the error word; the limit is 1 s, far beyond the microseconds
    // co-resident CTAs take to arrive.
    int passed = 1;
    if (lane == 0) passed = fu_grid_barrier(a.timeout_ns) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, passed, 0) == 0) {
      if (lane == 0) fu_fail(sh, a.ctl, 512u);
    } else if (lane == 0) {
      *reinterpret_cast<volatile int*>(&sh.grid_ready) = 1;
    }
  }
  const unsigned per_seq_units = static_cast<unsigned>(a.RB) * static_cast<unsigned>(a.S);
  int merged = 0;
  uint64_t last_progress = global_ns();
  for (;;) {
    // Control decisions are taken on lane 0's reads and broadcast: a lane that
    // read the shared words at another moment must not leave the loop (or skip
    // a step) on its own, since the warp's shuffles below need every lane.
    __syncwarp();
    int want = -1, stop = 0, need_res = 0;
    if (lane == 0) {
      want = *reinterpret_cast<volatile int*>(&sh.res_want);
      const int issued = *reinterpret_cast<volatile int*>(&sh.units_issued);
      stop = (want < 0 && issued >= 0 && merged >= issued) || fu_aborted(sh);
      need_res = want >= 0 && *reinterpret_cast<volatile int*>(&sh.res_have) != want;
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) break;
    want = __shfl_sync(0xffffffffu, want, 0);
    need_res = __shfl_sync(0xffffffffu, need_res, 0);
    bool progress = false;
    // the readiness poll is issued first and read after the merges
    unsigned v = 0;
    if (lane == 0 && need_res) v = ld_relaxed_u32(fu_ready(a, want));
    {
      const int su = lane < FU_WSLOTS ? *reinterpret_cast<volatile int*>(&sh.slot_unit[lane]) : 0;
      unsigned m = __ballot_sync(0xffffffffu, su != 0);
      while (m) {
        const int sl = __ffs(m) - 1;
        m &= m - 1u;
        const int unit = __shfl_sync(0xffffffffu, su, sl) - 1;
        __threadfence_block();
        const float2 wp = lane < FU_CW ? sh.wpart[sl][lane] : make_float2(kNegInf, 0.f);
        __syncwarp();
        __threadfence_block();
        if (lane == 0) *reinterpret_cast<volatile int*>(&sh.slot_unit[sl]) = 0;   // partials are in registers
        const float4 u = merge_unit(wp, lane, a.c);
        if (lane == 0) {
          a.part[unit] = u;
          __threadfence_block();
          red_release_add_u32(fu_cnt1(a, static_cast<int>(static_cast<unsigned>(unit) / per_seq_units)), 1u);
        }
        ++merged;
        progress = true;
      }
    }
    const unsigned v_res = __shfl_sync(0xffffffffu, v, 0);
    if (need_res && v_res != 0u) {
      __threadfence();   // acquire: the scan's SeqInfo stores are visible from here on
      if (lane == 0) {
        *reinterpret_cast<volatile unsigned*>(&sh.res_word) = v_res;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&sh.res_have) = want;
      }
      progress = true;
    }
    __syncwarp();
    if (progress) {
      last_progress = global_ns();
      continue;
    }
    if (__any_sync(0xffffffffu, global_ns() - last_progress > 4 * a.timeout_ns)) {
      if (lane == 0) fu_fail(sh, a.ctl, 64u);
      break;
    }
    __nanosleep(64);
  }
}

// ---------------------------------------------------------------------------
// finisher (one warp): the scans of sequences b = blockIdx (mod grid) and the
// picks of sequences b = blockIdx + grid - grid/2 (mod grid), each started as
// soon as the sequence's counter is complete
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS>
__device__ void fu_finisher(const FusedArgs& a, FuShared& sh, int lane) {
  const unsigned G = gridDim.x;
  const unsigned per_seq = static_cast<unsigned>(a.RB) * static_cast<unsigned>(a.S);
  unsigned bs = blockIdx.x;                              // next scan
  unsigned bp = (blockIdx.x + G - G / 2) % G;            // next pick
  ScanInputs in{};
  if (bs < static_cast<unsigned>(a.B)) in = scan_inputs<TP, TQ, PROBS>(a, static_cast<int>(bs), lane);
  // the counters polled below are valid once every CTA has cleared its share
  if (!fu_wait_grid(sh, a.timeout_ns)) {
    if (lane == 0 && !fu_aborted(sh)) fu_fail(sh, a.ctl, 256u);
    return;
  }
  uint64_t last_progress = global_ns();
  while (bs < static_cast<unsigned>(a.B) || bp < static_cast<unsigned>(a.B)) {
    bool progress = false;
    // both polls in one round (lane 1: the next scan's sweep counter, lane 2:
    // the next pick's residual counter)
    unsigned v = 0;
    if (lane == 1 && bs < static_cast<unsigned>(a.B)) v = ld_relaxed_u32(fu_cnt1(a, static_cast<int>(bs)));
    if (lane == 2 && bp < static_cast<unsigned>(a.B)) v = ld_relaxed_u32(fu_cnt2(a, static_cast<int>(bp)));
    const unsigned v_scan = __shfl_sync(0xffffffffu, v, 1);
    const unsigned v_pick = __shfl_sync(0xffffffffu, v, 2);
    // (the test hook asks one sequence's scan for one unit more than exists)
    const unsigned need_scan = per_seq + (static_cast<int>(bs) == a.debug_stall_b ? 1u : 0u);
    if (bs < static_cast<unsigned>(a.B) && v_scan == need_scan) {
      __threadfence();
      finish_scan<TP, TQ, PROBS>(a, static_cast<int>(bs), lane, in, sh.scan_scratch);
      bs += G;
      if (bs < static_cast<unsigned>(a.B)) in = scan_inputs<TP, TQ, PROBS>(a, static_cast<int>(bs), lane);
      progress = true;
    }
    if (bp < static_cast<unsigned>(a.B) && v_pick == static_cast<unsigned>(a.Sr)) {
      __threadfence();
      finish_pick<TP, TQ, PROBS>(a, static_cast<int>(bp), lane);
      bp += G;
      progress = true;
    }
    __syncwarp();
    if (progress) {
      last_progress = global_ns();
      continue;
    }
    const bool stop = __any_sync(0xffffffffu, fu_aborted(sh) || global_ns() - last_progress > 4 * a.timeout_ns);
    if (stop) {
      if (lane == 0) fu_fail(sh, a.ctl, 32u);
      break;
    }
    __nanosleep(FU_IDLE_NS);
  }
}

// ---------------------------------------------------------------------------
// the kernel (cooperative launch: every CTA resident)
// ---------------------------------------------------------------------------
constexpr size_t fu_smem_bytes() { return FU_NSTAGE * FU_STAGE + sizeof(FuShared) + 128; }

template <class TP, class TQ, bool PROBS>
__global__ void __launch_bounds__(FU_THREADS, FU_CTAS_PER_SM) fused_sample_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) unsigned char fu_smem[];
  unsigned char* ring = fu_smem;
  FuShared& sh = *reinterpret_cast<FuShared*>(fu_smem + FU_NSTAGE * FU_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < FU_NSTAGE; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], FU_CW);
      sh.unit_cnt[s] = 0;
    }
    sh.abort = 0;
    sh.res_have = -1;
    sh.grid_ready = 0;
    sh.units_issued = -1;
    for (int i = 0; i < FU_WSLOTS; ++i) sh.slot_unit[i] = 0;
    // the sequence of this CTA's first residual unit, set before any warp
    // starts, so the finisher cannot leave before the producer asks for it
    const unsigned RU = static_cast<unsigned>(a.B) * static_cast<unsigned>(a.Sr);
    sh.res_want = blockIdx.x < RU ? static_cast<int>(blockIdx.x / a.Sr) : -1;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) fu_producer<TP, TQ, PROBS>(a, ring, sh);
  } else if (warp == FU_MERGE_WARP) {
    fu_merger(a, sh, lane);
  } else if (warp == FU_FIN_WARP) {
    fu_finisher<TP, TQ, PROBS>(a, sh, lane);
  } else {
    fu_consumer<TP, TQ, PROBS>(a, ring, sh, warp - 1, lane);
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
