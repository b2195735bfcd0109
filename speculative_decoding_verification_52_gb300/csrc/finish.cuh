// finish.cuh -- per-sequence decisions after the vocabulary sweep.
//
//  finish_greedy_kernel   greedy chain rule ("Speculative decoding and EAGLE",
//                         section "The exactness rule", greedy case): one warp
//                         per sequence, lane t owns position t.
//  finish_tree_kernel     greedy tree rule ("Tree attention verification"): one
//                         CTA per sequence.
//  finish_sample_kernel   sampling rule ("The exactness rule"; "Speculative
//                         decoding: draft, verify, repeat", steps 1-3;
//                         "Speculative Decoding: from idea to SOTA", section 3):
//                         one thread-block cluster per sequence.  Every CTA of
//                         the cluster rebuilds the row normalisers from the
//                         sweep's partials and runs the accept scan; then the
//                         cluster re-reads the stopping row(s), each CTA one
//                         vocabulary slice, and draws the replacement (or bonus)
//                         token by an inverse CDF whose slice totals are
//                         exchanged through distributed shared memory.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// row normaliser from S partials: M = row max, AM = fl(M * c), Srow = sum of
// 2^(z*c - AM) over the row (double).  state 0 ok, 1 invalid row, 2 poisoned.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void merge_row_stats(const float2* part, int S, float c, float& M, float& AM,
                                                double& Srow, int& state) {
  M = kNegInf;
  bool poison = false;
  for (int j = 0; j < S; ++j) {
    const float2 p = part[j];
    if (p.x != p.x) poison = true;
    else M = fmaxf(M, p.x);
  }
  AM = 0.f;
  Srow = 0.0;
  if (poison) { state = 2; return; }
  if (M == kNegInf) { state = 1; return; }
  AM = __fmul_rn(M, c);
  double acc = 0.0;
  for (int j = 0; j < S; ++j) {
    const float2 p = part[j];
    if (p.x == kNegInf) continue;
    acc += static_cast<double>(p.y) *
           exp2(static_cast<double>(__fmul_rn(p.x, c)) - static_cast<double>(AM));
  }
  Srow = acc;
  state = (isfinite(acc) && acc > 0.0) ? 0 : 1;
}

// row argmax from S partials: g = index, state 0 ok, 1 NaN row, 2 poisoned.
__device__ __forceinline__ void merge_row_argmax(const float2* part, int S, int& g, int& state) {
  ArgmaxAcc acc;
  acc.init();
  bool poison = false;
  for (int j = 0; j < S; ++j) {
    const float2 p = part[j];
    if (__float_as_int(p.y) == kIdxPoison) poison = true;
    acc.merge(p.x, __float_as_int(p.y));
  }
  g = acc.idx;
  if (poison) state = 2;
  else if (acc.best != acc.best || acc.idx == kIdxNone) state = 1;
  else state = 0;
}

// ---------------------------------------------------------------------------
// greedy chain
// ---------------------------------------------------------------------------
struct FinishGreedyArgs {
  const float2* part;      // rows b*(K+1)+t, S partials each
  const int32_t* tokens;   // [B, K]
  int B, K, V, S;
  int32_t* out_tokens;     // [B, K+1]
  int32_t* num_accepted;   // [B]
};

constexpr int FG_THREADS = 256;

__global__ void __launch_bounds__(FG_THREADS) finish_greedy_kernel(const FinishGreedyArgs a) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (FG_THREADS / 32) + (threadIdx.x >> 5);
  if (b >= a.B) return;
  const int K = a.K, W = K + 1;
  int g = -1, state = 0, x = -1;
  if (lane <= K) merge_row_argmax(a.part + (static_cast<long long>(b) * W + lane) * a.S, a.S, g, state);
  if (lane < K) x = a.tokens[static_cast<long long>(b) * K + lane];
  const bool tok_bad = lane < K && (x < 0 || x >= a.V);
  const unsigned bad_tok = __ballot_sync(0xffffffffu, tok_bad);
  const unsigned mismatch = __ballot_sync(0xffffffffu, lane < K && g != x);
  const int tstar = mismatch ? (__ffs(mismatch) - 1) : K;   // first mismatch, else K
  const unsigned bad_row = __ballot_sync(0xffffffffu, lane <= tstar && state == 1);
  const unsigned to_row = __ballot_sync(0xffffffffu, lane <= tstar && state == 2);
  // rows after the stop are not read by the rule; a bad row at or before it decides
  int out;
  int nacc = tstar;
  if (bad_tok || bad_row || to_row) {
    out = -1;
    nacc = (to_row && !bad_tok) ? -2 : -1;
  } else {
    out = lane < tstar ? x : (lane == tstar ? g : -1);
  }
  if (lane <= K) a.out_tokens[static_cast<long long>(b) * W + lane] = out;
  if (lane == 0) a.num_accepted[b] = nacc;
}

// ---------------------------------------------------------------------------
// greedy tree
// ---------------------------------------------------------------------------
struct FinishTreeArgs {
  const float2* part;         // rows b*N+i, S partials each
  const int32_t* parents;     // [N]
  const int32_t* node_tokens; // [B, N]
  int B, N, V, S, max_depth;
  int32_t* out_tokens;        // [B, max_depth+1]
  int32_t* num_accepted;      // [B]
  int32_t* out_path;          // [B, max_depth+1] or null
};

constexpr int FT_THREADS = 256;
constexpr int FT_MAX_N = 1024;

__global__ void __launch_bounds__(FT_THREADS) finish_tree_kernel(const FinishTreeArgs a) {
  __shared__ int s_g[FT_MAX_N];
  __shared__ int s_state[FT_MAX_N];
  __shared__ int s_par[FT_MAX_N];
  __shared__ int s_depth[FT_MAX_N];
  __shared__ unsigned char s_acc[FT_MAX_N];
  const int b = blockIdx.x;
  const int N = a.N, W = a.max_depth + 1;
  for (int i = threadIdx.x; i < N; i += FT_THREADS) {
    int g, st;
    merge_row_argmax(a.part + (static_cast<long long>(b) * N + i) * a.S, a.S, g, st);
    s_g[i] = g;
    s_state[i] = st;
    s_par[i] = a.parents[i];
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const int32_t* tok = a.node_tokens + static_cast<long long>(b) * N;
  int32_t* out = a.out_tokens + static_cast<long long>(b) * W;
  int32_t* path = a.out_path ? a.out_path + static_cast<long long>(b) * W : nullptr;
  // topology check (parents[0] = -1, 0 <= parents[i] < i, depth <= max_depth)
  bool topo = (s_par[0] == -1);
  s_depth[0] = 0;
  for (int i = 1; topo && i < N; ++i) {
    const int p = s_par[i];
    if (p < 0 || p >= i) { topo = false; break; }
    s_depth[i] = s_depth[p] + 1;
    if (s_depth[i] > a.max_depth) topo = false;
  }
  int status = topo ? 0 : -1;
  int best = 0;
  if (topo) {
    // acceptance propagates parent -> child in index order (parents[i] < i)
    s_acc[0] = 1;
    if (s_state[0] != 0) status = s_state[0] == 2 ? -2 : -1;
    for (int i = 1; status == 0 && i < N; ++i) {
      const int p = s_par[i];
      const bool acc = s_acc[p] && tok[i] == s_g[p];
      s_acc[i] = acc;
      if (acc) {
        if (s_state[i] != 0) { status = s_state[i] == 2 ? -2 : -1; break; }
        if (s_depth[i] > s_depth[best]) best = i;
      }
    }
  }
  for (int j = 0; j < W; ++j) {
    out[j] = -1;
    if (path) path[j] = -1;
  }
  if (status != 0) {
    a.num_accepted[b] = status;
    return;
  }
  const int d = s_depth[best];
  int node = best;
  for (int j = d - 1; j >= 0; --j) {
    out[j] = tok[node];
    if (path) path[j] = node;
    node = s_par[node];
  }
  out[d] = s_g[best];
  a.num_accepted[b] = d;
}

// ---------------------------------------------------------------------------
// sampling
// ---------------------------------------------------------------------------
struct FinishSampleArgs {
  const unsigned char* target;   // [B, K+1, V]
  const unsigned char* draft;    // [B, K, V] logits or f32 probs (null if K == 0)
  const int32_t* tokens;         // [B, K]
  const float* uni;              // [B, K+1, 2]
  const float2* part;            // target rows b*(K+1)+t, then draft rows B*(K+1)+b*K+t
  int B, K, V, S;
  int L;                         // vocabulary slice per CTA of the cluster
  float c;                       // log2(e)/T, identical to the sweep's
  int32_t* out_tokens;
  int32_t* num_accepted;
  int debug_b, debug_t;          // debug_b < 0: no forced stop
  float* debug_row;
  float* debug_mass;
};

constexpr int FS_THREADS = 256;
constexpr int FS_WARPS = FS_THREADS / 32;
constexpr int FS_MAX_ROWS = 2 * 31 + 1;
constexpr int FS_MAX_L = 24576;   // per-CTA slice bound (shared memory)

__host__ __device__ constexpr int fs_skew(int i) { return i + (i >> 5); }
__host__ __device__ constexpr size_t fs_smem_bytes(int L) {
  return 2u * static_cast<size_t>(fs_skew(L) + 1) * sizeof(float);
}

// block-wide sum of one double (all threads get the result)
__device__ __forceinline__ double block_sum_d(double v, double* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < FS_WARPS; ++w) t += scratch[w];
  return t;
}

template <class TP, class TQ, bool PROBS, bool VEC>
__global__ void __launch_bounds__(FS_THREADS) finish_sample_kernel(const FinishSampleArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / CL;
  const int K = a.K, W = K + 1, V = a.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(16) float fs_dyn[];
  __shared__ float s_A[FS_MAX_ROWS];
  __shared__ double s_S[FS_MAX_ROWS];
  __shared__ int s_state[FS_MAX_ROWS];
  __shared__ double s_scr[FS_WARPS];
  __shared__ double s_wsum[FS_WARPS];
  __shared__ int s_status, s_tstar;
  // cluster-visible slots (read or updated by other CTAs through DSMEM)
  __shared__ double cl_sum[2];
  __shared__ double cl_tot;
  __shared__ int cl_pick, cl_last;

  // ---- phase 0: row normalisers + accept scan (redundant in every CTA) ----
  const int nrows = PROBS ? W : W + K;
  for (int r = tid; r < nrows; r += FS_THREADS) {
    const long long row = (r < W) ? static_cast<long long>(b) * W + r
                                  : static_cast<long long>(a.B) * W + static_cast<long long>(b) * K + (r - W);
    float M, AM;
    double Sr;
    int st;
    merge_row_stats(a.part + row * a.S, a.S, a.c, M, AM, Sr, st);
    s_A[r] = AM;
    s_S[r] = Sr;
    s_state[r] = st;
  }
  if (tid == 0) { cl_pick = 0x7fffffff; cl_last = -1; }
  __syncthreads();
  if (tid == 0) {
    int status = 0, tstar = K;
    const int32_t* tok = a.tokens + static_cast<long long>(b) * K;
    for (int t = 0; t < K; ++t)
      if (tok[t] < 0 || tok[t] >= V) status = -1;
    const bool forced = (b == a.debug_b);
    for (int t = 0; status == 0 && !forced && t < K; ++t) {
      if (s_state[t] != 0) { status = s_state[t] == 2 ? -2 : -1; break; }
      const int x = tok[t];
      const long long off = (static_cast<long long>(b) * W + t) * V + x;
      const double zp = static_cast<double>(TP::load(a.target, off));
      const double pa = exp2(zp * static_cast<double>(a.c) - static_cast<double>(s_A[t])) / s_S[t];
      double qc;
      const long long offq = (static_cast<long long>(b) * K + t) * V + x;
      if (PROBS) {
        const float qv = F32T::load(a.draft, offq);
        if (qv != qv || qv < 0.f) { status = -1; break; }
        qc = static_cast<double>(qv);
      } else {
        const int r = W + t;
        if (s_state[r] != 0) { status = s_state[r] == 2 ? -2 : -1; break; }
        const double zq = static_cast<double>(TQ::load(a.draft, offq));
        qc = exp2(zq * static_cast<double>(a.c) - static_cast<double>(s_A[r])) / s_S[r];
      }
      const double u = static_cast<double>(a.uni[(static_cast<long long>(b) * W + t) * 2]);
      const bool accept = (qc == 0.0) || (u < pa / qc);
      if (!accept) { tstar = t; break; }
    }
    if (forced) tstar = a.debug_t;
    // the rows the replacement draw reads must be valid
    if (status == 0 && s_state[tstar] != 0) status = s_state[tstar] == 2 ? -2 : -1;
    if (status == 0 && tstar < K && !PROBS && s_state[W + tstar] != 0) status = s_state[W + tstar] == 2 ? -2 : -1;
    s_status = status;
    s_tstar = tstar;
  }
  __syncthreads();
  const int status = s_status, tstar = s_tstar;
  if (status != 0) {
    if (rank == 0) {
      for (int j = tid; j < W; j += FS_THREADS) a.out_tokens[static_cast<long long>(b) * W + j] = -1;
      if (tid == 0) a.num_accepted[b] = status;
    }
    return;   // uniform across the cluster: no CTA reaches a cluster barrier
  }

  // ---- phase 1: exponentials of the stopping row(s) for this CTA's slice ---
  const bool has_q = tstar < K;
  const int v0 = rank * a.L;
  const int n = max(0, min(V, v0 + a.L) - v0);
  float* EP = fs_dyn;
  float* EQ = fs_dyn + fs_skew(a.L) + 1;
  const float c = a.c;
  const float nAP = -s_A[tstar];
  const float nAQ = PROBS ? 0.f : -s_A[W + (has_q ? tstar : 0)];
  const unsigned char* prow = a.target + (static_cast<long long>(b) * W + tstar) * V * TP::esz;
  const unsigned char* qrow =
      has_q ? a.draft + (static_cast<long long>(b) * K + tstar) * V * (PROBS ? 4 : TQ::esz) : nullptr;
  float sp = 0.f, sq = 0.f;
  if (VEC) {
    const uint4* pv = reinterpret_cast<const uint4*>(prow + static_cast<long long>(v0) * TP::esz);
    for (int i = tid; i < n / TP::vpe; i += FS_THREADS) {
      const uint4 q = __ldg(pv + i);
      float x[TP::vpe];
      TP::unpack(q, x);
#pragma unroll
      for (int k = 0; k < TP::vpe; ++k) {
        const float e = ex2_approx(__fmaf_rn(x[k], c, nAP));
        EP[fs_skew(i * TP::vpe + k)] = e;
        sp += e;
      }
    }
    if (has_q) {
      if (PROBS) {
        const uint4* qv = reinterpret_cast<const uint4*>(qrow + static_cast<long long>(v0) * 4);
        for (int i = tid; i < n / 4; i += FS_THREADS) {
          const uint4 q = __ldg(qv + i);
          float x[4];
          F32T::unpack(q, x);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            EQ[fs_skew(i * 4 + k)] = x[k];
            sq += x[k];
          }
        }
      } else {
        const uint4* qv = reinterpret_cast<const uint4*>(qrow + static_cast<long long>(v0) * TQ::esz);
        for (int i = tid; i < n / TQ::vpe; i += FS_THREADS) {
          const uint4 q = __ldg(qv + i);
          float x[TQ::vpe];
          TQ::unpack(q, x);
#pragma unroll
          for (int k = 0; k < TQ::vpe; ++k) {
            const float e = ex2_approx(__fmaf_rn(x[k], c, nAQ));
            EQ[fs_skew(i * TQ::vpe + k)] = e;
            sq += e;
          }
        }
      }
    }
  } else {
    for (int i = tid; i < n; i += FS_THREADS) {
      const float e = ex2_approx(__fmaf_rn(TP::load(prow, v0 + i), c, nAP));
      EP[fs_skew(i)] = e;
      sp += e;
      if (has_q) {
        const float eq = PROBS ? F32T::load(qrow, v0 + i) : ex2_approx(__fmaf_rn(TQ::load(qrow, v0 + i), c, nAQ));
        EQ[fs_skew(i)] = eq;
        sq += eq;
      }
    }
  }
  const double bsp = block_sum_d(static_cast<double>(sp), s_scr);
  const double bsq = block_sum_d(static_cast<double>(sq), s_scr);
  if (tid == 0) { cl_sum[0] = bsp; cl_sum[1] = bsq; }
  cluster.sync();
  double Sp = 0.0, Sq = 0.0;
  for (int r = 0; r < CL; ++r) {
    const double* rs = cluster.map_shared_rank(cl_sum, r);
    Sp += rs[0];
    Sq += rs[1];
  }
  const float inv_p = static_cast<float>(1.0 / Sp);
  const float inv_q = PROBS ? 1.f : static_cast<float>(1.0 / Sq);

  // ---- phase 2: residual weights, slice prefix sums, inverse CDF ----------
  const int seg = (n + FS_THREADS - 1) / FS_THREADS;
  const int k0 = min(n, tid * seg), k1 = min(n, k0 + seg);
  const double u1 = static_cast<double>(a.uni[(static_cast<long long>(b) * W + tstar) * 2 + 1]);
  bool use_q = has_q;
  double R = 0.0, prefix = 0.0, excl = 0.0;
  float Tt = 0.f;
  for (int pass = 0; pass < 2; ++pass) {
    Tt = 0.f;
    int lastpos = -1;
    for (int k = k0; k < k1; ++k) {
      const float wp = __fmul_rn(EP[fs_skew(k)], inv_p);
      const float w = use_q ? fmaxf(0.f, __fmaf_rn(-EQ[fs_skew(k)], inv_q, wp)) : wp;
      Tt += w;
      if (w > 0.f) lastpos = v0 + k;
    }
    // block exclusive scan of the per-thread totals (double)
    double x = static_cast<double>(Tt);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    double wex = 0.0, tot = 0.0;
    for (int w = 0; w < FS_WARPS; ++w) {
      if (w < warp) wex += s_wsum[w];
      tot += s_wsum[w];
    }
    excl = wex + (x - static_cast<double>(Tt));
    int lp = lastpos;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
    if (lane == 0 && lp >= 0) atomicMax(cluster.map_shared_rank(&cl_last, 0), lp);
    if (tid == 0) cl_tot = tot;
    cluster.sync();
    R = 0.0;
    prefix = 0.0;
    for (int r = 0; r < CL; ++r) {
      const double t = *cluster.map_shared_rank(&cl_tot, r);
      if (r < rank) prefix += t;
      R += t;
    }
    if (R > 0.0 || !use_q) break;
    use_q = false;   // residual mass zero: draw from p_t instead
    cluster.sync();  // everyone has read cl_tot before it is rewritten
    if (rank == 0 && tid == 0) cl_last = -1;
    cluster.sync();
  }

  const double target = u1 * R;
  const double base = prefix + excl;
  if (Tt > 0.f && base <= target && base + static_cast<double>(Tt) > target) {
    float run = 0.f;
    for (int k = k0; k < k1; ++k) {
      const float wp = __fmul_rn(EP[fs_skew(k)], inv_p);
      const float w = use_q ? fmaxf(0.f, __fmaf_rn(-EQ[fs_skew(k)], inv_q, wp)) : wp;
      run += w;
      if (base + static_cast<double>(run) > target) {
        atomicMin(cluster.map_shared_rank(&cl_pick, 0), v0 + k);
        break;
      }
    }
  }
  if (b == a.debug_b && R > 0.0) {
    for (int k = k0; k < k1; ++k) {
      const float wp = __fmul_rn(EP[fs_skew(k)], inv_p);
      const float w = use_q ? fmaxf(0.f, __fmaf_rn(-EQ[fs_skew(k)], inv_q, wp)) : wp;
      a.debug_row[v0 + k] = static_cast<float>(static_cast<double>(w) / R);
    }
    if (rank == 0 && tid == 0) *a.debug_mass = static_cast<float>(R);
  }
  cluster.sync();
  if (rank == 0) {
    const int pick = (cl_pick != 0x7fffffff) ? cl_pick : cl_last;
    const int32_t* tok = a.tokens + static_cast<long long>(b) * K;
    for (int j = tid; j < W; j += FS_THREADS)
      a.out_tokens[static_cast<long long>(b) * W + j] = j < tstar ? tok[j] : (j == tstar ? pick : -1);
    if (tid == 0) a.num_accepted[b] = tstar;
  }
}

}  // namespace sv
