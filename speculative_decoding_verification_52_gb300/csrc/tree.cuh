// tree.cuh -- greedy tree verification in one persistent kernel that sweeps
// only the rows the rule needs ("Speculative decoding and EAGLE", section
// "Tree attention verification"; "Speculative Decoding: from idea to SOTA",
// section 6).
//
// Node i of a sequence is accepted iff its parent is accepted and its token
// equals the argmax of the parent's row; the root is accepted.  Only accepted
// nodes' rows are ever needed (their argmax decides their children, and the
// deepest one's argmax is the bonus token), so rows are swept on demand:
//
//   work unit   (sequence b, node i, slice j) of an accepted node: the
//               first-index argmax partial of one slice of node i's row.  The
//               root units of every sequence are implicit; all others come from
//               a global FIFO of unit ids.
//   producer    (1 thread) claims FIFO positions with an atomic counter, one
//               position ahead, waits until the position is filled, and streams
//               the unit's bytes into a ring of 16 KB shared-memory stages with
//               1-D bulk async copies.
//   consumers   (8 warps) fold each stage into per-thread argmax accumulators;
//               at a unit's end each warp writes its partial and the last warp
//               adds the unit to the node's counter with a release reduction.
//   finisher    (1 warp) owns sequences b = blockIdx (mod grid).  It keeps one
//               bit per node for "accepted" and "resolved" (node l + 32w is bit w
//               of lane l), polls the counters of accepted, unresolved nodes,
//               and resolves a complete node: merges its partials into g, tests
//               its children's tokens against g, and appends the accepted
//               children's units to the FIFO.  When no accepted node is left
//               unresolved it writes the path to the deepest accepted node
//               (smallest index on ties) and its argmax.
//
// Chain mode runs the greedy chain rule ("The exactness rule", greedy case)
// through the same machinery: node t is the drafted position t (parent t - 1,
// token x_{t-1}), and a draft token outside [0, V) makes the sequence invalid.
// A chain's levels depend on one another, so chain mode sweeps TR_AHEAD rows
// ahead: rows 0..TR_AHEAD of every sequence are implicit units, and when row t
// resolves with x_t == argmax (position t+1 accepted) row t+1+TR_AHEAD is
// queued, before the rows between are known to be needed.  At most TR_AHEAD
// rows past the first mismatch are read; producers skip queued rows of
// sequences that have already finished.
//
// The tree topology (parents[]) is checked and its depths computed once per
// CTA in shared memory.  Every wait is bounded in time; a timeout sets an error
// word and the last CTA to leave marks every sequence -2.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int TR_CW = 8;                          // consumer warps
constexpr int TR_CT = TR_CW * 32;
constexpr int TR_THREADS = TR_CT + 64;            // + producer warp + finisher warp
constexpr int TR_FIN_WARP = TR_CW + 1;
constexpr int TR_STAGE = 16384;
constexpr int TR_NSTAGE = 4;
constexpr int TR_CTAS_PER_SM = 3;
constexpr int TR_MAX_N = 1024;                    // node bits: 32 lanes x 32 words
constexpr int TR_MAX_SEQ = 4;                     // sequences per finisher warp
constexpr int TR_AHEAD = 1;                       // chain mode: rows swept ahead of the last resolved one

struct TrCtl {                   // zeroed before every call (96 bytes reserved)
  unsigned err;                  // a wait timed out
  unsigned left;                 // CTAs that have left
  unsigned seqs_done;            // sequences whose outputs are written
  unsigned pad0[5];
  unsigned qhead;                // FIFO positions claimed by producers
  unsigned pad1[7];
  unsigned qtail;                // FIFO positions reserved by finishers
  unsigned pad2[7];
};
static_assert(sizeof(TrCtl) == 96, "tree control block layout");

struct TreeArgs {
  const unsigned char* target;   // [B, N, V]
  const int32_t* parents;        // [N] (unused in chain mode)
  const int32_t* node_tokens;    // [B, N]; chain mode: draft tokens [B, N - 1]
  int B, N, V, S, L, max_depth;  // S slices of L elements per row
  int chain;                     // 1: chain of N nodes, node t's token = draft token t - 1
  unsigned qcap;                 // FIFO capacity = B * (N - 1) * S
  TrCtl* ctl;
  unsigned* cnt;                 // [B * N] units completed per node
  unsigned* fifo;                // [qcap] unit id + 1, 0 = not yet written
  unsigned* sdone;               // [B] 1 once the sequence's outputs are written (chain look-ahead)
  float2* part;                  // [B * N * S * TR_CW] warp partials
  int32_t* out_tokens;           // [B, max_depth + 1]
  int32_t* num_accepted;         // [B]
  int32_t* out_path;             // [B, max_depth + 1] or null
  unsigned long long timeout_ns;
};

struct TrStageDesc {
  int stop, uid, e0, n, flags;
};

struct TrShared {
  uint64_t full[TR_NSTAGE];
  uint64_t empty[TR_NSTAGE];
  TrStageDesc desc[TR_NSTAGE];
  int unit_cnt[TR_NSTAGE];
  int abort;
  int topo_ok;
  short par[TR_MAX_N];           // parents (the root's is -1)
  unsigned short depth[TR_MAX_N];
};

// token proposed by node c >= 1 of sequence b
__device__ __forceinline__ int tr_token(const TreeArgs& a, int b, int c) {
  return a.chain ? __ldg(a.node_tokens + static_cast<long long>(b) * (a.N - 1) + (c - 1))
                 : __ldg(a.node_tokens + static_cast<long long>(b) * a.N + c);
}

__device__ __forceinline__ bool tr_aborted(const TrShared& sh) {
  return *reinterpret_cast<const volatile int*>(&sh.abort) != 0;
}
__device__ __forceinline__ void tr_fail(TrShared& sh, TrCtl* ctl, unsigned bit) {
  *reinterpret_cast<volatile int*>(&sh.abort) = 1;
  atomicOr(&ctl->err, bit);
}

// parents[0] == -1, 0 <= parents[i] < i, depth <= max_depth; depths by pointer
// jumping (depth[i] accumulates along ever longer ancestor jumps), with the
// still idle stage ring as scratch.  Result in sh.topo_ok and sh.depth.  All
// threads of the CTA take part.
__device__ void tree_topology(const TreeArgs& a, TrShared& sh, unsigned char* ring) {
  short(*anc)[TR_MAX_N] = reinterpret_cast<short(*)[TR_MAX_N]>(ring);
  unsigned short(*dep)[TR_MAX_N] = reinterpret_cast<unsigned short(*)[TR_MAX_N]>(ring + 2 * TR_MAX_N * sizeof(short));
  if (threadIdx.x == 0) sh.topo_ok = a.chain ? (a.N - 1 <= a.max_depth) : 1;
  __syncthreads();
  if (a.chain) {
    for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
      sh.par[i] = static_cast<short>(i - 1);
      sh.depth[i] = static_cast<unsigned short>(i);
    }
    __syncthreads();
    return;
  }
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const int p = a.parents[i];
    const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
    if (!ok) sh.topo_ok = 0;
    sh.par[i] = static_cast<short>(ok ? p : -1);
    anc[0][i] = static_cast<short>(i == 0 || !ok ? -1 : p);
    dep[0][i] = static_cast<unsigned short>(i == 0 || !ok ? 0 : 1);
  }
  __syncthreads();
  int cur = 0;
  for (int round = 0; round < 11; ++round) {   // 2^11 > TR_MAX_N: every chain is jumped to the root
    for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
      const int an = anc[cur][i];
      if (an >= 0) {
        dep[cur ^ 1][i] = static_cast<unsigned short>(dep[cur][i] + dep[cur][an]);
        anc[cur ^ 1][i] = anc[cur][an];
      } else {
        dep[cur ^ 1][i] = dep[cur][i];
        anc[cur ^ 1][i] = -1;
      }
    }
    __syncthreads();
    cur ^= 1;
  }
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const unsigned short d = dep[cur][i];
    sh.depth[i] = d;
    if (d > a.max_depth) sh.topo_ok = 0;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// producer (one thread)
// ---------------------------------------------------------------------------
template <class T>
__device__ void tr_producer(const TreeArgs& a, unsigned char* ring, TrShared& sh) {
  int stage = 0;
  uint32_t phase = 0;
  int last_parity[TR_NSTAGE];
#pragma unroll
  for (int s = 0; s < TR_NSTAGE; ++s) last_parity[s] = -1;
  auto next_stage = [&]() -> bool {
    if (tr_aborted(sh)) return false;
    if (!mbar_wait(&sh.empty[stage], phase ^ 1u, a.timeout_ns)) {
      tr_fail(sh, a.ctl, 1u);
      return false;
    }
    return true;
  };
  auto advance = [&]() {
    if (++stage == TR_NSTAGE) { stage = 0; phase ^= 1u; }
  };

  // implicit units: node 0 of every sequence, and in chain mode nodes 1..TR_AHEAD too
  const unsigned roots = static_cast<unsigned>(a.B) * static_cast<unsigned>(a.S);
  const unsigned implicit = (a.chain ? static_cast<unsigned>(min(a.N, TR_AHEAD + 1)) : 1u) * roots;
  const unsigned B = static_cast<unsigned>(a.B);
  bool ok = sh.topo_ok != 0;
  unsigned k = ok ? atomicAdd(&a.ctl->qhead, 1u) : 0u;
  while (ok) {
    const unsigned kc = k;
    k = atomicAdd(&a.ctl->qhead, 1u);   // next claim, in flight while this unit streams
    unsigned uid;
    if (kc < implicit) {
      const unsigned node = kc / roots;
      const unsigned r = kc - node * roots;
      uid = (r / a.S * a.N + node) * a.S + r % a.S;   // (b, node, slice j)
    } else {
      // wait until position kc is written, or every sequence is finished
      const unsigned q = kc - implicit;
      const uint64_t t0 = global_ns();
      unsigned v = 0;
      for (;;) {
        if (q < a.qcap && (v = ld_relaxed_u32(a.fifo + q)) != 0u) break;
        if (ld_relaxed_u32(&a.ctl->seqs_done) >= B || tr_aborted(sh)) break;
        if (global_ns() - t0 > a.timeout_ns) {
          tr_fail(sh, a.ctl, 2u);
          break;
        }
        __nanosleep(128);
      }
      if (v == 0u) break;
      uid = v - 1u;
      // a queued look-ahead row of a chain that has already finished is not needed
      if (a.chain && ld_relaxed_u32(a.sdone + uid / a.S / a.N) != 0u) continue;
    }
    const unsigned row = uid / a.S;   // b * N + node
    const int j = static_cast<int>(uid - row * a.S);
    const int e0 = j * a.L, e1 = min(a.V, e0 + a.L);
    const unsigned char* src = a.target + (static_cast<long long>(row) * a.V + e0) * T::esz;
    const uint32_t bytes = static_cast<uint32_t>((e1 - e0) * T::esz);
    for (uint32_t off = 0; off < bytes; off += TR_STAGE) {
      const uint32_t n = min(static_cast<uint32_t>(TR_STAGE), bytes - off);
      if (!next_stage()) { ok = false; break; }
      TrStageDesc& d = sh.desc[stage];
      d.stop = 0;
      d.uid = static_cast<int>(uid);
      d.e0 = e0 + static_cast<int>(off) / T::esz;
      d.n = static_cast<int>(n);
      d.flags = (off == 0 ? 1 : 0) | (off + n >= bytes ? 2 : 0);
      mbar_arrive_expect_tx(&sh.full[stage], n);
      bulk_g2s(ring + stage * TR_STAGE, src + off, n, &sh.full[stage]);
      last_parity[stage] = static_cast<int>(phase);
      advance();
    }
  }
  if (next_stage()) {
    sh.desc[stage].stop = 1;
    mbar_arrive(&sh.full[stage]);
    last_parity[stage] = -1;
  }
  // do not leave while a copy may still land in this CTA's shared memory
#pragma unroll
  for (int s = 0; s < TR_NSTAGE; ++s)
    if (last_parity[s] >= 0 && !mbar_wait(&sh.full[s], static_cast<uint32_t>(last_parity[s]), a.timeout_ns))
      atomicOr(&a.ctl->err, 8u);
}

// ---------------------------------------------------------------------------
// consumers (eight warps)
// ---------------------------------------------------------------------------
template <class T>
__device__ void tr_consumer(const TreeArgs& a, unsigned char* ring, TrShared& sh, int cw, int lane) {
  const int ctid = cw * 32 + lane;
  int stage = 0;
  uint32_t phase = 0;
  ArgmaxAcc acc;
  acc.init();
  for (;;) {
    if (__any_sync(0xffffffffu, tr_aborted(sh))) break;
    if (!__all_sync(0xffffffffu, mbar_wait(&sh.full[stage], phase, a.timeout_ns))) {
      tr_fail(sh, a.ctl, 4u);
      break;
    }
    const TrStageDesc d = sh.desc[stage];
    if (d.stop) break;
    if (d.flags & 1) acc.init();
    const int cur = stage;
    const uint4* buf = reinterpret_cast<const uint4*>(ring + stage * TR_STAGE);
    const int nvec = d.n >> 4;
#pragma unroll 4
    for (int v = ctid; v < nvec; v += TR_CT) {
      float x[T::vpe];
      T::unpack(buf[v], x);
      acc.template add<T::vpe>(x, d.e0 + v * T::vpe);
    }
    if (++stage == TR_NSTAGE) { stage = 0; phase ^= 1u; }
    if (!(d.flags & 2)) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[cur]);
      continue;
    }
    acc.finalize();
    acc.warp_reduce();
    if (lane == 0) {
      a.part[static_cast<long long>(d.uid) * TR_CW + cw] = acc.pack();
      __threadfence_block();
      const int prev = atomicAdd(&sh.unit_cnt[cur], 1);
      if (prev == TR_CW - 1) {
        sh.unit_cnt[cur] = 0;   // (before the stage is released: its next unit counts from zero)
        __threadfence_block();
        // The stage is released first: the release reduction below waits
        // until the unit's partials are visible device-wide, and the ring
        // should not wait with it.
        mbar_arrive(&sh.empty[cur]);
        red_release_add_u32(a.cnt + d.uid / a.S, 1u);
      } else {
        mbar_arrive(&sh.empty[cur]);
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// finisher (one warp)
// ---------------------------------------------------------------------------
__device__ void tr_write_invalid(const TreeArgs& a, int b, int status, int lane) {
  const int W = a.max_depth + 1;
  for (int j = lane; j < W; j += 32) {
    a.out_tokens[static_cast<long long>(b) * W + j] = -1;
    if (a.out_path) a.out_path[static_cast<long long>(b) * W + j] = -1;
  }
  if (lane == 0) a.num_accepted[b] = status;
}

// outputs of a finished sequence: path root -> best (root excluded), then g
__device__ void tr_write_path(const TreeArgs& a, const TrShared& sh, int b, int best, int g, int lane) {
  const int W = a.max_depth + 1;
  const int d = sh.depth[best];
  int32_t* out = a.out_tokens + static_cast<long long>(b) * W;
  int32_t* path = a.out_path ? a.out_path + static_cast<long long>(b) * W : nullptr;
  for (int j = d + 1 + lane; j < W; j += 32) {
    out[j] = -1;
    if (path) path[j] = -1;
  }
  if (lane == 0) {
    int node = best;
    for (int j = d - 1; j >= 0; --j) {
      out[j] = tr_token(a, b, node);
      if (path) path[j] = node;
      node = sh.par[node];
    }
    out[d] = g;
    if (path) path[d] = -1;
    a.num_accepted[b] = d;
  }
}

__device__ void tr_finisher(const TreeArgs& a, TrShared& sh, int lane) {
  const unsigned G = gridDim.x;
  int nseq = 0;
  int seq[TR_MAX_SEQ];
  for (unsigned b = blockIdx.x; b < static_cast<unsigned>(a.B) && nseq < TR_MAX_SEQ; b += G) seq[nseq++] = b;
  if (nseq == 0) return;
  if (!sh.topo_ok) {
    for (int s = 0; s < nseq; ++s) tr_write_invalid(a, seq[s], -1, lane);
    if (lane == 0) atomicAdd(&a.ctl->seqs_done, static_cast<unsigned>(nseq));
    return;
  }
  unsigned accm[TR_MAX_SEQ], resm[TR_MAX_SEQ];
  int best[TR_MAX_SEQ], bestg[TR_MAX_SEQ];
  bool live[TR_MAX_SEQ];
  int nlive = nseq;
#pragma unroll
  for (int s = 0; s < TR_MAX_SEQ; ++s) {
    accm[s] = (lane == 0) ? 1u : 0u;   // the root (node 0 = lane 0, word 0) is accepted
    resm[s] = 0u;
    best[s] = -1;
    bestg[s] = -1;
    live[s] = s < nseq;
    if (a.chain && s < nseq) {
      // the chain rule rejects the whole sequence for a draft token outside [0, V)
      bool bad = false;
      for (int t = lane; t < a.N - 1; t += 32) {
        const int x = tr_token(a, seq[s], t + 1);
        bad |= x < 0 || x >= a.V;
      }
      if (__any_sync(0xffffffffu, bad)) {
        tr_write_invalid(a, seq[s], -1, lane);
        live[s] = false;
        --nlive;
        if (lane == 0) {
          a.sdone[seq[s]] = 1u;
          atomicAdd(&a.ctl->seqs_done, 1u);
        }
      }
    }
  }
  const unsigned S = static_cast<unsigned>(a.S);
  uint64_t last_progress = global_ns();
  while (nlive > 0) {
    bool progress = false;
#pragma unroll
    for (int s = 0; s < TR_MAX_SEQ; ++s) {
      if (!live[s]) continue;
      const int b = seq[s];
      // poll the counters of this lane's accepted, unresolved nodes
      unsigned pend = accm[s] & ~resm[s], ready = 0u;
      for (unsigned m = pend; m; m &= m - 1u) {
        const int w = __ffs(m) - 1;
        const int node = lane + 32 * w;
        if (ld_relaxed_u32(a.cnt + static_cast<long long>(b) * a.N + node) == S) ready |= 1u << w;
      }
      // resolve the ready nodes one at a time, lowest (word, lane) first
      for (;;) {
        unsigned any_w = __reduce_or_sync(0xffffffffu, ready);
        if (!any_w) break;
        const int w = __ffs(any_w) - 1;
        const unsigned lanes = __ballot_sync(0xffffffffu, (ready >> w) & 1u);
        const int l = __ffs(lanes) - 1;
        const int node = l + 32 * w;
        if (lane == l) ready &= ~(1u << w);
        __threadfence();   // acquire: the partials counted by the node's counter are visible
        // merge the node's S x TR_CW partials (first index on ties)
        ArgmaxAcc acc;
        acc.init();
        const float2* pp = a.part + (static_cast<long long>(b) * a.N + node) * S * TR_CW;
        for (int i = lane; i < static_cast<int>(S) * TR_CW; i += 32) {
          const float2 p = __ldcg(pp + i);
          acc.merge(p.x, __float_as_int(p.y));
        }
        acc.warp_reduce();
        const int g = acc.idx;
        if (acc.best != acc.best || g == kIdxNone) {   // NaN in an accepted node's row
          tr_write_invalid(a, b, -1, lane);
          live[s] = false;
          --nlive;
          if (lane == 0) {
            if (a.chain) a.sdone[b] = 1u;
            atomicAdd(&a.ctl->seqs_done, 1u);
          }
          progress = true;
          break;
        }
        if (lane == l) resm[s] |= 1u << w;
        const int dn = sh.depth[node];
        if (best[s] < 0 || dn > sh.depth[best[s]] || (dn == sh.depth[best[s]] && node < best[s])) {
          best[s] = node;
          bestg[s] = g;
        }
        // children of `node` whose token equals g are accepted; their units
        // are appended to the FIFO (c % 32 == lane, so each lane owns its bits).
        // In chain mode the accepted child's row is already queued (TR_AHEAD
        // rows ahead), so the row TR_AHEAD beyond it is appended instead.
        for (int c0 = (node + 1) & ~31; c0 < a.N; c0 += 32) {
          const int c = c0 + lane;
          const bool take = c > node && c < a.N && sh.par[c] == node && tr_token(a, b, c) == g;
          const unsigned tb = __ballot_sync(0xffffffffu, take);
          if (!tb) continue;
          if (take) accm[s] |= 1u << (c >> 5);
          const bool q_this = take && (!a.chain || c + TR_AHEAD < a.N);
          const unsigned qb = __ballot_sync(0xffffffffu, q_this);
          if (!qb) continue;
          unsigned base = 0;
          if (lane == 0) base = atomicAdd(&a.ctl->qtail, static_cast<unsigned>(__popc(qb)) * S);
          base = __shfl_sync(0xffffffffu, base, 0);
          if (q_this) {
            const unsigned r = __popc(qb & ((1u << lane) - 1u));
            const unsigned u0 = (static_cast<unsigned>(b) * a.N + (a.chain ? c + TR_AHEAD : c)) * S;
            for (unsigned j = 0; j < S; ++j) {
              const unsigned q = base + r * S + j;
              if (q < a.qcap) a.fifo[q] = u0 + j + 1u;
            }
          }
        }
        progress = true;
      }
      if (!live[s]) continue;
      // finished when no accepted node is left unresolved
      if (!__any_sync(0xffffffffu, (accm[s] & ~resm[s]) != 0u)) {
        tr_write_path(a, sh, b, best[s], bestg[s], lane);
        live[s] = false;
        --nlive;
        if (lane == 0) {
          if (a.chain) a.sdone[b] = 1u;
          atomicAdd(&a.ctl->seqs_done, 1u);
        }
        progress = true;
      }
    }
    __syncwarp();
    if (progress) {
      last_progress = global_ns();
      continue;
    }
    const bool stop = __any_sync(0xffffffffu, tr_aborted(sh) || global_ns() - last_progress > 4 * a.timeout_ns);
    if (stop) {
      if (lane == 0) tr_fail(sh, a.ctl, 32u);
      break;
    }
    __nanosleep(200);
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
constexpr size_t tr_smem_bytes() { return TR_NSTAGE * TR_STAGE + sizeof(TrShared) + 128; }

template <class T>
__global__ void __launch_bounds__(TR_THREADS, TR_CTAS_PER_SM) tree_greedy_kernel(const TreeArgs a) {
  extern __shared__ __align__(128) unsigned char tr_smem[];
  unsigned char* ring = tr_smem;
  TrShared& sh = *reinterpret_cast<TrShared*>(tr_smem + TR_NSTAGE * TR_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < TR_NSTAGE; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], TR_CW);
      sh.unit_cnt[s] = 0;
    }
    sh.abort = 0;
    mbar_fence_init();
  }
  tree_topology(a, sh, ring);   // ends with __syncthreads

  if (warp == 0) {
    if (lane == 0) tr_producer<T>(a, ring, sh);
  } else if (warp == TR_FIN_WARP) {
    tr_finisher(a, sh, lane);
  } else {
    tr_consumer<T>(a, ring, sh, warp - 1, lane);
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned left = atomicAdd(&a.ctl->left, 1u);
    if (left + 1u == gridDim.x) {
      __threadfence();
      if (ld_acquire_u32(&a.ctl->err) != 0u) {
        const int W = a.max_depth + 1;
        for (long long i = 0; i < static_cast<long long>(a.B) * W; ++i) {
          a.out_tokens[i] = -1;
          if (a.out_path) a.out_path[i] = -1;
        }
        for (int b = 0; b < a.B; ++b) a.num_accepted[b] = -2;
      }
    }
  }
}

}  // namespace sv
