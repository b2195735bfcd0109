// tree_draft.cuh -- top-k tree drafting: the children of every node of a
// static candidate tree take the tokens of the node's draft row in decreasing
// logit order, with their draft log-probabilities ("Speculative decoding and
// EAGLE", section "Make it": an EAGLE-style drafter whose tree branches are the
// top-k tokens at each node; exercise 4: the top-3 branches at each depth).
//
// One CTA per (sequence, node).  The CTA finds the node's children (the nodes
// whose parent it is, in index order) and checks the topology; a node without
// children has nothing to draft and leaves.  Otherwise the CTA streams the
// node's draft row once through a ring of shared-memory stages filled by bulk
// async copies and keeps
//   - per thread, the online softmax normaliser (m, sum 2^(z c - fl(m c))),
//     c = log2(e)/T;
//   - per CTA, in shared memory, the n best elements seen so far (n = the
//     node's number of children) as 64-bit keys (orderable float bits << 32 |
//     ~index): a larger key is a larger logit, or an equal logit at a smaller
//     index, so key order is the drafting order.  An element is offered to
//     the list only when its value reaches the CTA's bound: the value of the
//     list's last key, which n distinct elements reach.
// Child r of the node receives key r of the list.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int TD_THREADS = 256;
constexpr int TD_WARPS = TD_THREADS / 32;
constexpr int TD_MAX_N = 1024;
constexpr int TD_MAX_CHILDREN = 16;
constexpr int TD_STAGE = 4 * 16 * TD_THREADS;   // bytes per ring stage: 4 vectors per thread
constexpr int TD_NS = 3;                    // ring stages (4 CTAs of 256 threads fit an SM)

struct TreeDraftArgs {
  const unsigned char* draft;   // [B, N, V]
  const int32_t* parents;       // [N]
  int B, N, V;
  int max_children;             // a node with more children makes the topology invalid
  int vec;                      // rows may be read with 16-byte loads
  float c;                      // log2(e) / T
  int32_t* node_tokens;         // [B, N]
  float* node_logq;             // [B, N]
};

__device__ __forceinline__ uint32_t td_ord(float x) {   // monotone map of non-NaN floats to uint32, -inf > 0
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float td_unord(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ unsigned long long td_key(float x, int idx) {
  return (static_cast<unsigned long long>(td_ord(x)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}

// element i of a 16-byte vector, without indexing registers at run time
template <class T>
__device__ __forceinline__ float td_elem(const uint4& q, int i) {
  if constexpr (T::esz == 2) {
    const uint32_t w = (i & 4) ? ((i & 2) ? q.w : q.z) : ((i & 2) ? q.y : q.x);
    return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
  } else {
    return __uint_as_float((i & 2) ? ((i & 1) ? q.w : q.z) : ((i & 1) ? q.y : q.x));
  }
}

// Offer a key to the CTA's list top[0..n), kept in descending order.  At each
// level an atomic maximum leaves the larger of the level's key and the carried
// one in place, and the smaller is carried to the next level: no key is lost
// or duplicated, a level only grows, and a key carried into a level never
// exceeds the level above it, so the list is descending at every moment.  A
// key carried off the end lost to every key the list then held (and levels
// only grow), so the list ends as the n best keys offered.  The value of the
// last key is then published as the CTA's bound: n distinct elements reach it,
// so an element below it is not among the n best.
__device__ __forceinline__ void td_offer(unsigned long long* top, unsigned* bound, int n, unsigned long long key) {
  if (key < *reinterpret_cast<volatile unsigned long long*>(&top[n - 1])) return;   // n listed keys beat it
#pragma unroll 1
  for (int j = 0; j < n && key != 0ull; ++j) {
    const unsigned long long old = atomicMax(&top[j], key);
    key = old < key ? old : key;
  }
  const unsigned long long last = *reinterpret_cast<volatile unsigned long long*>(&top[n - 1]);
  if (last != 0ull) atomicMax(bound, static_cast<unsigned>(last >> 32));
}

// A first bound for a warp that has seen nothing else: the n-th largest of
// the lanes' values v, each a distinct element of the row (lanes holding no
// element pass -inf).  n distinct elements reach it, so nothing below it can
// be among the n best.  Returns -inf (no bound) when fewer than n lanes hold
// a finite value.
__device__ __forceinline__ float td_seed(float v, int n, int lane) {
  float kth = kNegInf;
#pragma unroll 1
  for (int r = 0; r < n; ++r) {
    float m = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    kth = m;
    const unsigned hit = __ballot_sync(0xffffffffu, v == m);
    if (lane == __ffs(hit) - 1) v = kNegInf;   // one lane per round leaves
  }
  return kth > kNegInf ? kth : kNegInf;   // a NaN kth (every lane NaN) is no bound either
}

template <class T>
__global__ void __launch_bounds__(TD_THREADS, 4) tree_draft_kernel(TreeDraftArgs a) {
  __shared__ int s_cnt[TD_MAX_N];            // children per node (topology check)
  __shared__ int s_children[TD_MAX_CHILDREN];
  __shared__ int s_wcnt[TD_WARPS];
  __shared__ int s_nchild;
  __shared__ int s_bad;
  __shared__ unsigned long long s_top[TD_MAX_CHILDREN];   // the CTA's best keys so far, descending
  __shared__ unsigned s_bound;                            // orderable value they all reach (0: none yet)
  __shared__ float2 s_norm[TD_WARPS];
  extern __shared__ __align__(128) unsigned char s_ring[];   // TD_NS * TD_STAGE bytes (vector rows only)
  __shared__ __align__(8) uint64_t s_full[TD_NS];
  __shared__ __align__(8) uint64_t s_empty[TD_NS];
  __shared__ int s_timeout;

  const int N = a.N, V = a.V;
  const int b = static_cast<int>(blockIdx.x / N), p = static_cast<int>(blockIdx.x % N);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < N; i += TD_THREADS) s_cnt[i] = 0;
  if (tid < TD_MAX_CHILDREN) s_top[tid] = 0ull;
  if (tid == 0) {
    s_nchild = 0;
    s_bad = 0;
    s_timeout = 0;
    s_bound = 0u;
  }
  __syncthreads();
  // The topology check runs in every CTA over the whole parent array, so all
  // CTAs of a malformed tree reach the same verdict; the children of p are
  // collected in index order (warp ballots, then a scan over the warps).
  for (int base = 0; base < N; base += TD_THREADS) {
    const int i = base + tid;
    int par = -1;
    if (i < N) {
      par = a.parents[i];
      const bool bad = (i == 0) ? (par != -1) : (par < 0 || par >= i);
      if (bad) s_bad = 1;
      else if (i > 0) atomicAdd(&s_cnt[par], 1);
    }
    const bool mine = i < N && i > 0 && par == p;
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) s_wcnt[warp] = __popc(m);
    __syncthreads();
    int off = s_nchild, tot = 0;
#pragma unroll
    for (int w = 0; w < TD_WARPS; ++w) {
      off += w < warp ? s_wcnt[w] : 0;
      tot += s_wcnt[w];
    }
    if (mine) {
      const int slot = off + __popc(m & ((1u << lane) - 1u));
      if (slot < TD_MAX_CHILDREN) s_children[slot] = i;
    }
    __syncthreads();
    if (tid == 0) s_nchild += tot;
    __syncthreads();
  }
  for (int i = tid; i < N; i += TD_THREADS)
    if (s_cnt[i] > a.max_children) s_bad = 1;
  __syncthreads();
  const int nchild = s_nchild;   // <= max_children <= TD_MAX_CHILDREN unless the topology is bad
  const bool topo_bad = s_bad != 0;

  int32_t* tok = a.node_tokens + static_cast<long long>(b) * N;
  float* lq = a.node_logq + static_cast<long long>(b) * N;
  const float qnan = __int_as_float(0x7fc00000);
  if (topo_bad) {   // the root's CTA marks every node of the sequence
    if (p == 0)
      for (int i = tid; i < N; i += TD_THREADS) {
        tok[i] = -1;
        lq[i] = qnan;
      }
    return;
  }
  if (p == 0 && tid == 0) {
    tok[0] = -1;
    lq[0] = 0.f;
  }
  if (nchild == 0) return;

  // ---- stream the row ------------------------------------------------------
  const unsigned char* row = a.draft + (static_cast<long long>(b) * N + p) * static_cast<long long>(V) * T::esz;
  const float c = a.c;
  StatsAcc acc;
  acc.init();
  // the CTA's bound as it stands: it only rises, so a stale read is still a
  // valid (lower) bound; every bound test admits equal values and the key
  // comparison orders ties
  auto bound = [&]() {
    const unsigned bo = *reinterpret_cast<volatile unsigned*>(&s_bound);
    return bo != 0u ? td_unord(bo) : kNegInf;
  };

  if (a.vec) {
    // The row streams through a ring of TD_NS shared-memory stages of
    // TD_STAGE bytes, filled by bulk async copies (one thread issues them; a
    // full mbarrier per stage counts the bytes, an empty one the warps that
    // are done with it).  A stage is one group of 4 vectors
    // per thread: one packed maximum serves the normaliser (one rescale at most
    // per group) and the bound test; exponents and sums run on packed fp32
    // pairs.  Vectors past the row's end read as -inf.
    constexpr int G = 4;
    const int nv = V / T::vpe;
    const long long row_bytes = static_cast<long long>(V) * T::esz;
    const int nchunks = static_cast<int>((row_bytes + TD_STAGE - 1) / TD_STAGE);
    const uint32_t ninf = T::esz == 2 ? 0xff80ff80u : __float_as_uint(kNegInf);
    if (tid == 0) {
      for (int st = 0; st < TD_NS; ++st) {
        mbar_init(&s_full[st], 1);
        mbar_init(&s_empty[st], TD_WARPS);
      }
      mbar_fence_init();
    }
    __syncthreads();
    auto issue = [&](int ch) {   // thread 0
      const int st = ch % TD_NS;
      const long long off = static_cast<long long>(ch) * TD_STAGE;
      const uint32_t bytes = static_cast<uint32_t>(min(static_cast<long long>(TD_STAGE), row_bytes - off));
      mbar_arrive_expect_tx(&s_full[st], bytes);
      bulk_g2s(s_ring + st * TD_STAGE, row + off, bytes, &s_full[st]);
    };
    int issued = 0;   // thread 0: chunks whose copies were issued
    if (tid == 0)
      for (; issued < min(TD_NS, nchunks); ++issued) issue(issued);
    // Warps run decoupled: a stage is refilled once every warp has released
    // it (the empty barrier), one chunk after its use, so no warp waits for
    // another except through the ring.
    bool tmo = false;
    int ch = 0;
    for (; ch < nchunks; ++ch) {
      const int st = ch % TD_NS;
      if (tid == 0 && ch > 0 && ch - 1 + TD_NS < nchunks) {
        const int pc = ch - 1;   // the previous chunk's stage: refill it once released
        if (!mbar_wait(&s_empty[pc % TD_NS], static_cast<uint32_t>((pc / TD_NS) & 1), 1000000000ull)) tmo = true;
        else issue(issued++);
      }
      if (!tmo && !mbar_wait(&s_full[st], static_cast<uint32_t>((ch / TD_NS) & 1), 1000000000ull)) tmo = true;
      if (__any_sync(0xffffffffu, tmo)) {
        s_timeout = 1;
        break;
      }
      const int v0 = ch * (TD_STAGE / 16) + tid;
      uint4 q[G];
      const uint4* sv4 = reinterpret_cast<const uint4*>(s_ring + st * TD_STAGE);
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const int v = v0 + u * TD_THREADS;
        q[u] = v < nv ? sv4[tid + u * TD_THREADS] : make_uint4(ninf, ninf, ninf, ninf);
      }
      __syncwarp();   // the warp has its copy of the stage: release it
      if (lane == 0) mbar_arrive(&s_empty[st]);
      // the group maximum (packed for bf16)
      float vm;
      if constexpr (T::esz == 2) {
        uint32_t m4[G];
#pragma unroll
        for (int u = 0; u < G; ++u) m4[u] = bf16x2_max(bf16x2_max(q[u].x, q[u].y), bf16x2_max(q[u].z, q[u].w));
        const uint32_t mx = bf16x2_max(bf16x2_max(m4[0], m4[1]), bf16x2_max(m4[2], m4[3]));
        vm = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
      } else {
        float vmu[G];
#pragma unroll
        for (int u = 0; u < G; ++u)
          vmu[u] = fmaxf(fmaxf(__uint_as_float(q[u].x), __uint_as_float(q[u].y)),
                         fmaxf(__uint_as_float(q[u].z), __uint_as_float(q[u].w)));
        vm = fmaxf(fmaxf(vmu[0], vmu[1]), fmaxf(vmu[2], vmu[3]));
      }
      if (vm > acc.m) {
        const float An = __fmul_rn(vm, c);
        acc.s = (acc.m == kNegInf) ? 0.f : acc.s * ex2_approx(__fadd_rn(-acc.nA, -An));
        acc.m = vm;
        acc.nA = -An;
      }
      const unsigned long long c2 = f2_pack(c, c), n2 = f2_pack(acc.nA, acc.nA);
      unsigned long long s2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
        if constexpr (T::esz == 2) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a0, a1;
            f2_unpack(f2_fma(bf16x2_to_f2(w[i]), c2, n2), a0, a1);
            s2 = f2_add(s2, f2_pack(ex2_approx(a0), ex2_approx(a1)));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; i += 2) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(w[i]), __uint_as_float(w[i + 1])), c2, n2), a0, a1);
            s2 = f2_add(s2, f2_pack(ex2_approx(a0), ex2_approx(a1)));
          }
        }
      }
      float s0, s1;
      f2_unpack(s2, s0, s1);
      acc.s += s0 + s1;
      float thr = bound();
      if (ch == 0) {
        // nothing listed yet: seed the bound from the lanes' group maxima
        const float kth = td_seed(vm, nchild, lane);
        if (kth > kNegInf) {
          if (lane == 0) atomicMax(&s_bound, td_ord(kth));
          thr = fmaxf(thr, kth);
        }
      }
      // NaN never passes the tests (bf16x2 max skips it; a NaN maximum fails
      // the comparison).  The elements that reach the bound are collected as
      // bits of a mask and offered one by one.
      if (vm >= thr) {
        unsigned pass = 0u;
#pragma unroll
        for (int u = 0; u < G; ++u) {
          if (v0 + u * TD_THREADS < nv) {
            float x[T::vpe];
            T::unpack(q[u], x);
#pragma unroll
            for (int i = 0; i < T::vpe; ++i)
              if (x[i] >= thr) pass |= 1u << (u * T::vpe + i);
          }
        }
        while (pass != 0u) {
          const int bit = __ffs(pass) - 1;
          pass &= pass - 1u;
          const int u = bit / T::vpe, i = bit - u * T::vpe;
          const uint4 qq = u == 0 ? q[0] : u == 1 ? q[1] : u == 2 ? q[2] : q[3];
          td_offer(s_top, &s_bound, nchild, td_key(td_elem<T>(qq, i), (v0 + u * TD_THREADS) * T::vpe + i));
        }
      }
    }
    __syncthreads();
    if (s_timeout) {
      // let every copy still in flight land before this CTA leaves
      // (thread 0 has waited for every chunk before the one it stopped at;
      // the ones from there on are each the latest use of their stage)
      if (tid == 0)
        for (int c2 = ch; c2 < issued; ++c2)
          mbar_wait(&s_full[c2 % TD_NS], static_cast<uint32_t>((c2 / TD_NS) & 1), 1000000000ull);
      __syncthreads();
      if (tid < nchild && tid < TD_MAX_CHILDREN) {
        tok[s_children[tid]] = -2;
        lq[s_children[tid]] = qnan;
      }
      return;
    }
  } else {
    // element loads (rows not 16-byte aligned): rounds of one element per
    // thread, all lanes of a warp in every round
    for (int base = 0; base < V; base += TD_THREADS) {
      const int e = base + tid;
      float x[T::vpe];
      x[0] = e < V ? T::load(row, e) : kNegInf;
#pragma unroll
      for (int i = 1; i < T::vpe; ++i) x[i] = kNegInf;
      acc.template add<1>(x, c);
      float thr = bound();
      if (base == 0) {
        const float kth = td_seed(x[0], nchild, lane);
        if (kth > kNegInf) {
          if (lane == 0) atomicMax(&s_bound, td_ord(kth));
          thr = fmaxf(thr, kth);
        }
      }
      if (e < V && x[0] >= thr) td_offer(s_top, &s_bound, nchild, td_key(x[0], e));
    }
  }

  // ---- merge ----------------------------------------------------------------
  acc.warp_reduce(c);
  if (lane == 0) s_norm[warp] = acc.pack();
  __syncthreads();   // also: every offer to the list has completed
  if (warp != 0) return;
  StatsAcc tot;
  tot.init();
  if (lane < TD_WARPS) tot.unpack(s_norm[lane]);
  else tot.unpack(make_float2(kNegInf, 0.f));
  tot.nA = (tot.m == kNegInf) ? 0.f : -__fmul_rn(tot.m, c);
  tot.warp_reduce(c);

  // a row is usable iff its maximum is finite and its sum positive and finite
  // (NaN or +inf anywhere poison the sum; no finite entry leaves m = -inf)
  const bool row_ok = isfinite(tot.m) && isfinite(tot.s) && tot.s > 0.f;
  const float A = __fmul_rn(tot.m, c);
  const float l2s = row_ok ? log2f(tot.s) : 0.f;
  for (int r = lane; r < nchild; r += 32) {
    const unsigned long long key = s_top[r];
    const int child = s_children[r];
    if (!row_ok || key == 0ull) {
      tok[child] = -1;
      lq[child] = qnan;
    } else {
      const float z = td_unord(static_cast<uint32_t>(key >> 32));
      tok[child] = static_cast<int32_t>(~static_cast<uint32_t>(key));
      // log q = ln2 (z c - fl(M c) - log2 S), the exponent formed exactly:
      // the product's error by fma, the difference's by two-sum (Knuth)
      const float pz = __fmul_rn(z, c);
      const float pe = __fmaf_rn(z, c, -pz);
      const float hi = __fsub_rn(pz, A);
      const float bb = __fsub_rn(hi, pz);
      const float lo = __fadd_rn(__fsub_rn(pz, __fsub_rn(hi, bb)), __fsub_rn(-A, bb));
      lq[child] = 0.69314718f * __fadd_rn(__fsub_rn(hi, l2s), __fadd_rn(lo, pe));
    }
  }
}

}  // namespace sv
