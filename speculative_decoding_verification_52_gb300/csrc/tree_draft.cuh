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
// async copies and keeps, per thread,
//   - the online softmax normaliser (m, sum 2^(z c - fl(m c))), c = log2(e)/T;
//   - the KM best elements as 64-bit keys (orderable float bits << 32 |
//     ~index): a larger key is a larger logit, or an equal logit at a smaller
//     index, so key order is the drafting order.  Elements are offered to the
//     list only when they reach a bound that no element below it can beat: the
//     KM-th best key of the warp's lists, or of any warp of the CTA.
// The lists are merged per warp and then across warps in KM rounds of
// argmax extraction; child r of the node receives key r.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int TD_THREADS = 256;
constexpr int TD_WARPS = TD_THREADS / 32;
constexpr int TD_MAX_N = 1024;
constexpr int TD_MAX_CHILDREN = 16;
constexpr int TD_STAGE = 4 * 16 * TD_THREADS;   // bytes per ring stage: 4 vectors per thread
constexpr int TD_NS = 4;                    // ring stages
constexpr int TD_BOUND_EVERY = 4;           // groups between refreshes of the warp's top-KM bound (power of 2)

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

// insert key into the descending list k[0..KM) (the caller checked key > k[KM-1])
template <int KM>
__device__ __forceinline__ void td_insert(unsigned long long (&k)[KM], unsigned long long key) {
  k[KM - 1] = key;
#pragma unroll
  for (int j = KM - 1; j > 0; --j) {
    if (k[j] > k[j - 1]) {
      const unsigned long long t = k[j];
      k[j] = k[j - 1];
      k[j - 1] = t;
    }
  }
}

// KM rounds of warp-wide argmax extraction over the lanes' descending lists;
// every lane returns the merged top KM in out[] (the lanes' lists are consumed)
template <int KM>
__device__ __forceinline__ void td_warp_merge(unsigned long long (&k)[KM], unsigned long long (&out)[KM], int lane) {
#pragma unroll
  for (int r = 0; r < KM; ++r) {
    unsigned long long best = k[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    out[r] = best;
    // keys are unique (they carry the index), except the empty key 0
    const unsigned win = __ballot_sync(0xffffffffu, k[0] == best);
    if (lane == __ffs(win) - 1) {
#pragma unroll
      for (int j = 0; j + 1 < KM; ++j) k[j] = k[j + 1];
      k[KM - 1] = 0ull;
    }
  }
}

// the KM-th largest key in the union of the warp's lists (0 if the union holds
// fewer than KM keys): KM rounds of "each lane's largest key below the bound,
// then the warp's maximum"; keys are unique (they carry the index)
template <int KM>
__device__ __forceinline__ unsigned long long td_warp_kth(const unsigned long long (&k)[KM]) {
  unsigned long long bound = ~0ull, res = 0ull;
#pragma unroll
  for (int r = 0; r < KM; ++r) {
    unsigned long long mine = 0ull;
#pragma unroll
    for (int j = KM - 1; j >= 0; --j)
      if (k[j] < bound) mine = k[j];   // descending list: the last hit is the largest below the bound
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = __shfl_xor_sync(0xffffffffu, mine, o);
      mine = other > mine ? other : mine;
    }
    res = mine;
    bound = mine;
  }
  return res;
}

template <class T, int KM>
__global__ void __launch_bounds__(TD_THREADS) tree_draft_kernel(TreeDraftArgs a) {
  __shared__ int s_cnt[TD_MAX_N];            // children per node (topology check)
  __shared__ int s_children[TD_MAX_CHILDREN];
  __shared__ int s_wcnt[TD_WARPS];
  __shared__ int s_nchild;
  __shared__ int s_bad;
  __shared__ unsigned long long s_keys[TD_WARPS][KM];
  __shared__ float2 s_norm[TD_WARPS];
  extern __shared__ __align__(128) unsigned char s_ring[];   // TD_NS * TD_STAGE bytes (vector rows only)
  __shared__ __align__(8) uint64_t s_full[TD_NS];
  __shared__ __align__(8) uint64_t s_empty[TD_NS];
  __shared__ int s_timeout;
  __shared__ unsigned long long s_wkey[TD_WARPS];   // each warp's KM-th best key at its last refresh

  const int N = a.N, V = a.V;
  const int b = static_cast<int>(blockIdx.x / N), p = static_cast<int>(blockIdx.x % N);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < N; i += TD_THREADS) s_cnt[i] = 0;
  if (tid == 0) {
    s_nchild = 0;
    s_bad = 0;
    s_timeout = 0;
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
  const int nchild = s_nchild;
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
  unsigned long long k[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) k[j] = 0ull;
  bool full = false;
  float thr = kNegInf;    // value of the thread's KM-th best once its list is full
  bool wbound = false;    // some lane of the warp has a full list ...
  float wthr = kNegInf;   // ... and this is the largest such KM-th value (a bound for every lane)

  // insert the elements of one vector (index e0..) that beat the list
  auto insert_vec = [&](const float* x, int e0, int cnt) {
    // one compare per element against the tighter of the two bounds; with
    // neither (the list is not full and the warp holds fewer than KM keys)
    // every non-NaN element is examined
    const bool open = !wbound && !full;
    const float lim = fmaxf(wbound ? wthr : kNegInf, full ? thr : kNegInf);
    bool any = false;
#pragma unroll
    for (int i = 0; i < T::vpe; ++i) {
      if (i < cnt && (x[i] >= lim || (open && x[i] == x[i]))) {
        const unsigned long long key = td_key(x[i], e0 + i);
        if (key > k[KM - 1]) {
          td_insert<KM>(k, key);
          any = true;
        }
      }
    }
    if (any) {
      full = k[KM - 1] != 0ull;
      thr = full ? td_unord(static_cast<uint32_t>(k[KM - 1] >> 32)) : kNegInf;
    }
  };

  if (a.vec) {
    // The row streams through a ring of TD_NS shared-memory stages of
    // TD_STAGE bytes, filled by bulk async copies (one thread issues them; a
    // full mbarrier per stage counts the bytes, an empty one the warps that
    // are done with it).  A stage is one group of 4 vectors
    // per thread: one packed maximum serves the normaliser (one rescale at most
    // per group) and the top-k filter; exponents and sums run on packed fp32
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
    if (tid < TD_WARPS) s_wkey[tid] = 0ull;
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
      if (ch > 0 && ((ch - 1) & (TD_BOUND_EVERY - 1)) == 0) {
        // every warp's published bound is a bound for the whole CTA (each
        // warp's KM best are in the CTA's union): take the largest.  Warps
        // are not in step, so a bound may come from later indices: every
        // bound test admits equal values and the key comparison orders ties.
        unsigned long long ck = 0ull;
#pragma unroll
        for (int w = 0; w < TD_WARPS; ++w) {
          const unsigned long long wv = *reinterpret_cast<volatile unsigned long long*>(&s_wkey[w]);
          ck = wv > ck ? wv : ck;
        }
        if (ck != 0ull) {
          const float cv = td_unord(static_cast<uint32_t>(ck >> 32));
          wthr = wbound ? fmaxf(wthr, cv) : cv;
          wbound = true;
        }
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
      // per-vector maxima (packed for bf16), then the group maximum
      float vmu[G];
      float vm;
      if constexpr (T::esz == 2) {
        uint32_t m4[G];
#pragma unroll
        for (int u = 0; u < G; ++u) m4[u] = bf16x2_max(bf16x2_max(q[u].x, q[u].y), bf16x2_max(q[u].z, q[u].w));
        const uint32_t mx = bf16x2_max(bf16x2_max(m4[0], m4[1]), bf16x2_max(m4[2], m4[3]));
        vm = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
#pragma unroll
        for (int u = 0; u < G; ++u) vmu[u] = fmaxf(__uint_as_float(m4[u] << 16), __uint_as_float(m4[u] & 0xffff0000u));
      } else {
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
      if (ch == 0) {
        // No list holds anything yet: seed the bound with the KM-th largest of
        // the lanes' group maxima (KM distinct elements reach it, so nothing
        // below it can be in the top KM).  Indices interleave across lanes in
        // this group, so equal values must still be examined: the bound is
        // lowered by one ulp, and the bound tests admit equal values anyway.
        float v = vm, kth = kNegInf;
#pragma unroll
        for (int r = 0; r < KM; ++r) {
          float m = v;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          kth = m;
          const unsigned hit = __ballot_sync(0xffffffffu, v == m);
          if (lane == __ffs(hit) - 1) v = kNegInf;   // one lane per round leaves
        }
        wbound = kth > kNegInf;
        wthr = wbound ? nextafterf(kth, kNegInf) : kNegInf;
      }
      // NaN never passes these filters (bf16x2 max skips it; the sum above
      // turns NaN).  A warp takes this branch whenever one lane does, so the
      // per-vector test keeps the cost of the lanes that only follow small.
      if (!wbound || vm >= wthr) {
#pragma unroll
        for (int u = 0; u < G; ++u) {
          const int v = v0 + u * TD_THREADS;
          if (v < nv && (!wbound || vmu[u] >= wthr)) {
            float x[T::vpe];
            T::unpack(q[u], x);
            insert_vec(x, v * T::vpe, T::vpe);
          }
        }
      }
      // The KM-th best key of the union of the warp's lists bounds what can
      // still enter the warp's (hence the CTA's) top KM.  The bound tests admit
      // equal values and the key comparison then orders ties by index, so the
      // filter never drops a member of the top KM; an older bound is lower,
      // hence still valid, so it is refreshed only every TD_BOUND_EVERY groups.
      // Until the warp holds KM keys there is no bound and every group is
      // examined.
      if ((ch & (TD_BOUND_EVERY - 1)) == 0 || ch < 2) {
        // the exact bound: the KM-th best key the warp holds
        const unsigned long long wk = td_warp_kth<KM>(k);
        wbound = wk != 0ull;
        wthr = wbound ? td_unord(static_cast<uint32_t>(wk >> 32)) : kNegInf;
        if (lane == 0) *reinterpret_cast<volatile unsigned long long*>(&s_wkey[warp]) = wk;
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
    for (int e = tid; e < V; e += TD_THREADS) {
      float x[T::vpe];
      x[0] = T::load(row, e);
#pragma unroll
      for (int i = 1; i < T::vpe; ++i) x[i] = kNegInf;
      acc.template add<1>(x, c);
      if (!full || x[0] > thr) insert_vec(x, e, 1);
    }
  }

  // ---- merge ----------------------------------------------------------------
  acc.warp_reduce(c);
  unsigned long long wk[KM];
  td_warp_merge<KM>(k, wk, lane);
  if (lane == 0) {
    s_norm[warp] = acc.pack();
#pragma unroll
    for (int j = 0; j < KM; ++j) s_keys[warp][j] = wk[j];
  }
  __syncthreads();
  if (warp != 0) return;
  StatsAcc tot;
  tot.init();
  if (lane < TD_WARPS) tot.unpack(s_norm[lane]);
  else tot.unpack(make_float2(kNegInf, 0.f));
  tot.nA = (tot.m == kNegInf) ? 0.f : -__fmul_rn(tot.m, c);
  tot.warp_reduce(c);
  unsigned long long lk[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) lk[j] = lane < TD_WARPS ? s_keys[lane][j] : 0ull;
  unsigned long long fk[KM];
  td_warp_merge<KM>(lk, fk, lane);

  // a row is usable iff its maximum is finite and its sum positive and finite
  // (NaN or +inf anywhere poison the sum; no finite entry leaves m = -inf)
  const bool row_ok = isfinite(tot.m) && isfinite(tot.s) && tot.s > 0.f;
  const float A = __fmul_rn(tot.m, c);
  const float l2s = row_ok ? log2f(tot.s) : 0.f;
  for (int r = lane; r < nchild; r += 32) {
    unsigned long long key = 0ull;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j == r) key = fk[j];
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
