// spec_verify.cu -- host side of the C ABI declared in include/spec_verify.h:
// argument validation, workspace layout, launch configuration, kernel dispatch.
//
// Pipeline of one call (all launches on the caller's stream, no sync):
//   1. sweep      persistent grid over every (row, slice) unit: per-slice
//                 softmax-normaliser partials (sampling) or argmax partials
//                 (greedy, tree) into the workspace;
//   2. finish     per-sequence decisions: the greedy chain rule (one warp per
//                 sequence), the greedy tree rule (one CTA per sequence) or the
//                 sampling rule (one thread-block cluster per sequence, which
//                 re-reads only the stopping row pair).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "finish.cuh"
#include "fused.cuh"
#include "spec_verify.h"
#include "sweep.cuh"
#include "tree.cuh"
#include "tree_mask.cuh"
#include "kv_commit.cuh"
#include "row_stats.cuh"
#include "row_stats_stream.cuh"
#include "tree_draft.cuh"

namespace {

using namespace sv;

thread_local char g_err[512] = "";

spec_status_t fail(spec_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

spec_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(SPEC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMinSlice = 2048;            // smallest sweep slice (elements)
constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitNs = 1000000000ull;   // bounded waits: 1 s

int max_slices(int V) { return std::max(1, (V + kMinSlice - 1) / kMinSlice); }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

struct DevInfo {
  bool ready = false;
  int sms = 0;
  int max_cluster = 8;
};
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

// Unique id of the calling thread's current CUDA context, plus one (0: no
// context yet, or the driver entry points are unavailable).  A device reset or
// a re-created primary context gets a new id, so per-device caches keyed on it
// are set up again instead of reusing state of a context that is gone.
unsigned long long current_ctx_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(fn);
    cudaGetLastError();
  });
  if (!get_current || !get_id) return 0;
  void* ctx = nullptr;
  if (get_current(&ctx) != 0 || !ctx) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != 0) return 0;
  return id + 1;
}

// per-kernel one-time attribute setup, per device and context (attributes do
// not survive a device reset); without a context id it runs every time
template <class F>
bool once_per_device(int dev, F&& f) {
  static unsigned long long done[kMaxDevices] = {};   // context id the setup ran in
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 0 || dev >= kMaxDevices) return false;
  const unsigned long long id = current_ctx_id();
  if (id == 0 || done[dev] != id) {
    if (!f()) return false;
    done[dev] = current_ctx_id();   // (the setup may have created the context)
  }
  return true;
}

spec_status_t device_info(DevInfo& out, int& dev) {
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    int major = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (major < 10) return fail(SPEC_ERR_UNSUPPORTED, "compute capability %d.x: this library is built for sm_103a", major);
    d.ready = true;
  }
  out = d;
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// sweep configuration
// ---------------------------------------------------------------------------
// Pick the slice count S: slices of 8k-32k elements, enough units to cover the
// grid, and the least tail imbalance (max units per CTA x slice length).
void choose_slices(int V, long long rows, int grid, int& S, int& L) {
  const int smax = max_slices(V);
  int lo = std::max(1, ceil_div(V, 32768));
  lo = std::max(lo, static_cast<int>(std::min<long long>(smax, (grid + rows - 1) / rows)));
  lo = std::min(lo, smax);
  int hi = std::max(lo, std::min(smax, ceil_div(V, 8192)));
  long long best_cost = -1;
  S = lo;
  L = V;
  for (int s = lo; s <= hi; ++s) {
    int l = ceil_div(V, s);
    l = (l + 7) / 8 * 8;
    const int s_eff = ceil_div(V, l);
    const long long units = rows * s_eff;
    const long long per_cta = (units + grid - 1) / grid;
    const long long cost = per_cta * l;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      S = s_eff;
      L = l;
    }
  }
}

// occupancy of the TMA sweep (resident CTAs per SM); also sets its shared-memory limit
template <class TA, class TB, int MODE>
int sweep_per_sm(int dev) {
  static int per_sm[kMaxDevices];
  auto kern = sweep_tma_kernel<TA, TB, MODE>;
  once_per_device(dev, [&] {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SW_SMEM) != cudaSuccess) return false;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, SW_THREADS, SW_SMEM) != cudaSuccess) return false;
    per_sm[dev] = std::max(1, n);
    return true;
  });
  return per_sm[dev];
}

// Launch the sweep over rows [seg0 rows0 | seg1 rows1]; returns the slice count used.
template <class TA, class TB, int MODE>
spec_status_t launch_sweep(const DevInfo& di, int dev, bool vec, const unsigned char* seg0, long long rows0,
                           const unsigned char* seg1, long long rows1, int V, float c, float2* part,
                           cudaStream_t st, int& S_out) {
  const long long rows = rows0 + rows1;
  SweepArgs a{};
  a.seg0 = seg0;
  a.seg1 = seg1;
  a.rows0 = rows0;
  a.V = V;
  a.c = c;
  a.part = part;
  a.timeout_ns = kWaitNs;
  if (vec) {
    const int per_sm = sweep_per_sm<TA, TB, MODE>(dev);
    if (per_sm <= 0) return fail(SPEC_ERR_CUDA, "sweep kernel setup failed: %s", cudaGetErrorString(cudaGetLastError()));
    const int grid_cap = di.sms * per_sm;
    choose_slices(V, rows, grid_cap, a.S, a.L);
    a.units = rows * a.S;
    const int grid = static_cast<int>(std::min<long long>(a.units, grid_cap));
    sweep_tma_kernel<TA, TB, MODE><<<grid, SW_THREADS, SW_SMEM, st>>>(a);
  } else {
    const int grid_cap = di.sms * 8;
    choose_slices(V, rows, grid_cap, a.S, a.L);
    a.units = rows * a.S;
    const int grid = static_cast<int>(std::min<long long>(a.units, grid_cap));
    sweep_scalar_kernel<TA, TB, MODE><<<grid, SS_THREADS, 0, st>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sweep launch");
  S_out = a.S;
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// test hooks of the sampling path, passed down by the diagnostic entry points
// (spec_debug_residual: force a stop and dump the residual row; spec_debug_stall:
// one sequence's accept scan waits for a sweep unit that never comes, with a
// short wait limit).  Production calls pass none.
// ---------------------------------------------------------------------------
struct SampleHooks {
  int debug_b = -1, debug_t = -1;
  float* debug_row = nullptr;
  float* debug_mass = nullptr;
  int stall_b = -1;
  unsigned long long timeout_ns = 0;
  bool applied = false;   // set when the fused kernel took the hooks
};

// ---------------------------------------------------------------------------
// profiling events
// ---------------------------------------------------------------------------
struct Prof {
  bool on = false;
  int max_calls = 0;
  int calls = 0;
  std::vector<cudaEvent_t> ev;
} g_prof;

void prof_mark(int slot, cudaStream_t st) {
  if (!g_prof.on || g_prof.calls >= g_prof.max_calls) return;
  cudaEventRecord(g_prof.ev[3 * g_prof.calls + slot], st);
  if (slot == 2) ++g_prof.calls;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int esz_of(spec_dtype_t d) { return d == SPEC_BF16 ? 2 : 4; }
bool dtype_ok(spec_dtype_t d) { return d == SPEC_F32 || d == SPEC_BF16; }

// ---------------------------------------------------------------------------
// greedy chain
// ---------------------------------------------------------------------------
template <class T>
spec_status_t run_tree_pruned(const DevInfo& di, int dev, const void* target, const int32_t* parents,
                              const int32_t* node_tokens, int B, int N, int V, int max_depth, int32_t* out,
                              int32_t* nacc, int32_t* path, void* ws, cudaStream_t st, bool chain);

template <class T>
spec_status_t run_greedy(const DevInfo& di, int dev, const void* target, const int32_t* tokens, int B, int K, int V,
                         int32_t* out, int32_t* nacc, void* ws, cudaStream_t st) {
  const bool vec = aligned16(target) && (static_cast<long long>(V) * T::esz) % 16 == 0;
  if (vec) {
    // the chain as a tree of K+1 nodes: rows after the first mismatch are not read
    const spec_status_t s = run_tree_pruned<T>(di, dev, target, nullptr, tokens, B, K + 1, V, K, out, nacc, nullptr,
                                               ws, st, true);
    if (s != SPEC_ERR_UNSUPPORTED) return s;
  }
  // full sweep of the K+1 target rows, then one warp per sequence
  const long long rows = static_cast<long long>(B) * (K + 1);
  float2* part = reinterpret_cast<float2*>(ws);
  prof_mark(0, st);
  int S = 0;
  spec_status_t s = launch_sweep<T, T, MODE_ARGMAX>(di, dev, vec, static_cast<const unsigned char*>(target), rows,
                                                    nullptr, 0, V, 0.f, part, st, S);
  if (s != SPEC_OK) return s;
  prof_mark(1, st);
  FinishGreedyArgs a{};
  a.part = part;
  a.tokens = tokens;
  a.B = B;
  a.K = K;
  a.V = V;
  a.S = S;
  a.out_tokens = out;
  a.num_accepted = nacc;
  finish_greedy_kernel<<<ceil_div(B, FG_THREADS / 32), FG_THREADS, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "greedy finish launch");
  prof_mark(2, st);
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// sampling
// ---------------------------------------------------------------------------
template <class TP, class TQ, bool PROBS, bool VEC>
spec_status_t launch_finish_sample(const DevInfo& di, int dev, const FinishSampleArgs& a, int CL, cudaStream_t st) {
  auto kern = finish_sample_kernel<TP, TQ, PROBS, VEC>;
  const size_t smem = fs_smem_bytes(a.L);
  if (!once_per_device(dev, [&] {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return false;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(fs_smem_bytes(FS_MAX_L))) != cudaSuccess)
          return false;
        return true;
      }))
    return fail(SPEC_ERR_CUDA, "finish kernel setup failed: %s", cudaGetErrorString(cudaGetLastError()));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B) * CL);
  cfg.blockDim = dim3(FS_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return cuda_fail(e, "sampling finish launch");
  return SPEC_OK;
}

// largest usable cluster size for the sampling finisher on this device
template <class TP, class TQ, bool PROBS, bool VEC>
int finish_max_cluster(int dev) {
  static int mc[kMaxDevices];
  auto kern = finish_sample_kernel<TP, TQ, PROBS, VEC>;
  once_per_device(dev, [&] {
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(fs_smem_bytes(FS_MAX_L)));
    mc[dev] = 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(FS_THREADS);
    cfg.dynamicSmemBytes = fs_smem_bytes(FS_MAX_L);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) mc[dev] = 16;
    cudaGetLastError();
    return true;
  });
  return mc[dev] > 0 ? mc[dev] : 8;
}

// Workspace of the fused sampling kernel:
//   [FuCtl | flags[B * FU_FLAG_STRIDE]]   cleared by the kernel
//   [info[B] | bsum[B * ceil(V/256)] | part[rows * S] (float4)]
struct FusedLayout {
  size_t zero_bytes, info_off, bsum_off, part_off, total;
};
FusedLayout fused_layout(int B, int K, int V) {
  FusedLayout l{};
  const size_t nb = static_cast<size_t>((V + FU_BLK - 1) / FU_BLK);
  l.zero_bytes = align_up(32 + sizeof(unsigned) * FU_FLAG_STRIDE * static_cast<size_t>(B), 32);
  l.info_off = l.zero_bytes;
  l.bsum_off = align_up(l.info_off + sizeof(SeqInfo) * static_cast<size_t>(B), 16);
  l.part_off = align_up(l.bsum_off + sizeof(float) * static_cast<size_t>(B) * nb, 16);
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(2 * K + 1);
  l.total = align_up(l.part_off + rows * static_cast<size_t>(max_slices(V)) * sizeof(float4), 256);
  return l;
}

template <class TP, class TQ, bool PROBS>
int fused_per_sm(int dev) {
  static int per_sm[kMaxDevices];
  auto kern = fused_sample_kernel<TP, TQ, PROBS>;
  once_per_device(dev, [&] {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(fu_smem_bytes())) !=
        cudaSuccess)
      return false;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, FU_THREADS, fu_smem_bytes()) != cudaSuccess)
      return false;
    per_sm[dev] = std::max(1, n);
    return true;
  });
  return per_sm[dev];
}

template <class TP, class TQ, bool PROBS>
spec_status_t run_sample_fused(const DevInfo& di, int dev, const void* target, const void* draft,
                               const int32_t* tokens, const float* uni, float c, int B, int K, int V, int32_t* out,
                               int32_t* nacc, void* ws, SampleHooks* hooks, cudaStream_t st) {
  constexpr int QE = PROBS ? 4 : TQ::esz;
  const int per_sm = fused_per_sm<TP, TQ, PROBS>(dev);
  if (per_sm <= 0) return fail(SPEC_ERR_CUDA, "fused kernel setup failed: %s", cudaGetErrorString(cudaGetLastError()));
  // a cooperative launch: the grid never exceeds what is resident at once
  const int grid_cap = std::min(FU_MAX_GRID, di.sms * per_sm);
  const int RB = PROBS ? K + 1 : 2 * K + 1;
  const long long rows = static_cast<long long>(B) * RB;
  // Sweep slices are whole ring stages (a row's last slice ends in its only
  // partial stage), about four stages per unit; small batches use smaller
  // units so that every CTA gets at least two.
  const int smax = max_slices(V);
  const int stage_elems = FU_STAGE / std::max(TP::esz, QE);
  const int row_stages = ceil_div(V, stage_elems);
  int per_unit = 4;
  while (per_unit > 1 && rows * ceil_div(row_stages, per_unit) < 2LL * grid_cap) --per_unit;
  int L = per_unit * stage_elems;
  int S = ceil_div(V, L);
  if (S > smax) {   // (only for tiny per-unit sizes) keep the partial count within the workspace bound
    L = (ceil_div(V, smax) + 7) / 8 * 8;
    S = ceil_div(V, L);
  }
  const long long U = rows * S;
  const int RE = (TP::esz == 2 && QE == 2) ? 4096 : 2048;   // residual stage: 16 KB of P+Q at most
  const int Lr = 2 * RE;
  const int Sr = ceil_div(V, Lr);
  const long long RU = static_cast<long long>(B) * Sr;
  if (U >= (1LL << 31) || RU >= (1LL << 31)) return fail(SPEC_ERR_UNSUPPORTED, "batch too large for one call");

  const FusedLayout lay = fused_layout(B, K, V);
  unsigned char* w = static_cast<unsigned char*>(ws);
  FusedArgs a{};
  a.target = static_cast<const unsigned char*>(target);
  a.draft = static_cast<const unsigned char*>(draft);
  a.tokens = tokens;
  a.uni = uni;
  a.B = B;
  a.K = K;
  a.V = V;
  a.RB = RB;
  a.S = S;
  a.L = L;
  a.Sr = Sr;
  a.Lr = Lr;
  a.RE = RE;
  a.U = static_cast<unsigned>(U);
  a.c = c;
  a.NB = ceil_div(V, FU_BLK);
  a.ctl = reinterpret_cast<FuCtl*>(w);
  a.flags = reinterpret_cast<unsigned*>(w + 32);
  a.zero_words = static_cast<unsigned>(lay.zero_bytes / 16);
  a.info = reinterpret_cast<SeqInfo*>(w + lay.info_off);
  a.bsum = reinterpret_cast<float*>(w + lay.bsum_off);
  a.part = reinterpret_cast<float4*>(w + lay.part_off);
  a.out_tokens = out;
  a.num_accepted = nacc;
  a.debug_b = hooks ? hooks->debug_b : -1;
  a.debug_t = hooks ? hooks->debug_t : -1;
  a.debug_row = hooks ? hooks->debug_row : nullptr;
  a.debug_mass = hooks ? hooks->debug_mass : nullptr;
  a.timeout_ns = kWaitNs;
  a.debug_stall_b = -1;
  if (hooks && hooks->stall_b >= 0) {   // test hook (spec_debug_stall)
    a.debug_stall_b = hooks->stall_b;
    a.timeout_ns = hooks->timeout_ns;
    hooks->applied = true;
  }
  const long long work = U + RU;
  const int grid = static_cast<int>(std::min<long long>(grid_cap, work));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(FU_THREADS);
  cfg.dynamicSmemBytes = fu_smem_bytes();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(0, st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, fused_sample_kernel<TP, TQ, PROBS>, a);
  if (e != cudaSuccess) return cuda_fail(e, "fused sampling launch (cooperative)");
  prof_mark(1, st);
  prof_mark(2, st);
  return SPEC_OK;
}

template <class TP, class TQ, bool PROBS>
spec_status_t run_sample(const DevInfo& di, int dev, const void* target, const void* draft, const int32_t* tokens,
                         const float* uni, float T, int B, int K, int V, int32_t* out, int32_t* nacc, void* ws,
                         SampleHooks* hooks, cudaStream_t st) {
  constexpr int QE = PROBS ? 4 : TQ::esz;
  const bool vec = aligned16(target) && (static_cast<long long>(V) * TP::esz) % 16 == 0 &&
                   (K == 0 || (aligned16(draft) && (static_cast<long long>(V) * QE) % 16 == 0)) && V % 8 == 0;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  if (vec)
    return run_sample_fused<TP, TQ, PROBS>(di, dev, target, draft, tokens, uni, c, B, K, V, out, nacc, ws, hooks,
                                           st);

  // scalar path for unaligned rows: sweep kernel + clustered finishing kernel
  const long long rows0 = static_cast<long long>(B) * (K + 1);
  const long long rows1 = PROBS ? 0 : static_cast<long long>(B) * K;
  float2* part = reinterpret_cast<float2*>(ws);
  prof_mark(0, st);
  int S = 0;
  spec_status_t s = launch_sweep<TP, TQ, MODE_STATS>(di, dev, false, static_cast<const unsigned char*>(target), rows0,
                                                     static_cast<const unsigned char*>(draft), rows1, V, c, part, st, S);
  if (s != SPEC_OK) return s;
  prof_mark(1, st);

  FinishSampleArgs a{};
  a.target = static_cast<const unsigned char*>(target);
  a.draft = static_cast<const unsigned char*>(draft);
  a.tokens = tokens;
  a.uni = uni;
  a.part = part;
  a.B = B;
  a.K = K;
  a.V = V;
  a.S = S;
  a.c = c;
  a.out_tokens = out;
  a.num_accepted = nacc;
  a.debug_b = hooks ? hooks->debug_b : -1;
  a.debug_t = hooks ? hooks->debug_t : -1;
  a.debug_row = hooks ? hooks->debug_row : nullptr;
  a.debug_mass = hooks ? hooks->debug_mass : nullptr;

  const int maxcl = finish_max_cluster<TP, TQ, PROBS, false>(dev);
  int CL = std::min(maxcl, std::max(1, ceil_div(V, 8192)));
  int L = (ceil_div(V, CL) + 7) / 8 * 8;
  while (L > FS_MAX_L && CL < maxcl) {
    ++CL;
    L = (ceil_div(V, CL) + 7) / 8 * 8;
  }
  if (L > FS_MAX_L) return fail(SPEC_ERR_UNSUPPORTED, "V=%d exceeds the sampling limit (%d)", V, FS_MAX_L * maxcl);
  a.L = L;
  s = launch_finish_sample<TP, TQ, PROBS, false>(di, dev, a, CL, st);
  if (s != SPEC_OK) return s;
  prof_mark(2, st);
  return SPEC_OK;
}

spec_status_t dispatch_sample(const DevInfo& di, int dev, const void* target, spec_dtype_t tdt, const void* draft,
                              spec_dtype_t ddt, spec_draft_kind_t kind, const int32_t* tokens, const float* uni,
                              float T, int B, int K, int V, int32_t* out, int32_t* nacc, void* ws,
                              SampleHooks* hooks, cudaStream_t st) {
#define SV_RUN(TP, TQ, PR) run_sample<TP, TQ, PR>(di, dev, target, draft, tokens, uni, T, B, K, V, out, nacc, ws, hooks, st)
  const bool probs = kind == SPEC_DRAFT_PROBS;
  if (tdt == SPEC_BF16) {
    if (probs) return SV_RUN(BF16T, F32T, true);
    return ddt == SPEC_BF16 ? SV_RUN(BF16T, BF16T, false) : SV_RUN(BF16T, F32T, false);
  }
  if (probs) return SV_RUN(F32T, F32T, true);
  return ddt == SPEC_BF16 ? SV_RUN(F32T, BF16T, false) : SV_RUN(F32T, F32T, false);
#undef SV_RUN
}

// ---------------------------------------------------------------------------
// greedy tree, pruned (one persistent kernel)
// ---------------------------------------------------------------------------
// Workspace of the pruned tree kernel:
//   [TrCtl (128 B) | cnt[B*N] | fifo[B*(N-1)*S] | sdone[B]]   zeroed per call
//   [part[B*N*S*8]]
struct TreeLayout {
  size_t fifo_off, sdone_off, zero_bytes, part_off, total;
};
TreeLayout tree_layout(int B, int N, int S) {
  TreeLayout l{};
  const size_t nodes = static_cast<size_t>(B) * static_cast<size_t>(N);
  const size_t qcap = static_cast<size_t>(B) * static_cast<size_t>(N - 1) * static_cast<size_t>(S);
  l.fifo_off = align_up(128 + sizeof(unsigned) * nodes, 128);
  l.sdone_off = l.fifo_off + sizeof(unsigned) * qcap;
  l.zero_bytes = l.sdone_off + sizeof(unsigned) * static_cast<size_t>(B);
  l.part_off = align_up(l.zero_bytes, 256);
  l.total = align_up(l.part_off + nodes * static_cast<size_t>(S) * TR_CW * sizeof(float2), 256);
  return l;
}
// most slices a row can have: a unit is at least one 16 KB stage of f32
int tree_max_slices(int V) { return std::max(1, ceil_div(V, TR_STAGE / 4)); }

template <class T>
int tree_per_sm(int dev) {
  static int per_sm[kMaxDevices];
  auto kern = tree_greedy_kernel<T>;
  once_per_device(dev, [&] {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(tr_smem_bytes())) !=
        cudaSuccess)
      return false;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, TR_THREADS, tr_smem_bytes()) != cudaSuccess)
      return false;
    per_sm[dev] = std::max(1, n);
    return true;
  });
  return per_sm[dev];
}

// Returns SPEC_ERR_UNSUPPORTED (nothing launched) when the batch needs more
// sequences per finisher than the kernel holds; the caller then takes the
// full-sweep path.
template <class T>
spec_status_t run_tree_pruned(const DevInfo& di, int dev, const void* target, const int32_t* parents,
                              const int32_t* node_tokens, int B, int N, int V, int max_depth, int32_t* out,
                              int32_t* nacc, int32_t* path, void* ws, cudaStream_t st, bool chain) {
  const int per_sm = tree_per_sm<T>(dev);
  if (per_sm <= 0) return fail(SPEC_ERR_CUDA, "tree kernel setup failed: %s", cudaGetErrorString(cudaGetLastError()));
  const int grid = di.sms * per_sm;
  if (N > TR_MAX_N || B > TR_MAX_SEQ * grid) return SPEC_ERR_UNSUPPORTED;
  // units of up to 4 stages; smaller when the roots alone would not give every CTA two units
  const int stage_elems = TR_STAGE / T::esz;
  const int row_stages = ceil_div(V, stage_elems);
  int per_unit = 4;
  while (per_unit > 1 && static_cast<long long>(B) * ceil_div(row_stages, per_unit) < 2LL * grid) --per_unit;
  const int L = per_unit * stage_elems;
  const int S = ceil_div(V, L);
  if (static_cast<long long>(B) * N * S >= (1LL << 31)) return SPEC_ERR_UNSUPPORTED;
  const TreeLayout lay = tree_layout(B, N, S);
  unsigned char* w = static_cast<unsigned char*>(ws);
  TreeArgs a{};
  a.target = static_cast<const unsigned char*>(target);
  a.parents = parents;
  a.node_tokens = node_tokens;
  a.B = B;
  a.N = N;
  a.V = V;
  a.S = S;
  a.L = L;
  a.max_depth = max_depth;
  a.chain = chain ? 1 : 0;
  a.qcap = static_cast<unsigned>(static_cast<long long>(B) * (N - 1) * S);
  a.ctl = reinterpret_cast<TrCtl*>(w);
  a.cnt = reinterpret_cast<unsigned*>(w + 128);
  a.fifo = reinterpret_cast<unsigned*>(w + lay.fifo_off);
  a.sdone = reinterpret_cast<unsigned*>(w + lay.sdone_off);
  a.part = reinterpret_cast<float2*>(w + lay.part_off);
  a.out_tokens = out;
  a.num_accepted = nacc;
  a.out_path = path;
  a.timeout_ns = kWaitNs;
  cudaError_t e = cudaMemsetAsync(ws, 0, lay.zero_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "tree workspace reset");
  prof_mark(0, st);
  // a cooperative launch: the finisher of CTA b mod grid owns sequence b and
  // producers wait on FIFO slots other CTAs fill, so every CTA must be
  // resident; a grid that cannot be fails here instead of stalling
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(TR_THREADS);
  cfg.dynamicSmemBytes = tr_smem_bytes();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tree_greedy_kernel<T>, a);
  if (e != cudaSuccess) return cuda_fail(e, "tree kernel launch (cooperative)");
  prof_mark(1, st);
  prof_mark(2, st);
  return SPEC_OK;
}

spec_status_t check_chain_args(const void* target, spec_dtype_t tdt, const int32_t* tokens, int B, int K, int V,
                               int32_t* out, int32_t* nacc) {
  if (B < 0) return fail(SPEC_ERR_INVALID_ARG, "B=%d must be >= 0", B);
  if (K < 0 || K > SPEC_MAX_K) return fail(SPEC_ERR_INVALID_ARG, "K=%d outside [0, %d]", K, SPEC_MAX_K);
  if (V < 1) return fail(SPEC_ERR_INVALID_ARG, "V=%d must be >= 1", V);
  if (!dtype_ok(tdt)) return fail(SPEC_ERR_INVALID_ARG, "bad target dtype %d", static_cast<int>(tdt));
  if (B == 0) return SPEC_OK;
  if (!target || !out || !nacc) return fail(SPEC_ERR_INVALID_ARG, "NULL target/out_tokens/num_accepted");
  if (K > 0 && !tokens) return fail(SPEC_ERR_INVALID_ARG, "NULL draft_tokens with K > 0");
  if (static_cast<long long>(B) * (2 * K + 1) * static_cast<long long>(max_slices(V)) > (1LL << 40))
    return fail(SPEC_ERR_UNSUPPORTED, "batch too large");
  return SPEC_OK;
}

spec_status_t check_ws(void* ws, size_t have, size_t need) {
  if (need == 0) return SPEC_OK;
  if (!ws) return fail(SPEC_ERR_WORKSPACE, "NULL workspace (need %zu bytes)", need);
  if (!aligned16(ws)) return fail(SPEC_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  if (have < need) return fail(SPEC_ERR_WORKSPACE, "workspace %zu bytes < required %zu", have, need);
  return SPEC_OK;
}

spec_status_t sample_entry(const void* target, spec_dtype_t tdt, const void* draft, spec_dtype_t ddt,
                           spec_draft_kind_t kind, const int32_t* tokens, const float* uni, float T, int B, int K,
                           int V, int32_t* out, int32_t* nacc, void* ws, size_t wsb, SampleHooks* hooks,
                           void* stream) {
  spec_status_t s = check_chain_args(target, tdt, tokens, B, K, V, out, nacc);
  if (s != SPEC_OK || B == 0) return s;
  if (!(T >= 0.f) || !std::isfinite(T)) return fail(SPEC_ERR_INVALID_ARG, "temperature %g must be finite and >= 0", T);
  if (T > 0.f && T < 1e-4f) return fail(SPEC_ERR_UNSUPPORTED, "temperature %g below 1e-4", T);
  if (kind != SPEC_DRAFT_LOGITS && kind != SPEC_DRAFT_PROBS) return fail(SPEC_ERR_INVALID_ARG, "bad draft kind");
  if (kind == SPEC_DRAFT_PROBS && ddt != SPEC_F32) return fail(SPEC_ERR_INVALID_ARG, "draft probabilities must be f32");
  if (K > 0 && !dtype_ok(ddt)) return fail(SPEC_ERR_INVALID_ARG, "bad draft dtype %d", static_cast<int>(ddt));
  if (T > 0.f && (!uni || (K > 0 && !draft))) return fail(SPEC_ERR_INVALID_ARG, "NULL draft/uniforms");
  s = check_ws(ws, wsb, spec_workspace_bytes(B, K, V));
  if (s != SPEC_OK) return s;
  int dev;
  DevInfo di;
  s = device_info(di, dev);
  if (s != SPEC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0.f) {
    return tdt == SPEC_BF16 ? run_greedy<BF16T>(di, dev, target, tokens, B, K, V, out, nacc, ws, st)
                            : run_greedy<F32T>(di, dev, target, tokens, B, K, V, out, nacc, ws, st);
  }
  if (V > FS_MAX_L * 16) return fail(SPEC_ERR_UNSUPPORTED, "V=%d above the sampling limit %d", V, FS_MAX_L * 16);
  return dispatch_sample(di, dev, target, tdt, draft, K > 0 ? ddt : SPEC_F32, kind, tokens, uni, T, B, K, V, out,
                         nacc, ws, hooks, st);
}

// ---------------------------------------------------------------------------
// acceptance statistics (one cluster per position pair)
// ---------------------------------------------------------------------------
// Slice length and cluster size: the smallest power-of-two cluster (up to 8)
// whose per-CTA slice pair fits RS_TARGET_SMEM; beyond that the cluster stays at
// 8 and the slice grows up to RS_MAX_SMEM.  L is a multiple of 16 elements so
// every slice starts 16-byte aligned; CS = ceil(V / L) leaves no empty CTA.
bool row_stats_shape(int V, int bytes_per_pair, int& L, int& CS) {
  auto slice = [&](int cs) { return (ceil_div(V, cs) + 15) / 16 * 16; };
  int cs = 1;
  while (cs < RS_MAX_CLUSTER && static_cast<long long>(slice(cs)) * bytes_per_pair > RS_TARGET_SMEM) cs *= 2;
  L = slice(cs);
  CS = ceil_div(V, L);
  return static_cast<long long>(L) * bytes_per_pair <= RS_MAX_SMEM;
}

template <class TP, class TQ, bool PROBS>
spec_status_t launch_row_stats(int dev, const RowStatsArgs& a, cudaStream_t st) {
  auto kern = row_stats_kernel<TP, TQ, PROBS>;
  if (!once_per_device(dev, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RS_MAX_SMEM) == cudaSuccess;
      }))
    return fail(SPEC_ERR_CUDA, "row stats kernel setup failed: %s", cudaGetErrorString(cudaGetLastError()));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(a.B) * a.K * a.CS));
  cfg.blockDim = dim3(RS_THREADS);
  cfg.dynamicSmemBytes = static_cast<size_t>(a.L) * (TP::esz + TQ::esz);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.CS);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return cuda_fail(e, "row stats launch");
  return SPEC_OK;
}

// logits rows of one dtype that bulk copies can stream: one persistent CTA per
// SM, two passes over each position pair's rows (no exchange between CTAs)
template <class T>
spec_status_t launch_row_stats_stream(int dev, int sms, const RowStatsArgs& a, cudaStream_t st) {
  auto kern = row_stats_stream_kernel<T>;
  constexpr int smem = RT_NS * RT_STAGE;
  if (!once_per_device(dev, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
      }))
    return fail(SPEC_ERR_CUDA, "row stats kernel setup failed: %s", cudaGetErrorString(cudaGetLastError()));
  const long long pairs = static_cast<long long>(a.B) * a.K;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(pairs, std::max(1, sms)));
  kern<<<grid, RT_THREADS, smem, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "row stats launch");
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// top-k tree drafting
// ---------------------------------------------------------------------------
template <class T>
spec_status_t launch_tree_draft(int dev, unsigned grid, size_t smem, const TreeDraftArgs& a, cudaStream_t st) {
  auto kern = tree_draft_kernel<T>;
  if (!once_per_device(dev, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TD_NS * TD_STAGE) ==
               cudaSuccess;
      }))
    return fail(SPEC_ERR_CUDA, "tree draft kernel setup failed: %s", cudaGetErrorString(cudaGetLastError()));
  kern<<<grid, TD_THREADS, smem, st>>>(a);
  return SPEC_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// fixed scratch for spec_verify_sample_noalloc
// ---------------------------------------------------------------------------
// A file-scope device array stands in for the caller's workspace, so that call
// allocates nothing.  It holds kNoallocScratchBytes (16 MiB: the B=256, K=5,
// V=128256 batch needs 3.4 MB).  Every call on a device uses the same array:
// calls that may overlap on the GPU (other streams, other host threads) race
// on it.  The part of it that must start at zero (the fused kernel's control
// block and counters) is cleared on the call's stream by every call, exactly as
// for a caller-supplied workspace; the rest is written before it is read.
constexpr size_t kNoallocScratchBytes = static_cast<size_t>(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

// Device address of the array in the current device's context.  Resolved once
// per device and context, on the first call made with that device current;
// later calls in the same context only read the cached pointer.  A call in a
// new context of the device (after cudaDeviceReset, or once the primary
// context was released and re-created) resolves it again, since the array then
// lives at a new address.
spec_status_t noalloc_scratch(int dev, void** out) {
  static void* ptr[kMaxDevices] = {};
  static unsigned long long ctx[kMaxDevices] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_UNSUPPORTED, "device ordinal %d", dev);
  const unsigned long long id = current_ctx_id();
  if (!ptr[dev] || id == 0 || ctx[dev] != id) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fixed scratch)");
    if (!p) return fail(SPEC_ERR_CUDA, "cudaGetSymbolAddress returned a NULL scratch address");
    ptr[dev] = p;
    ctx[dev] = current_ctx_id();   // (the lookup may have created the context)
  }
  *out = ptr[dev];
  return SPEC_OK;
}

}  // namespace

// ===========================================================================
// exported C ABI
// ===========================================================================
extern "C" {

size_t spec_workspace_bytes(int B, int K, int V) {
  if (B < 0 || K < 0 || K > SPEC_MAX_K || V < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(2 * K + 1);
  const size_t plain = align_up(rows * static_cast<size_t>(max_slices(V)) * sizeof(float2), 256);
  const size_t chain = tree_layout(B, K + 1, tree_max_slices(V)).total;   // greedy rule, pruned kernel
  return std::max(std::max(plain, chain), fused_layout(B, K, V).total);
}

size_t spec_tree_workspace_bytes(int B, int N, int V) {
  if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(N);
  const size_t full = align_up(rows * static_cast<size_t>(max_slices(V)) * sizeof(float2), 256);
  return std::max(full, tree_layout(B, N, tree_max_slices(V)).total);
}

spec_status_t spec_verify_sample(const void* target_logits, spec_dtype_t target_dtype, const void* draft,
                                 spec_dtype_t draft_dtype, spec_draft_kind_t draft_kind, const int32_t* draft_tokens,
                                 const float* uniforms, float temperature, int B, int K, int V, int32_t* out_tokens,
                                 int32_t* num_accepted, void* workspace, size_t workspace_bytes, void* stream) {
  try {
    return sample_entry(target_logits, target_dtype, draft, draft_dtype, draft_kind, draft_tokens, uniforms,
                        temperature, B, K, V, out_tokens, num_accepted, workspace, workspace_bytes, nullptr, stream);
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_verify_sample_noalloc(const void* target_logits, spec_dtype_t target_dtype, const void* draft,
                                         spec_dtype_t draft_dtype, spec_draft_kind_t draft_kind,
                                         const int32_t* draft_tokens, const float* uniforms, float temperature, int B,
                                         int K, int V, int32_t* out_tokens, int32_t* num_accepted, void* stream) {
  try {
    const size_t need = spec_workspace_bytes(B, K, V);
    if (B == 0 || need == 0)   // empty batch or bad sizes: argument checks only, nothing launched
      return sample_entry(target_logits, target_dtype, draft, draft_dtype, draft_kind, draft_tokens, uniforms,
                          temperature, B, K, V, out_tokens, num_accepted, nullptr, 0, nullptr, stream);
    if (need > kNoallocScratchBytes)
      return fail(SPEC_ERR_UNSUPPORTED,
                  "B=%d K=%d V=%d needs %zu scratch bytes; spec_verify_sample_noalloc holds %zu "
                  "(use spec_verify_sample with a caller workspace)",
                  B, K, V, need, kNoallocScratchBytes);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    void* ws = nullptr;
    spec_status_t s = noalloc_scratch(dev, &ws);
    if (s != SPEC_OK) return s;
    return sample_entry(target_logits, target_dtype, draft, draft_dtype, draft_kind, draft_tokens, uniforms,
                        temperature, B, K, V, out_tokens, num_accepted, ws, kNoallocScratchBytes, nullptr, stream);
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_debug_residual(const void* target_logits, spec_dtype_t target_dtype, const void* draft,
                                  spec_dtype_t draft_dtype, spec_draft_kind_t draft_kind, const int32_t* draft_tokens,
                                  const float* uniforms, float temperature, int B, int K, int V, int debug_b,
                                  int debug_t, float* out_row, float* out_mass, int32_t* out_tokens,
                                  int32_t* num_accepted, void* workspace, size_t workspace_bytes, void* stream) {
  try {
    if (debug_b < 0 || debug_b >= B || debug_t < 0 || debug_t > K)
      return fail(SPEC_ERR_INVALID_ARG, "debug position (%d, %d) outside the batch", debug_b, debug_t);
    if (!out_row || !out_mass) return fail(SPEC_ERR_INVALID_ARG, "NULL out_row/out_mass");
    if (!(temperature > 0.f)) return fail(SPEC_ERR_INVALID_ARG, "the residual needs temperature > 0");
    SampleHooks hooks;
    hooks.debug_b = debug_b;
    hooks.debug_t = debug_t;
    hooks.debug_row = out_row;
    hooks.debug_mass = out_mass;
    return sample_entry(target_logits, target_dtype, draft, draft_dtype, draft_kind, draft_tokens, uniforms,
                        temperature, B, K, V, out_tokens, num_accepted, workspace, workspace_bytes, &hooks, stream);
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_verify_greedy(const void* target_logits, spec_dtype_t target_dtype, const int32_t* draft_tokens,
                                 int B, int K, int V, int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  try {
    spec_status_t s = check_chain_args(target_logits, target_dtype, draft_tokens, B, K, V, out_tokens, num_accepted);
    if (s != SPEC_OK || B == 0) return s;
    s = check_ws(workspace, workspace_bytes, spec_workspace_bytes(B, K, V));
    if (s != SPEC_OK) return s;
    int dev;
    DevInfo di;
    s = device_info(di, dev);
    if (s != SPEC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return target_dtype == SPEC_BF16
               ? run_greedy<BF16T>(di, dev, target_logits, draft_tokens, B, K, V, out_tokens, num_accepted, workspace, st)
               : run_greedy<F32T>(di, dev, target_logits, draft_tokens, B, K, V, out_tokens, num_accepted, workspace, st);
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_verify_tree_greedy(const void* target_logits, spec_dtype_t target_dtype, const int32_t* parents,
                                      const int32_t* node_tokens, int B, int N, int V, int max_depth,
                                      int32_t* out_tokens, int32_t* num_accepted, int32_t* out_path, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  try {
    if (B < 0) return fail(SPEC_ERR_INVALID_ARG, "B=%d must be >= 0", B);
    if (N < 1 || N > SPEC_MAX_TREE_NODES) return fail(SPEC_ERR_INVALID_ARG, "N=%d outside [1, %d]", N, SPEC_MAX_TREE_NODES);
    if (V < 1) return fail(SPEC_ERR_INVALID_ARG, "V=%d must be >= 1", V);
    if (max_depth < 0 || max_depth >= N) return fail(SPEC_ERR_INVALID_ARG, "max_depth=%d outside [0, N)", max_depth);
    if (!dtype_ok(target_dtype)) return fail(SPEC_ERR_INVALID_ARG, "bad target dtype");
    if (B == 0) return SPEC_OK;
    if (!target_logits || !parents || !node_tokens || !out_tokens || !num_accepted)
      return fail(SPEC_ERR_INVALID_ARG, "NULL pointer argument");
    spec_status_t s = check_ws(workspace, workspace_bytes, spec_tree_workspace_bytes(B, N, V));
    if (s != SPEC_OK) return s;
    int dev;
    DevInfo di;
    s = device_info(di, dev);
    if (s != SPEC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long rows = static_cast<long long>(B) * N;
    const int esz = esz_of(target_dtype);
    const bool vec = aligned16(target_logits) && (static_cast<long long>(V) * esz) % 16 == 0;
    if (vec) {
      // pruned: only accepted nodes' rows are swept
      s = target_dtype == SPEC_BF16
              ? run_tree_pruned<BF16T>(di, dev, target_logits, parents, node_tokens, B, N, V, max_depth, out_tokens,
                                       num_accepted, out_path, workspace, st, false)
              : run_tree_pruned<F32T>(di, dev, target_logits, parents, node_tokens, B, N, V, max_depth, out_tokens,
                                      num_accepted, out_path, workspace, st, false);
      if (s != SPEC_ERR_UNSUPPORTED) return s;
    }
    // full sweep of every node row, then one CTA per sequence resolves the tree
    float2* part = reinterpret_cast<float2*>(workspace);
    prof_mark(0, st);
    int S = 0;
    if (target_dtype == SPEC_BF16)
      s = launch_sweep<BF16T, BF16T, MODE_ARGMAX>(di, dev, vec, static_cast<const unsigned char*>(target_logits), rows,
                                                  nullptr, 0, V, 0.f, part, st, S);
    else
      s = launch_sweep<F32T, F32T, MODE_ARGMAX>(di, dev, vec, static_cast<const unsigned char*>(target_logits), rows,
                                                nullptr, 0, V, 0.f, part, st, S);
    if (s != SPEC_OK) return s;
    prof_mark(1, st);
    FinishTreeArgs a{};
    a.part = part;
    a.parents = parents;
    a.node_tokens = node_tokens;
    a.B = B;
    a.N = N;
    a.V = V;
    a.S = S;
    a.max_depth = max_depth;
    a.out_tokens = out_tokens;
    a.num_accepted = num_accepted;
    a.out_path = out_path;
    finish_tree_kernel<<<B, FT_THREADS, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "tree finish launch");
    prof_mark(2, st);
    return SPEC_OK;
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_tree_mask(const int32_t* parents, int B, int N, uint32_t* masks, int32_t* status, void* stream) {
  try {
    if (B < 0) return fail(SPEC_ERR_INVALID_ARG, "B=%d must be >= 0", B);
    if (N < 1 || N > TM_MAX_N) return fail(SPEC_ERR_INVALID_ARG, "N=%d outside [1, %d]", N, TM_MAX_N);
    if (B == 0) return SPEC_OK;
    if (!parents || !masks || !status) return fail(SPEC_ERR_INVALID_ARG, "NULL parents/masks/status");
    int dev;
    DevInfo di;
    spec_status_t s = device_info(di, dev);
    if (s != SPEC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int NW = (N + 31) / 32;
    const int grid = std::min(B, di.sms * 16);
    const size_t psmem = (sizeof(int) * static_cast<size_t>(N) + 15) & ~size_t(15);
    // rows of up to 16 words built run by run (the output base must allow the
    // vector stores: rows of NW words are then 4 * NW-byte aligned)
    const bool vec = (reinterpret_cast<uintptr_t>(masks) & 15u) == 0;
    auto rsmem = [&](int nwt) { return psmem + sizeof(uint32_t) * TM_THREADS * static_cast<size_t>(nwt); };
    prof_mark(0, st);
    if (vec && NW == 1) tree_mask_run_kernel<1><<<grid, TM_THREADS, rsmem(1), st>>>(parents, B, N, masks, status);
    else if (vec && NW == 2) tree_mask_run_kernel<2><<<grid, TM_THREADS, rsmem(2), st>>>(parents, B, N, masks, status);
    else if (vec && NW <= 4) tree_mask_run_kernel<4><<<grid, TM_THREADS, rsmem(4), st>>>(parents, B, N, masks, status);
    else if (vec && NW <= 8) tree_mask_run_kernel<8><<<grid, TM_THREADS, rsmem(8), st>>>(parents, B, N, masks, status);
    else if (vec && NW <= 16) tree_mask_run_kernel<16><<<grid, TM_THREADS, rsmem(16), st>>>(parents, B, N, masks, status);
    else {
      const size_t smem = psmem + sizeof(uint32_t) * TM_THREADS * NW;
      tree_mask_kernel<<<std::min(B, di.sms * 8), TM_THREADS, smem, st>>>(parents, B, N, masks, status);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "tree mask launch");
    prof_mark(1, st);
    prof_mark(2, st);
    return SPEC_OK;
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_kv_commit(void* cache, const int32_t* lengths, const void* scratch, const int32_t* path,
                             const int32_t* count, int B, int Lmax, int N, int W, size_t entry_bytes,
                             int32_t* new_lengths, void* stream) {
  try {
    if (B < 0 || Lmax < 0 || N < 1 || entry_bytes < 1 || (path && W < 1))
      return fail(SPEC_ERR_INVALID_ARG, "bad sizes B=%d Lmax=%d N=%d W=%d entry_bytes=%zu", B, Lmax, N, W, entry_bytes);
    if (B == 0) return SPEC_OK;
    if (!cache || !lengths || !scratch || !count || !new_lengths)
      return fail(SPEC_ERR_INVALID_ARG, "NULL cache/lengths/scratch/count/new_lengths");
    int dev;
    DevInfo di;
    spec_status_t s = device_info(di, dev);
    if (s != SPEC_OK) return s;
    KvCommitArgs a{};
    a.cache = static_cast<unsigned char*>(cache);
    a.lengths = lengths;
    a.scratch = static_cast<const unsigned char*>(scratch);
    a.path = path;
    a.count = count;
    a.B = B;
    a.Lmax = Lmax;
    a.N = N;
    a.W = path ? W : 0;
    a.J = path ? W : N;
    a.E = entry_bytes;
    a.new_lengths = new_lengths;
    a.vec = entry_bytes % 16 == 0 && aligned16(cache) && aligned16(scratch);
    const long long pairs = static_cast<long long>(B) * a.J;
    const int grid = static_cast<int>(std::min<long long>(pairs, static_cast<long long>(di.sms) * 16));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    prof_mark(0, st);
    kv_commit_kernel<<<grid, KV_THREADS, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kv commit launch");
    prof_mark(1, st);
    prof_mark(2, st);
    return SPEC_OK;
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_row_stats(const void* target_logits, spec_dtype_t target_dtype, const void* draft,
                             spec_dtype_t draft_dtype, spec_draft_kind_t draft_kind, float temperature, int B, int K,
                             int V, float* alpha, float* kl, float* tv, void* stream) {
  try {
    if (B < 0 || K < 0 || K > SPEC_MAX_K || V < 1)
      return fail(SPEC_ERR_INVALID_ARG, "bad sizes B=%d K=%d V=%d", B, K, V);
    if (!dtype_ok(target_dtype) || !dtype_ok(draft_dtype)) return fail(SPEC_ERR_INVALID_ARG, "bad dtype");
    if (draft_kind != SPEC_DRAFT_LOGITS && draft_kind != SPEC_DRAFT_PROBS)
      return fail(SPEC_ERR_INVALID_ARG, "bad draft kind");
    const bool probs = draft_kind == SPEC_DRAFT_PROBS;
    if (probs && draft_dtype != SPEC_F32) return fail(SPEC_ERR_INVALID_ARG, "draft probabilities must be float32");
    if (!(temperature > 0.f) || !std::isfinite(temperature))
      return fail(SPEC_ERR_INVALID_ARG, "temperature must be > 0 and finite");
    if (temperature < 1e-4f) return fail(SPEC_ERR_UNSUPPORTED, "temperature %g below 1e-4", temperature);
    if (B == 0 || K == 0) return SPEC_OK;
    if (!target_logits || !draft || !alpha || !kl || !tv)
      return fail(SPEC_ERR_INVALID_ARG, "NULL target/draft/alpha/kl/tv");
    const int ep = esz_of(target_dtype), eq = esz_of(draft_dtype);
    RowStatsArgs a{};
    a.target = static_cast<const unsigned char*>(target_logits);
    a.draft = static_cast<const unsigned char*>(draft);
    a.B = B;
    a.K = K;
    a.V = V;
    if (!row_stats_shape(V, ep + eq, a.L, a.CS))
      return fail(SPEC_ERR_UNSUPPORTED, "V=%d: a slice pair of %d bytes per CTA exceeds %d", V, a.L * (ep + eq),
                  RS_MAX_SMEM);
    if (static_cast<long long>(B) * K * a.CS > 0x7fffffffLL) return fail(SPEC_ERR_UNSUPPORTED, "grid too large");
    int dev;
    DevInfo di;
    spec_status_t s = device_info(di, dev);
    if (s != SPEC_OK) return s;
    a.vec = aligned16(target_logits) && aligned16(draft) && (static_cast<long long>(V) * ep) % 16 == 0 &&
            (static_cast<long long>(V) * eq) % 16 == 0;
    a.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    a.alpha = alpha;
    a.kl = kl;
    a.tv = tv;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    prof_mark(0, st);
    // The streaming kernel takes logits rows of one dtype that bulk copies can
    // stream and that do not fit one CTA's slice; a pair that fits one CTA is
    // cheaper in the cluster kernel (a cluster of one: no exchange, and every
    // pair a CTA of its own).
    if (!probs && a.vec && target_dtype == draft_dtype && a.CS > 1)
      s = target_dtype == SPEC_BF16 ? launch_row_stats_stream<BF16T>(dev, di.sms, a, st)
                                    : launch_row_stats_stream<F32T>(dev, di.sms, a, st);
    else if (probs)
      s = target_dtype == SPEC_BF16 ? launch_row_stats<BF16T, F32T, true>(dev, a, st)
                                    : launch_row_stats<F32T, F32T, true>(dev, a, st);
    else if (target_dtype == SPEC_BF16)
      s = draft_dtype == SPEC_BF16 ? launch_row_stats<BF16T, BF16T, false>(dev, a, st)
                                   : launch_row_stats<BF16T, F32T, false>(dev, a, st);
    else
      s = draft_dtype == SPEC_BF16 ? launch_row_stats<F32T, BF16T, false>(dev, a, st)
                                   : launch_row_stats<F32T, F32T, false>(dev, a, st);
    if (s != SPEC_OK) return s;
    prof_mark(1, st);
    prof_mark(2, st);
    return SPEC_OK;
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_tree_draft(const void* draft_logits, spec_dtype_t draft_dtype, const int32_t* parents, int B,
                              int N, int V, int max_children, float temperature, int32_t* node_tokens,
                              float* node_logq, void* stream) {
  try {
    if (B < 0 || N < 1 || N > TD_MAX_N || V < 1)
      return fail(SPEC_ERR_INVALID_ARG, "bad sizes B=%d N=%d V=%d (N in [1, %d])", B, N, V, TD_MAX_N);
    if (max_children < 1 || max_children > TD_MAX_CHILDREN)
      return fail(SPEC_ERR_INVALID_ARG, "max_children=%d outside [1, %d]", max_children, TD_MAX_CHILDREN);
    if (!dtype_ok(draft_dtype)) return fail(SPEC_ERR_INVALID_ARG, "bad dtype");
    if (!(temperature > 0.f) || !std::isfinite(temperature))
      return fail(SPEC_ERR_INVALID_ARG, "temperature must be > 0 and finite");
    if (temperature < 1e-4f) return fail(SPEC_ERR_UNSUPPORTED, "temperature %g below 1e-4", temperature);
    if (static_cast<long long>(B) * N > 0x7fffffffLL) return fail(SPEC_ERR_UNSUPPORTED, "grid too large");
    if (B == 0) return SPEC_OK;
    if (!draft_logits || !parents || !node_tokens || !node_logq)
      return fail(SPEC_ERR_INVALID_ARG, "NULL draft/parents/node_tokens/node_logq");
    int dev;
    DevInfo di;
    spec_status_t s = device_info(di, dev);
    if (s != SPEC_OK) return s;
    TreeDraftArgs a{};
    a.draft = static_cast<const unsigned char*>(draft_logits);
    a.parents = parents;
    a.B = B;
    a.N = N;
    a.V = V;
    a.max_children = max_children;
    const int esz = esz_of(draft_dtype);
    a.vec = aligned16(draft_logits) && (static_cast<long long>(V) * esz) % 16 == 0;
    a.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    a.node_tokens = node_tokens;
    a.node_logq = node_logq;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const unsigned grid = static_cast<unsigned>(static_cast<long long>(B) * N);
    prof_mark(0, st);
    const size_t smem = a.vec ? static_cast<size_t>(TD_NS) * TD_STAGE : 0;
    s = draft_dtype == SPEC_BF16 ? launch_tree_draft<BF16T>(dev, grid, smem, a, st)
                                 : launch_tree_draft<F32T>(dev, grid, smem, a, st);
    if (s != SPEC_OK) return s;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "tree draft launch");
    prof_mark(1, st);
    prof_mark(2, st);
    return SPEC_OK;
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_debug_stall(const void* target_logits, spec_dtype_t target_dtype, const void* draft,
                               spec_dtype_t draft_dtype, spec_draft_kind_t draft_kind, const int32_t* draft_tokens,
                               const float* uniforms, float temperature, int B, int K, int V, int stall_b,
                               unsigned timeout_us, int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                               size_t workspace_bytes, void* stream) {
  try {
    if (stall_b < 0 || stall_b >= B) return fail(SPEC_ERR_INVALID_ARG, "stall_b=%d outside the batch", stall_b);
    if (timeout_us < 100 || timeout_us > 1000000u)
      return fail(SPEC_ERR_INVALID_ARG, "timeout_us=%u outside [100, 1000000]", timeout_us);
    if (!(temperature > 0.f)) return fail(SPEC_ERR_INVALID_ARG, "the stall hook needs the sampling rule (T > 0)");
    SampleHooks hooks;
    hooks.stall_b = stall_b;
    hooks.timeout_ns = static_cast<unsigned long long>(timeout_us) * 1000ull;
    spec_status_t s = sample_entry(target_logits, target_dtype, draft, draft_dtype, draft_kind, draft_tokens,
                                   uniforms, temperature, B, K, V, out_tokens, num_accepted, workspace,
                                   workspace_bytes, &hooks, stream);
    if (s == SPEC_OK && !hooks.applied)
      return fail(SPEC_ERR_UNSUPPORTED, "the stall hook needs the fused sampling path (16-byte aligned rows)");
    return s;
  } catch (...) {
    return fail(SPEC_ERR_CUDA, "unexpected host exception");
  }
}

spec_status_t spec_profile_begin(int max_calls) {
  if (max_calls < 1) return fail(SPEC_ERR_INVALID_ARG, "max_calls must be >= 1");
  for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
  g_prof = Prof{};
  g_prof.ev.resize(static_cast<size_t>(3) * max_calls);
  for (auto& e : g_prof.ev) {
    cudaError_t r = cudaEventCreate(&e);
    if (r != cudaSuccess) return cuda_fail(r, "cudaEventCreate");
  }
  g_prof.max_calls = max_calls;
  g_prof.on = true;
  return SPEC_OK;
}

spec_status_t spec_profile_end(float* sweep_ms, float* finish_ms, int* calls) {
  if (!g_prof.on) return fail(SPEC_ERR_INVALID_ARG, "profiling was not started");
  g_prof.on = false;
  double a = 0.0, b = 0.0;
  for (int i = 0; i < g_prof.calls; ++i) {
    float t0 = 0.f, t1 = 0.f;
    cudaError_t r = cudaEventSynchronize(g_prof.ev[3 * i + 2]);
    if (r != cudaSuccess) return cuda_fail(r, "cudaEventSynchronize");
    cudaEventElapsedTime(&t0, g_prof.ev[3 * i], g_prof.ev[3 * i + 1]);
    cudaEventElapsedTime(&t1, g_prof.ev[3 * i + 1], g_prof.ev[3 * i + 2]);
    a += t0;
    b += t1;
  }
  if (sweep_ms) *sweep_ms = static_cast<float>(a);
  if (finish_ms) *finish_ms = static_cast<float>(b);
  if (calls) *calls = g_prof.calls;
  for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  return SPEC_OK;
}

const char* spec_status_string(spec_status_t s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
  }
  return "SPEC_ERR_UNKNOWN";
}

const char* spec_last_error(void) { return g_err; }

}  // extern "C"
