// C ABI entry points of libdash_attn: argument checks, schedule-table cache, the
// deadlock check of the persistent grid, and the kernel launches.
#include "dash_attn.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "bwd_aux.cuh"
#include "tc_shared.cuh"
#include "bwd_main.cuh"
#include "fwd_tc.cuh"
#include "gemm_splitk.cuh"
#include "sched.h"

static_assert(dash::kStatusBounds == DASH_ERR_BOUNDS, "bounds status: one code");
static_assert(dash::kStatusSyncTimeout == DASH_ERR_SYNC_TIMEOUT, "timeout status: one code");

namespace {

thread_local std::string g_last_error;

// Testing hooks (dash_debug_set_sync): bound on one semaphore wait and a skew added to
// every awaited ordinal (a skew > 0 makes every wait time out).
long long g_timeout_ns = 10ll * 1000 * 1000 * 1000;
int g_ordinal_skew = 0;
unsigned long long* g_trace = nullptr;   // dash_debug_set_trace
int g_check_narrow = 0;                  // dash_debug_narrow_checks (checked build only)

dash_status_t cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return DASH_ERR_CUDA;
}

#define DASH_CUDA(call)                                   \
  do {                                                    \
    cudaError_t e_ = (call);                              \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);   \
  } while (0)

struct DeviceTables {
  int32_t* tasks = nullptr;
  int32_t* ord = nullptr;
  int32_t* cnt = nullptr;
  int num_slots = 0;
  int num_tasks = 0;
};

std::mutex g_mu;
std::map<std::tuple<int, int, int, int>, DeviceTables> g_tables;        // (dev, mask, sched, n)
// (mask, sched, n, heads, grid, head dim)
std::map<std::tuple<int, int, int, int, int, int>, bool> g_deadlock_free;
// What one grid follows, per (dev, mask, sched, n, heads, grid, head dim): each CTA's
// pieces of work (dash::deal) and, for the arrival-ordered schedules, the per-head dQ
// orders.
struct DealtTables {
  int32_t* ord = nullptr;       // [heads][n][n]; null: the schedule's own order
  int32_t* cta_off = nullptr;   // [grid + 1]
  int32_t* pieces = nullptr;    // [pieces][4]: head, first task, end task, split/part
  int num_pieces = 0;
};
std::map<std::tuple<int, int, int, int, int, int, int>, DealtTables> g_dealt;

// The pieces in the kernel's 16-byte form: (head, first task, end task, (split << 2) | part).
std::vector<int32_t> piece_words(const dash::Dealing& dl) {
  std::vector<int32_t> w;
  w.reserve(4 * dl.pieces.size());
  for (const dash::Piece& pc : dl.pieces)
    w.insert(w.end(), {pc.head, pc.t_begin, pc.t_end, (pc.split << 2) | pc.part});
  return w;
}
// their host copies, (mask, sched, n, heads, grid): building one sorts every task of the
// shape, so it is done once per shape
std::map<std::tuple<int, int, int, int, int, int>, std::shared_ptr<const std::vector<int32_t>>>
    g_host_dealt;

// Host copy of the per-head dQ orders of an arrival-ordered schedule on `grid` CTAs at
// head dimension `head_dim` (cached; the caller holds g_mu).
std::shared_ptr<const std::vector<int32_t>> host_dealt_locked(const dash::Schedule& sc,
                                                              int heads, int grid,
                                                              int head_dim) {
  auto key = std::make_tuple(sc.mask, sc.sched, sc.n, heads, grid, head_dim);
  auto it = g_host_dealt.find(key);
  if (it == g_host_dealt.end()) {
    auto v = std::make_shared<std::vector<int32_t>>();
    dash::dealt_orders(sc, heads, grid, head_dim, v.get());
    it = g_host_dealt.emplace(key, std::move(v)).first;
  }
  return it->second;
}

dash_status_t get_tables(int dev, int mask, int sched, int n, DeviceTables* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, mask, sched, n);
  auto it = g_tables.find(key);
  if (it != g_tables.end()) {
    *out = it->second;
    return DASH_OK;
  }
  dash::Schedule sc;
  int rc = dash::build_schedule(mask, sched, n, &sc);
  if (rc) return (dash_status_t)rc;
  DeviceTables t;
  t.num_slots = sc.num_slots;
  t.num_tasks = (int)sc.tasks.size();
  auto upload = [](const std::vector<int32_t>& v, int32_t** dst) -> cudaError_t {
    cudaError_t e = cudaMalloc(dst, v.size() * sizeof(int32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, v.data(), v.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
  };
  DASH_CUDA(upload(sc.tasks, &t.tasks));
  DASH_CUDA(upload(sc.ord, &t.ord));
  DASH_CUDA(upload(sc.cnt, &t.cnt));
  g_tables[key] = t;
  *out = t;
  return DASH_OK;
}

// Copies a host table to a new device allocation (freed with the caches).
cudaError_t upload_new(const std::vector<int32_t>& v, int32_t** dst) {
  cudaError_t e = cudaMalloc(dst, v.size() * sizeof(int32_t));
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(*dst, v.data(), v.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(*dst);
    *dst = nullptr;
  }
  return e;
}

// Points p at what a grid of `grid` CTAs follows: each CTA's pieces (dash::deal) and the
// dQ orders -- the schedule's own table for ascending/descending (one order for all
// heads), the per-head arrival orders of dash::dealt_orders for shift and symmetric shift
// (cached per shape).
dash_status_t set_dealing(int dev, int mask, int sched, int n, int heads, int grid,
                          int head_dim, const DeviceTables& tb, dash::BwdParams* p) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, mask, sched, n, heads, grid, head_dim);
  auto it = g_dealt.find(key);
  if (it == g_dealt.end()) {
    dash::Schedule sc;
    int rc = dash::build_schedule(mask, sched, n, &sc);
    if (rc) return (dash_status_t)rc;
    dash::Dealing dl;
    dash::deal(sc, heads, grid, head_dim, &dl);
    DealtTables d;
    d.num_pieces = (int)dl.pieces.size();
    cudaError_t e = upload_new(dl.cta_off, &d.cta_off);
    if (e == cudaSuccess) e = upload_new(piece_words(dl), &d.pieces);
    if (e == cudaSuccess && dash::arrival_ordered(sc))
      e = upload_new(*host_dealt_locked(sc, heads, grid, head_dim), &d.ord);
    if (e != cudaSuccess) {
      cudaFree(d.cta_off);
      cudaFree(d.pieces);
      cudaFree(d.ord);
      return cuda_fail(e, "uploading the dealing tables");
    }
    it = g_dealt.emplace(key, d).first;
  }
  p->ord = it->second.ord ? it->second.ord : tb.ord;
  p->ord_stride = it->second.ord ? (long long)n * n : 0;
  p->cta_off = it->second.cta_off;
  p->pieces = it->second.pieces;
  p->num_pieces = it->second.num_pieces;
  return DASH_OK;
}

// The backward main kernel for a head dimension: D = 64 runs the general kernel with
// 128-row Q tiles; D = 128 runs the kernel that keeps P in TMEM (whole 128 x 128 tasks).
struct MainKernel {
  void* fn;
  size_t smem;
  int br;   // Q/dO rows per TMA box and dQ accumulator box height
};
// `traced`: the main kernel is compiled twice per head dimension, with and without its
// wait-cycle trace; the traced build is launched only while a trace buffer is set.
// `split`: the dealing splits a KV tile over two CTAs (its epilogue is compiled only into
// those instances; the traced build always has it).
// `early` (D = 128): the instances that issue S(t+1) between the two halves of dQ^T(t).
// Measured on full 2x8192x16x128: faster only for shift's order in two interleaved chains
// (991 -> 1011 TFLOP/s); slower with unordered adds (1128 -> 1072), one chain (948 -> 939)
// and the ascending and descending orders (876 -> 855); about even for symmetric shift.
bool early_s(int schedule, int deterministic) {
  return schedule == DASH_SCHED_SHIFT && deterministic == 2;
}
MainKernel main_kernel(int D, bool traced, bool split, bool early) {
  using namespace dash::tc;
  if (D == 64)
    return {traced  ? (void*)bwd_main_kernel<64, true, true, false>
            : split ? (void*)bwd_main_kernel<64, false, true, false>
                    : (void*)bwd_main_kernel<64, false, false, false>,
            (size_t)LTc<64>::ALLOC, dash::kTile};
  void* fn;
  if (early)
    fn = traced  ? (void*)bwd_main_kernel<128, true, true, true>
         : split ? (void*)bwd_main_kernel<128, false, true, true>
                 : (void*)bwd_main_kernel<128, false, false, true>;
  else
    fn = traced  ? (void*)bwd_main_kernel<128, true, true, false>
         : split ? (void*)bwd_main_kernel<128, false, true, false>
                 : (void*)bwd_main_kernel<128, false, false, false>;
  return {fn, (size_t)LTc<128>::ALLOC, dash::kTile};
}

// The main kernel moves registers between warpgroups (setmaxnreg); its split adds up to
// exactly the per-thread count it is launched with, so any other count is refused here
// (a larger request than the pool holds would never be granted).
bool launch_regs_ok(const MainKernel& mk) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, mk.fn) != cudaSuccess) return false;
  return fa.numRegs == dash::tc::L128::REGS_LAUNCH;
}

// True when the schedule's waits are acyclic for `heads` heads on `grid` persistent CTAs
// dealt at head dimension `head_dim`.
bool deadlock_free(int mask, int sched, int n, int heads, int grid, int head_dim) {
  auto key = std::make_tuple(mask, sched, n, heads, grid, head_dim);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_deadlock_free.find(key);
    if (it != g_deadlock_free.end()) return it->second;
  }
  bool ok = true;
  if (sched == dash::SCHED_SHIFT || sched == dash::SCHED_SYMMETRIC_SHIFT) {
    // Ascending/descending wait only on lower KV indices, which are dealt earlier.
    dash::Schedule sc;
    if (dash::build_schedule(mask, sched, n, &sc) != 0) return false;
    double mk = 0;
    ok = dash::simulate(sc, heads, grid, head_dim, 1.0, 0.1, &mk, nullptr);
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_deadlock_free[key] = ok;
  return ok;
}

bool shape_ok(int B, int S, int H, int D) {
  if (B < 1 || S < 1 || H < 1) return false;
  if (D != 64 && D != 128) return false;
  if (S % dash::kTile) return false;
  if (S / dash::kTile > 32767) return false;
  if ((long long)B * S * H * D >= (1ll << 31)) return false;
  return true;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Forgets the static scratch's cached device addresses and table images (defined with
// dash_attn_bwd_static below; the caller holds g_mu).
void reset_static_state_locked();

// Profiling hook state: a pool of event pairs recorded around the main kernel.
constexpr int kProfPairs = 1024;
std::mutex g_prof_mu;
bool g_prof_on = false;
int g_prof_used = 0;
std::vector<cudaEvent_t> g_prof_ev;   // 2 * kProfPairs

cudaEvent_t prof_event(bool stop) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || g_prof_used >= kProfPairs) return nullptr;
  cudaEvent_t e = g_prof_ev[2 * g_prof_used + (stop ? 1 : 0)];
  if (stop) ++g_prof_used;
  return e;
}

// cuTensorMapEncodeTiled from the driver, fetched through the runtime (no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}

// 3D view [B*S][H][D] of a BSHD bf16 tensor; box = 64 columns x 1 head x `rows` rows,
// 128-byte swizzle (the layout the tensor-core descriptors expect).
bool map_bshd(CUtensorMap* m, const void* ptr, int B, int S, int H, int D, int rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)B * S};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
  const cuuint32_t es[3] = {1, 1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D view [rows][K] of a row-major bf16 matrix; box = 64 K-columns x 128 rows, 128-byte
// swizzle.
bool map_rows_k(CUtensorMap* m, const void* ptr, int rows, int K, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct WsLayout {
  size_t dsum, nlse2, qx, dox, dq_acc, sems, split_flags, split_acc, total;
};

static_assert(dash::kSplitTiles == dash::kMaxSplitTiles, "split tiles: one bound");

WsLayout ws_layout(int B, int S, int H, int D) {
  WsLayout w;
  const size_t rows = (size_t)B * H * S;
  w.dsum = dash::kWsHeaderBytes;
  w.nlse2 = round_up(w.dsum + rows * sizeof(float), 256);
  // score-offset blocks of the main kernel: 16 bf16 per row each
  w.qx = round_up(w.nlse2 + rows * sizeof(float), 256);
  w.dox = round_up(w.qx + rows * 32, 256);
  w.dq_acc = round_up(w.dox + rows * 32, 256);
  w.sems = round_up(w.dq_acc + dash::kDqChains * rows * D * sizeof(float), 256);   // k copies
  w.split_flags = round_up(
      w.sems + (size_t)B * H * (S / dash::kTile) * dash::kSemStride * sizeof(int), 256);
  // split KV tiles: only a grid's last partial round, with room for two halves per tile,
  // so fewer than half the units (B * H * S / 128 bounds them for every schedule)
  const size_t splits = std::min<size_t>((size_t)B * H * (S / dash::kTile) / 2, dash::kSplitTiles);
  w.split_acc = round_up(w.split_flags + dash::kSplitTiles * dash::kSplitFlags * sizeof(int), 256);
  w.total = round_up(w.split_acc + splits * 2 * dash::kTile * D * sizeof(float), 256);
  return w;
}

}  // namespace

extern "C" {

const char* dash_status_string(int status) {
  switch (status) {
    case DASH_OK: return "DASH_OK";
    case DASH_ERR_INVALID_ARG: return "DASH_ERR_INVALID_ARG";
    case DASH_ERR_UNSUPPORTED: return "DASH_ERR_UNSUPPORTED";
    case DASH_ERR_WORKSPACE_TOO_SMALL: return "DASH_ERR_WORKSPACE_TOO_SMALL";
    case DASH_ERR_CUDA: return "DASH_ERR_CUDA";
    case DASH_ERR_SYNC_TIMEOUT: return "DASH_ERR_SYNC_TIMEOUT";
    case DASH_ERR_DEADLOCK_RISK: return "DASH_ERR_DEADLOCK_RISK";
    case DASH_ERR_BOUNDS: return "DASH_ERR_BOUNDS";
    default: return "DASH_ERR_UNKNOWN";
  }
}

const char* dash_last_error(void) { return g_last_error.c_str(); }

void dash_debug_set_sync(long long timeout_ns, int ordinal_skew) {
  g_timeout_ns = timeout_ns > 0 ? timeout_ns : 10ll * 1000 * 1000 * 1000;
  g_ordinal_skew = ordinal_skew;
}

void dash_attn_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = -1;
  cudaGetDevice(&cur);
  for (auto& kv : g_tables) {
    cudaSetDevice(std::get<0>(kv.first));
    cudaFree(kv.second.tasks);
    cudaFree(kv.second.ord);
    cudaFree(kv.second.cnt);
  }
  for (auto& kv : g_dealt) {
    cudaSetDevice(std::get<0>(kv.first));
    cudaFree(kv.second.ord);
    cudaFree(kv.second.cta_off);
    cudaFree(kv.second.pieces);
  }
  if (cur >= 0) cudaSetDevice(cur);
  g_tables.clear();
  g_dealt.clear();
  g_host_dealt.clear();
  g_deadlock_free.clear();
  reset_static_state_locked();
}

size_t dash_attn_bwd_workspace_size(int B, int S, int H, int D) {
  if (!shape_ok(B, S, H, D)) return 0;
  return ws_layout(B, S, H, D).total;
}

dash_status_t dash_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int S, int H, int D, float scale, int mask, int* status,
                               cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return DASH_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || D < 1) return DASH_ERR_INVALID_ARG;
  if (mask != DASH_MASK_FULL && mask != DASH_MASK_CAUSAL) return DASH_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return DASH_ERR_INVALID_ARG;
  if (!shape_ok(B, S, H, D)) return DASH_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return DASH_ERR_INVALID_ARG;
  if (status && ((uintptr_t)status & 3u)) return DASH_ERR_INVALID_ARG;
  dash::FwdParams p{(const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
                    (__nv_bfloat16*)o, lse, B, S, H, D, scale, mask == DASH_MASK_CAUSAL,
                    scale * dash::kLog2e, status, g_timeout_ns, g_ordinal_skew > 0 ? 1 : 0};
  if (!encoder()) {
    g_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return DASH_ERR_CUDA;
  }
  dash::tc::TmaMaps maps;
  if (!map_bshd(&maps.q, q, B, S, H, D, dash::kTile) ||
      !map_bshd(&maps.k, k, B, S, H, D, dash::kTile) ||
      !map_bshd(&maps.v, v, B, S, H, D, dash::kTile)) {
    g_last_error = "cuTensorMapEncodeTiled rejected a tensor";
    return DASH_ERR_CUDA;
  }
  // one CTA per pair of adjacent 128-row Q tiles of one batch * head; blockIdx.x is the
  // batch * head and blockIdx.y counts the pairs from the last tiles, so blocks are handed
  // out pair rank by pair rank over all heads: under a causal mask, longest first
  dim3 grid(B * H, (S / dash::kTile + 1) / 2);
  void* kfn = D == 64 ? (void*)dash::tc::fwd_tc_kernel<64> : (void*)dash::tc::fwd_tc_kernel<128>;
  const size_t smem = D == 64 ? dash::tc::FwdL<64>::ALLOC : dash::tc::FwdL<128>::ALLOC;
  // the kernel moves registers between its warpgroups (setmaxnreg); the split adds up to
  // exactly the per-thread count it is launched with, so any other count is refused
  cudaFuncAttributes fa;
  DASH_CUDA(cudaFuncGetAttributes(&fa, kfn));
  if (fa.numRegs != dash::tc::kFwdRegsLaunch) {
    g_last_error = "forward kernel was not built with the register count its warp roles share";
    return DASH_ERR_CUDA;
  }
  DASH_CUDA(cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  if (status) DASH_CUDA(cudaMemsetAsync(status, 0, sizeof(int), stream));
  void* args[] = {&p, &maps};
  DASH_CUDA(cudaLaunchKernel(kfn, grid, dim3(dash::tc::kFwdThreads), args, smem, stream));
  return DASH_OK;
}

dash_status_t dash_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int S, int H, int D, float scale, int mask,
                            cudaStream_t stream) {
  return dash_attn_fwd_ex(q, k, v, o, lse, B, S, H, D, scale, mask, nullptr, stream);
}

dash_status_t dash_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            void* workspace, size_t workspace_bytes,
                            int B, int S, int H, int D, float scale, int mask, int schedule,
                            int deterministic, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !workspace)
    return DASH_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || D < 1) return DASH_ERR_INVALID_ARG;
  if (mask != DASH_MASK_FULL && mask != DASH_MASK_CAUSAL) return DASH_ERR_INVALID_ARG;
  if (schedule < DASH_SCHED_ASCENDING || schedule > DASH_SCHED_SYMMETRIC_SHIFT)
    return DASH_ERR_INVALID_ARG;
  if (deterministic < 0 || deterministic > dash::kDqChains) return DASH_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return DASH_ERR_INVALID_ARG;
  if (!shape_ok(B, S, H, D)) return DASH_ERR_UNSUPPORTED;
  for (const void* ptr : {q, k, v, o, dO, (const void*)lse, (const void*)dq, (const void*)dk,
                          (const void*)dv})
    if (!aligned16(ptr)) return DASH_ERR_INVALID_ARG;
  if (((uintptr_t)workspace & 255u) != 0) return DASH_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(B, S, H, D);
  if (workspace_bytes < wl.total) return DASH_ERR_WORKSPACE_TOO_SMALL;
  const int n = S / dash::kTile;
  {
    dash::Schedule probe;
    int rc = dash::build_schedule(mask, schedule, n, &probe);
    if (rc) return (dash_status_t)rc;
  }
  int dev = 0;
  DASH_CUDA(cudaGetDevice(&dev));
  DeviceTables tb;
  dash_status_t st = get_tables(dev, mask, schedule, n, &tb);
  if (st != DASH_OK) return st;

  char* ws = (char*)workspace;
  dash::BwdParams p;
  p.q = (const __nv_bfloat16*)q;
  p.k = (const __nv_bfloat16*)k;
  p.v = (const __nv_bfloat16*)v;
  p.o = (const __nv_bfloat16*)o;
  p.dO = (const __nv_bfloat16*)dO;
  p.lse = lse;
  p.dq = (__nv_bfloat16*)dq;
  p.dk = (__nv_bfloat16*)dk;
  p.dv = (__nv_bfloat16*)dv;
  p.ws_header = (int*)ws;
  p.Dsum = (float*)(ws + wl.dsum);
  p.nlse2 = (float*)(ws + wl.nlse2);
  p.qx = (__nv_bfloat16*)(ws + wl.qx);
  p.dox = (__nv_bfloat16*)(ws + wl.dox);
  p.dq_acc = (float*)(ws + wl.dq_acc);
  p.sems = (int*)(ws + wl.sems);
  p.split_flags = (int*)(ws + wl.split_flags);
  p.split_acc = (float*)(ws + wl.split_acc);
  p.tasks = tb.tasks;
  p.ord = tb.ord;
  p.cnt = tb.cnt;
  p.B = B;
  p.S = S;
  p.H = H;
  p.D = D;
  p.n = n;
  const int units = B * H * tb.num_slots;
  p.scale = scale;
  p.scale_log2 = scale * dash::kLog2e;
  p.causal = mask == DASH_MASK_CAUSAL;
  p.deterministic = deterministic != 0;
  p.chains = deterministic > 1 ? deterministic : 1;
  p.timeout_ns = g_timeout_ns;
  p.ordinal_skew = g_ordinal_skew;
  p.trace = g_trace;
  p.num_tasks = tb.num_tasks;
  p.check_n = n - g_check_narrow;

  p.num_sems = B * H * n * dash::kSemStride;

  // Persistent grid, one CTA per SM: every CTA must be resident at once (the ordered
  // reduction waits on other CTAs), so the launch is cooperative.
  if (!encoder()) {
    g_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return DASH_ERR_CUDA;
  }
  dash::tc::TmaMaps maps;
  int sms = 0;
  DASH_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  int grid = sms;                      // one CTA per SM (512 TMEM columns each)
  if (grid > units) grid = units;
  const MainKernel mk =
      main_kernel(D, g_trace != nullptr, dash::split_tiles(schedule, n, units, grid) > 0,
                  early_s(schedule, deterministic));
  const int br = mk.br;
  if (!map_bshd(&maps.q, q, B, S, H, D, br) || !map_bshd(&maps.dO, dO, B, S, H, D, br) ||
      !map_bshd(&maps.k, k, B, S, H, D, dash::kTile) ||
      !map_bshd(&maps.v, v, B, S, H, D, dash::kTile)) {
    g_last_error = "cuTensorMapEncodeTiled rejected a tensor";
    return DASH_ERR_CUDA;
  }
  const int threads = dash::tc::kThreads;
  const size_t smem = mk.smem;
  void* kfn = mk.fn;
  if (!launch_regs_ok(mk)) {
    g_last_error = "backward kernel was not built with the register count its warp roles share";
    return DASH_ERR_CUDA;
  }
  DASH_CUDA(cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per_sm = 0;
  DASH_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, threads, smem));
  if (per_sm < 1) {
    g_last_error = "backward kernel does not fit on one SM";
    return DASH_ERR_CUDA;
  }
  if (deterministic && !deadlock_free(mask, schedule, n, B * H, grid, D))
    return DASH_ERR_DEADLOCK_RISK;
  st = set_dealing(dev, mask, schedule, n, B * H, grid, D, tb, &p);
  if (st != DASH_OK) return st;

  dash::bwd_preprocess_kernel<<<sms * 4, 256, 0, stream>>>(p);
  DASH_CUDA(cudaGetLastError());
  void* args[] = {&p, &maps};
  cudaEvent_t ev0 = prof_event(false);
  if (ev0) DASH_CUDA(cudaEventRecord(ev0, stream));
  if (deterministic) {
    DASH_CUDA(cudaLaunchCooperativeKernel(kfn, dim3(grid), dim3(threads), args, smem, stream));
  } else {
    DASH_CUDA(cudaLaunchKernel(kfn, dim3(grid), dim3(threads), args, smem, stream));
  }
  if (ev0) DASH_CUDA(cudaEventRecord(prof_event(true), stream));
  dash::dq_convert_kernel<<<sms * 4, 256, 0, stream>>>(p);
  DASH_CUDA(cudaGetLastError());
  return DASH_OK;
}

dash_status_t dash_attn_get_status(const void* workspace, cudaStream_t stream) {
  if (!workspace) return DASH_ERR_INVALID_ARG;
  DASH_CUDA(cudaStreamSynchronize(stream));
  int words[8];
  DASH_CUDA(cudaMemcpy(words, workspace, sizeof(words), cudaMemcpyDeviceToHost));
  if (words[dash::WS_STATUS] == dash::kStatusSmemLayout) {
    g_last_error = "the backward kernel found its shared-memory base off a 1024-byte boundary";
    return DASH_ERR_CUDA;
  }
  if (words[dash::WS_STATUS] == dash::kStatusSyncTimeout && words[dash::WS_BH] < 0) {
    char buf[160];
    snprintf(buf, sizeof(buf), "a pipeline wait inside CTA %d timed out", words[dash::WS_QTILE]);
    g_last_error = buf;
    return DASH_ERR_SYNC_TIMEOUT;
  }
  if (words[dash::WS_STATUS] == dash::kStatusBounds) {
    static const char* const sites[] = {"?", "a CTA's piece range", "a piece", "a task",
                                         "a dQ ordinal"};
    const int site = words[dash::WS_QTILE];
    char buf[200];
    snprintf(buf, sizeof(buf), "bounds check failed on %s: bh/cta=%d value=%d bound=%d",
             sites[site >= 1 && site <= 4 ? site : 0], words[dash::WS_BH],
             words[dash::WS_EXPECT], words[dash::WS_SEEN]);
    g_last_error = buf;
    return DASH_ERR_BOUNDS;
  }
  if (words[dash::WS_STATUS] == dash::kStatusSyncTimeout) {
    char buf[160];
    snprintf(buf, sizeof(buf), "dQ reduction wait timed out: bh=%d q_tile=%d expected=%d seen=%d",
             words[dash::WS_BH], words[dash::WS_QTILE], words[dash::WS_EXPECT],
             words[dash::WS_SEEN]);
    g_last_error = buf;
    return DASH_ERR_SYNC_TIMEOUT;
  }
  return DASH_OK;
}

int dash_bounds_checks_enabled(void) { return DASH_BOUNDS_CHECKS; }

dash_status_t dash_debug_narrow_checks(int tiles) {
  if (!DASH_BOUNDS_CHECKS) {
    g_last_error = "this build has no bounds checks (build with checks=True)";
    return DASH_ERR_UNSUPPORTED;
  }
  if (tiles < 0) return DASH_ERR_INVALID_ARG;
  g_check_narrow = tiles;
  return DASH_OK;
}

void dash_debug_set_trace(void* device_counters) {
  g_trace = (unsigned long long*)device_counters;
}

dash_status_t dash_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on && g_prof_ev.empty()) {
    g_prof_ev.resize(2 * kProfPairs);
    for (auto& e : g_prof_ev) DASH_CUDA(cudaEventCreate(&e));
  }
  g_prof_on = on != 0;
  return DASH_OK;
}

dash_status_t dash_profile_read(double* total_ms, int* launches) {
  if (!total_ms || !launches) return DASH_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double sum = 0.0;
  for (int k = 0; k < g_prof_used; ++k) {
    DASH_CUDA(cudaEventSynchronize(g_prof_ev[2 * k + 1]));
    float ms = 0.f;
    DASH_CUDA(cudaEventElapsedTime(&ms, g_prof_ev[2 * k], g_prof_ev[2 * k + 1]));
    sum += ms;
  }
  *total_ms = sum;
  *launches = g_prof_used;
  g_prof_used = 0;
  return DASH_OK;
}

int dash_sched_num_slots(int mask, int schedule, int n) {
  dash::Schedule sc;
  int rc = dash::build_schedule(mask, schedule, n, &sc);
  return rc ? -rc : sc.num_slots;
}

int dash_sched_table(int mask, int schedule, int n, int32_t* slot_offsets, int32_t* tasks,
                     int cap, int32_t* ordinals) {
  dash::Schedule sc;
  int rc = dash::build_schedule(mask, schedule, n, &sc);
  if (rc) return -rc;
  if (!slot_offsets || !tasks || !ordinals || cap < (int)sc.tasks.size())
    return -DASH_ERR_INVALID_ARG;
  std::memcpy(slot_offsets, sc.slot_off.data(), sc.slot_off.size() * sizeof(int32_t));
  std::memcpy(tasks, sc.tasks.data(), sc.tasks.size() * sizeof(int32_t));
  std::memcpy(ordinals, sc.ord.data(), sc.ord.size() * sizeof(int32_t));
  return (int)sc.tasks.size();
}

dash_status_t dash_sched_dealt_table(int mask, int schedule, int n, int heads, int grid,
                                    int head_dim, int32_t* ordinals) {
  if (heads < 1 || grid < 1 || !ordinals || (head_dim != 64 && head_dim != 128))
    return DASH_ERR_INVALID_ARG;
  dash::Schedule sc;
  int rc = dash::build_schedule(mask, schedule, n, &sc);
  if (rc) return (dash_status_t)rc;
  std::vector<int32_t> ord;
  dash::dealt_orders(sc, heads, grid, head_dim, &ord);
  std::memcpy(ordinals, ord.data(), ord.size() * sizeof(int32_t));
  return DASH_OK;
}

int dash_sched_deal(int mask, int schedule, int n, int heads, int grid, int head_dim,
                    int32_t* cta_offsets, int32_t* pieces, int cap) {
  if (heads < 1 || grid < 1 || !cta_offsets || !pieces || cap < 0 ||
      (head_dim != 64 && head_dim != 128))
    return -DASH_ERR_INVALID_ARG;
  dash::Schedule sc;
  int rc = dash::build_schedule(mask, schedule, n, &sc);
  if (rc) return -rc;
  dash::Dealing dl;
  dash::deal(sc, heads, grid, head_dim, &dl);
  if ((size_t)cap < dl.pieces.size()) return -DASH_ERR_INVALID_ARG;
  std::memcpy(cta_offsets, dl.cta_off.data(), dl.cta_off.size() * sizeof(int32_t));
  for (size_t k = 0; k < dl.pieces.size(); ++k) {
    const dash::Piece& pc = dl.pieces[k];
    const int32_t w[5] = {pc.head, pc.t_begin, pc.t_end, pc.part, pc.split};
    std::memcpy(pieces + 5 * k, w, sizeof(w));
  }
  return (int)dl.pieces.size();
}

dash_status_t dash_sched_simulate(int mask, int schedule, int n, int heads, int num_sms,
                                  int head_dim, double c, double r, double* makespan,
                                  double* sm_end) {
  if (heads < 1 || num_sms < 1 || !makespan || !(c >= 0) || !(r >= 0) ||
      (head_dim != 64 && head_dim != 128))
    return DASH_ERR_INVALID_ARG;
  dash::Schedule sc;
  int rc = dash::build_schedule(mask, schedule, n, &sc);
  if (rc) return (dash_status_t)rc;
  std::vector<double> ends;
  if (!dash::simulate(sc, heads, num_sms, head_dim, c, r, makespan, &ends))
    return DASH_ERR_DEADLOCK_RISK;
  if (sm_end) std::memcpy(sm_end, ends.data(), ends.size() * sizeof(double));
  return DASH_OK;
}

size_t dash_gemm_splitk_workspace_size(int M, int N) {
  if (M < 128 || N < 128 || M % 128 || N % 128) return 0;
  return round_up(dash::kWsHeaderBytes + (size_t)(M / 128) * (N / 128) * sizeof(int), 256);
}

dash_status_t dash_gemm_splitk(const void* a, const void* b, float* c, void* workspace,
                               size_t workspace_bytes, int M, int N, int K, int splits,
                               int deterministic, cudaStream_t stream) {
  if (!a || !b || !c || !workspace) return DASH_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || splits < 1) return DASH_ERR_INVALID_ARG;
  if (deterministic != 0 && deterministic != 1) return DASH_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || ((uintptr_t)workspace & 255))
    return DASH_ERR_INVALID_ARG;
  if (M % 128 || N % 128 || K % (64 * splits) || (long long)M * N >= (1ll << 31))
    return DASH_ERR_UNSUPPORTED;
  if (workspace_bytes < dash_gemm_splitk_workspace_size(M, N)) return DASH_ERR_WORKSPACE_TOO_SMALL;
  if (!encoder()) {
    g_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return DASH_ERR_CUDA;
  }
  // output tiles of 256 rows of C when M allows (the MMA is then 256 wide and runs at the
  // tensor core's full rate), else 128
  const int tm = (M % 256 == 0) ? 256 : 128;
  dash::tc::GemmMaps maps;
  if (!map_rows_k(&maps.a, a, M, K, tm) || !map_rows_k(&maps.b, b, N, K, 128)) {
    g_last_error = "cuTensorMapEncodeTiled rejected a tensor";
    return DASH_ERR_CUDA;
  }
  unsigned char* ws = (unsigned char*)workspace;
  dash::tc::GemmParams p;
  p.c = c;
  p.status = (int*)ws;
  p.sems = (int*)(ws + dash::kWsHeaderBytes);
  p.M = M;
  p.N = N;
  p.K = K;
  p.splits = splits;
  p.kchunk = K / splits;
  p.deterministic = deterministic;
  p.timeout_ns = g_timeout_ns;
  // C, the status header and the tile semaphores start at zero
  DASH_CUDA(cudaMemsetAsync(c, 0, (size_t)M * N * sizeof(float), stream));
  DASH_CUDA(cudaMemsetAsync(ws, 0, dash_gemm_splitk_workspace_size(M, N), stream));
  int dev = 0, sms = 0;
  DASH_CUDA(cudaGetDevice(&dev));
  DASH_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int units = (M / tm) * (N / 128) * splits;
  const int grid = units < sms ? units : sms;
  void* kfn = tm == 256 ? (void*)dash::tc::gemm_splitk_kernel<256> : (void*)dash::tc::gemm_splitk_kernel<128>;
  const size_t smem = tm == 256 ? dash::tc::GemmL<256>::ALLOC : dash::tc::GemmL<128>::ALLOC;
  DASH_CUDA(cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  void* args[] = {&p, &maps};
  // deterministic: chunks wait on other CTAs' adds, so every CTA must be resident at once;
  // the waits follow the dealing order, so they cannot form a cycle on any grid
  if (deterministic)
    DASH_CUDA(cudaLaunchCooperativeKernel(kfn, dim3(grid), dim3(dash::tc::kGemmThreads), args,
                                          smem, stream));
  else
    DASH_CUDA(cudaLaunchKernel(kfn, dim3(grid), dim3(dash::tc::kGemmThreads), args, smem, stream));
  return DASH_OK;
}

dash_status_t dash_sched_simulate_ex(int mask, int schedule, int n, int heads, int num_sms,
                                     int head_dim, double c, double r, double h, int overlapped,
                                     double* makespan, double* sm_end) {
  if (heads < 1 || num_sms < 1 || !makespan || !(c >= 0) || !(r >= 0) || !(h >= 0) ||
      (overlapped != 0 && overlapped != 1) || (head_dim != 64 && head_dim != 128))
    return DASH_ERR_INVALID_ARG;
  dash::Schedule sc;
  int rc = dash::build_schedule(mask, schedule, n, &sc);
  if (rc) return (dash_status_t)rc;
  std::vector<double> ends;
  if (!dash::simulate_ex(sc, heads, num_sms, head_dim, c, r, h, overlapped != 0, makespan,
                         &ends))
    return DASH_ERR_DEADLOCK_RISK;
  if (sm_end) std::memcpy(sm_end, ends.data(), ends.size() * sizeof(double));
  return DASH_OK;
}

dash_status_t dash_sched_select(int mask, int n, int heads, int num_sms, int head_dim, double c,
                                double r, double h, int overlapped, int* schedule_out,
                                double* makespan_out) {
  if (!schedule_out || heads < 1 || num_sms < 1 || !(c >= 0) || !(r >= 0) || !(h >= 0) ||
      (overlapped != 0 && overlapped != 1) || (head_dim != 64 && head_dim != 128))
    return DASH_ERR_INVALID_ARG;
  if (mask != DASH_MASK_FULL && mask != DASH_MASK_CAUSAL) return DASH_ERR_INVALID_ARG;
  int best = -1;
  double best_mk = 0.0;
  for (int s = DASH_SCHED_ASCENDING; s <= DASH_SCHED_SYMMETRIC_SHIFT; ++s) {
    dash::Schedule sc;
    const int rc = dash::build_schedule(mask, s, n, &sc);
    if (rc == DASH_ERR_UNSUPPORTED) continue;          // schedule not defined for this mask/n
    if (rc) return (dash_status_t)rc;
    double mk = 0.0;
    if (!dash::simulate_ex(sc, heads, num_sms, head_dim, c, r, h, overlapped != 0, &mk,
                           nullptr))
      continue;                                        // its waits would deadlock this grid
    if (best < 0 || mk < best_mk) {                    // ties keep the lower enum value
      best = s;
      best_mk = mk;
    }
  }
  if (best < 0) return DASH_ERR_DEADLOCK_RISK;
  *schedule_out = best;
  if (makespan_out) *makespan_out = best_mk;
  return DASH_OK;
}

}  // extern "C"

// =====================================================================================
// Backward without device allocation (dash_attn_bwd_static).
//
// For callers that cannot allocate device memory at the time they run the backward --
// for example a runtime whose memory is fully reserved up front by its own pool, or code
// that must not enter the CUDA allocator at all -- this entry point takes its scratch
// from a fixed array that is part of the library's device image. Inputs and outputs are
// still the caller's buffers. The array is reserved on every GPU that loads the library
// and stays there until the process exits.
// =====================================================================================
namespace {

constexpr size_t kStaticScratchBytes = 64ull << 20;   // 64 MiB per device
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
unsigned char* g_static_ptr[kMaxDevices] = {};

// Device address of the scratch array on `dev` (the current device). Looked up once per
// device with that device current; later calls reuse it until dash_attn_shutdown, which
// forgets it (a device reset reloads the module, so the address must be looked up again).
dash_status_t static_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    g_last_error = "dash_attn_bwd_static: device index out of range";
    return DASH_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_ptr[dev] = (unsigned char*)ptr;
  }
  *out = g_static_ptr[dev];
  return DASH_OK;
}

__global__ void copy_status_kernel(const int* header, int* out) { *out = header[dash::WS_STATUS]; }

// Host image of the schedule tables that follow the workspace in the static scratch, in
// the scratch's own layout (offsets relative to the workspace's end), so that one copy
// moves all of them. Entries live until dash_attn_shutdown: a queued copy never reads
// host memory that has been freed.
struct StaticTables {
  std::vector<int32_t> image;
  // byte offsets of the piece, task, order and count tables (the CTA offsets come first)
  size_t piece_off, task_off, ord_off, cnt_off;
  int num_pieces, num_tasks;
};
std::map<std::tuple<int, int, int, int, int, int>, std::shared_ptr<const StaticTables>>
    g_static_tables;

dash_status_t static_tables(int mask, int schedule, int n, int heads, int grid, int head_dim,
                            std::shared_ptr<const StaticTables>* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(mask, schedule, n, heads, grid, head_dim);
  auto it = g_static_tables.find(key);
  if (it == g_static_tables.end()) {
    dash::Schedule sc;
    const int rc = dash::build_schedule(mask, schedule, n, &sc);
    if (rc) return (dash_status_t)rc;
    std::shared_ptr<const std::vector<int32_t>> dealt;
    if (dash::arrival_ordered(sc)) dealt = host_dealt_locked(sc, heads, grid, head_dim);
    const std::vector<int32_t>& ord = dealt ? *dealt : sc.ord;
    dash::Dealing dl;
    dash::deal(sc, heads, grid, head_dim, &dl);
    const std::vector<int32_t> words = piece_words(dl);
    auto t = std::make_shared<StaticTables>();
    t->num_pieces = (int)dl.pieces.size();
    t->num_tasks = (int)sc.tasks.size();
    t->piece_off = round_up(dl.cta_off.size() * 4, 256);
    t->task_off = round_up(t->piece_off + words.size() * 4, 256);
    t->ord_off = round_up(t->task_off + sc.tasks.size() * 4, 256);
    t->cnt_off = round_up(t->ord_off + ord.size() * 4, 256);
    t->image.assign(round_up(t->cnt_off + sc.cnt.size() * 4, 256) / 4, 0);
    std::memcpy(t->image.data(), dl.cta_off.data(), dl.cta_off.size() * 4);
    std::memcpy(t->image.data() + t->piece_off / 4, words.data(), words.size() * 4);
    std::memcpy(t->image.data() + t->task_off / 4, sc.tasks.data(), sc.tasks.size() * 4);
    std::memcpy(t->image.data() + t->ord_off / 4, ord.data(), ord.size() * 4);
    std::memcpy(t->image.data() + t->cnt_off / 4, sc.cnt.data(), sc.cnt.size() * 4);
    it = g_static_tables.emplace(key, std::move(t)).first;
  }
  *out = it->second;
  return DASH_OK;
}

void reset_static_state_locked() {
  g_static_tables.clear();
  std::lock_guard<std::mutex> lk(g_static_mu);
  for (auto& ptr : g_static_ptr) ptr = nullptr;
}

}  // namespace

extern "C" dash_status_t dash_attn_bwd_static(const void* q, const void* k, const void* v,
                                              const void* o, const void* dO, const float* lse,
                                              void* dq, void* dk, void* dv, int* status_out,
                                              int B, int S, int H, int D, float scale, int mask,
                                              int schedule, int deterministic,
                                              cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return DASH_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || D < 1) return DASH_ERR_INVALID_ARG;
  if (mask != DASH_MASK_FULL && mask != DASH_MASK_CAUSAL) return DASH_ERR_INVALID_ARG;
  if (schedule < DASH_SCHED_ASCENDING || schedule > DASH_SCHED_SYMMETRIC_SHIFT)
    return DASH_ERR_INVALID_ARG;
  if (deterministic < 0 || deterministic > dash::kDqChains) return DASH_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return DASH_ERR_INVALID_ARG;
  if (!shape_ok(B, S, H, D)) return DASH_ERR_UNSUPPORTED;
  for (const void* ptr : {q, k, v, o, dO, (const void*)lse, (const void*)dq, (const void*)dk,
                          (const void*)dv})
    if (!aligned16(ptr)) return DASH_ERR_INVALID_ARG;
  const int n = S / dash::kTile;
  {
    dash::Schedule probe;
    const int rc = dash::build_schedule(mask, schedule, n, &probe);
    if (rc) return (dash_status_t)rc;
  }
  int dev = 0, sms = 0;
  DASH_CUDA(cudaGetDevice(&dev));
  DASH_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int slots = dash_sched_num_slots(mask, schedule, n);
  const int units = B * H * slots;
  const int grid = sms < units ? sms : units;
  // the dQ orders of this grid (per head for shift and symmetric shift), as the regular
  // entry point uses them, with the other tables: built once per shape in host memory
  std::shared_ptr<const StaticTables> tb;
  dash_status_t st = static_tables(mask, schedule, n, B * H, grid, D, &tb);
  if (st != DASH_OK) return st;

  // scratch layout: the backward workspace, then the schedule tables
  const WsLayout wl = ws_layout(B, S, H, D);
  const size_t t_off = wl.total;
  const size_t need = t_off + tb->image.size() * 4;
  if (need > kStaticScratchBytes) {
    char buf[200];
    snprintf(buf, sizeof(buf),
             "dash_attn_bwd_static: this shape needs %zu bytes of scratch, more than the "
             "%zu-byte static scratch; use dash_attn_bwd with a caller-allocated workspace",
             need, kStaticScratchBytes);
    g_last_error = buf;
    return DASH_ERR_WORKSPACE_TOO_SMALL;
  }
  unsigned char* ws = nullptr;
  st = static_scratch(dev, &ws);
  if (st != DASH_OK) return st;

  dash::BwdParams p;
  p.q = (const __nv_bfloat16*)q;
  p.k = (const __nv_bfloat16*)k;
  p.v = (const __nv_bfloat16*)v;
  p.o = (const __nv_bfloat16*)o;
  p.dO = (const __nv_bfloat16*)dO;
  p.lse = lse;
  p.dq = (__nv_bfloat16*)dq;
  p.dk = (__nv_bfloat16*)dk;
  p.dv = (__nv_bfloat16*)dv;
  p.ws_header = (int*)ws;
  p.Dsum = (float*)(ws + wl.dsum);
  p.nlse2 = (float*)(ws + wl.nlse2);
  p.qx = (__nv_bfloat16*)(ws + wl.qx);
  p.dox = (__nv_bfloat16*)(ws + wl.dox);
  p.dq_acc = (float*)(ws + wl.dq_acc);
  p.sems = (int*)(ws + wl.sems);
  p.split_flags = (int*)(ws + wl.split_flags);
  p.split_acc = (float*)(ws + wl.split_acc);
  p.cta_off = (const int32_t*)(ws + t_off);
  p.pieces = (const int32_t*)(ws + t_off + tb->piece_off);
  p.tasks = (const int32_t*)(ws + t_off + tb->task_off);
  p.ord = (const int32_t*)(ws + t_off + tb->ord_off);
  p.ord_stride = (schedule == DASH_SCHED_SHIFT || schedule == DASH_SCHED_SYMMETRIC_SHIFT)
                     ? (long long)n * n : 0;
  p.cnt = (const int32_t*)(ws + t_off + tb->cnt_off);
  p.B = B;
  p.S = S;
  p.H = H;
  p.D = D;
  p.n = n;
  p.scale = scale;
  p.scale_log2 = scale * dash::kLog2e;
  p.causal = mask == DASH_MASK_CAUSAL;
  p.deterministic = deterministic != 0;
  p.chains = deterministic > 1 ? deterministic : 1;
  p.timeout_ns = g_timeout_ns;
  p.ordinal_skew = g_ordinal_skew;
  p.trace = nullptr;
  p.num_pieces = tb->num_pieces;
  p.num_tasks = tb->num_tasks;
  p.check_n = n - g_check_narrow;
  p.num_sems = B * H * n * dash::kSemStride;

  // Every refusal comes before the first queued operation: a refused call leaves the
  // stream and the scratch untouched.
  if (!encoder()) {
    g_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return DASH_ERR_CUDA;
  }
  dash::tc::TmaMaps maps;
  const MainKernel mk =
      main_kernel(D, false, dash::split_tiles(schedule, n, units, grid) > 0,
                  early_s(schedule, deterministic));
  const int br = mk.br;
  if (!map_bshd(&maps.q, q, B, S, H, D, br) || !map_bshd(&maps.dO, dO, B, S, H, D, br) ||
      !map_bshd(&maps.k, k, B, S, H, D, dash::kTile) ||
      !map_bshd(&maps.v, v, B, S, H, D, dash::kTile)) {
    g_last_error = "cuTensorMapEncodeTiled rejected a tensor";
    return DASH_ERR_CUDA;
  }
  const int threads = dash::tc::kThreads;
  const size_t smem = mk.smem;
  void* kfn = mk.fn;
  if (!launch_regs_ok(mk)) {
    g_last_error = "backward kernel was not built with the register count its warp roles share";
    return DASH_ERR_CUDA;
  }
  DASH_CUDA(cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per_sm = 0;
  DASH_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, threads, smem));
  if (per_sm < 1) {
    g_last_error = "backward kernel does not fit on one SM";
    return DASH_ERR_CUDA;
  }
  if (deterministic && !deadlock_free(mask, schedule, n, B * H, grid, D))
    return DASH_ERR_DEADLOCK_RISK;

  // Tables are written for every call: the array keeps whatever the last call left.
  DASH_CUDA(cudaMemcpyAsync(ws + t_off, tb->image.data(), tb->image.size() * 4,
                            cudaMemcpyHostToDevice, stream));
  dash::bwd_preprocess_kernel<<<sms * 4, 256, 0, stream>>>(p);
  DASH_CUDA(cudaGetLastError());
  void* args[] = {&p, &maps};
  if (deterministic) {
    DASH_CUDA(cudaLaunchCooperativeKernel(kfn, dim3(grid), dim3(threads), args, smem, stream));
  } else {
    DASH_CUDA(cudaLaunchKernel(kfn, dim3(grid), dim3(threads), args, smem, stream));
  }
  dash::dq_convert_kernel<<<sms * 4, 256, 0, stream>>>(p);
  DASH_CUDA(cudaGetLastError());
  if (status_out) {
    copy_status_kernel<<<1, 1, 0, stream>>>(p.ws_header, status_out);
    DASH_CUDA(cudaGetLastError());
  }
  return DASH_OK;
}
