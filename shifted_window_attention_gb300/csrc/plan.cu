// Window plans: host geometry and the device kernel that writes the token-id
// tables.
//
// Geometry follows "Window-Aligned Sequence Parallelism (SeedVR2)", section
// "Window layouts": window size normalised to the 45 x 80 (720p) reference
// area, regular cuts at multiples of the window size, shifted cuts moved by
// half a window and clipped at both grid ends (no cyclic roll), windows
// enumerated w-outermost / t-innermost, tokens row-major in (t, h, w) inside a
// window, canonical id (t*H + h)*W + w.  Offsets follow the cu_seqlens
// convention (prefix sums from 0).

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <tuple>
#include <utility>

#include "wsa_internal.h"

namespace wsa {

namespace {
thread_local std::string g_last_error;
}

wsa_status fail(wsa_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

wsa_status cuda_fail(cudaError_t e, const char* what) {
  std::string msg = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return fail(e == cudaErrorMemoryAllocation ? WSA_ERR_OOM : WSA_ERR_CUDA, msg);
}

void clear_error() { g_last_error.clear(); }

int sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace

// Host geometry, shared with the other translation units through
// wsa_internal.h.

// Window size in fp64 exactly as the note's formula reads; nearbyint rounds
// half-to-even in the default rounding mode (Python's round).
wsa_status window_size(int T, int H, int W, int nt, int nh, int nw, int max_temporal,
                       int* wt, int* wh, int* ww) {
  if (T <= 0 || H <= 0 || W <= 0 || nt <= 0 || nh <= 0 || nw <= 0 || max_temporal <= 0)
    return fail(WSA_ERR_INVALID_ARG, "grid sizes, window counts and max_temporal must be > 0");
  const double area = static_cast<double>(static_cast<long long>(H) * W);
  const double scale = std::sqrt(3600.0 / area);
  const double rh = std::nearbyint(static_cast<double>(H) * scale);
  const double rw = std::nearbyint(static_cast<double>(W) * scale);
  const long long h = ceil_div(static_cast<long long>(rh), nh);
  const long long w = ceil_div(static_cast<long long>(rw), nw);
  const long long t = ceil_div(std::min(T, max_temporal), nt);
  if (h <= 0 || w <= 0 || t <= 0)
    return fail(WSA_ERR_INVALID_ARG, "window size computes to zero for this grid");
  *wt = static_cast<int>(t);
  *wh = static_cast<int>(h);
  *ww = static_cast<int>(w);
  return WSA_OK;
}

// Half-open intervals cutting one axis.  Shifted: cuts at floor(w/2) + m*w,
// only when the axis is longer than its window; empty intervals dropped.
std::vector<std::pair<int, int>> axis_intervals(int size, int w, bool shifted) {
  std::vector<int> cuts;
  cuts.push_back(0);
  if (shifted && size > w) {
    for (long long c = w / 2; c < size; c += w) cuts.push_back(static_cast<int>(c));
  } else {
    for (long long c = w; c < size; c += w) cuts.push_back(static_cast<int>(c));
  }
  cuts.push_back(size);
  std::vector<std::pair<int, int>> out;
  for (size_t i = 0; i + 1 < cuts.size(); ++i)
    if (cuts[i + 1] > cuts[i]) out.emplace_back(cuts[i], cuts[i + 1]);
  return out;
}

void layout_boxes(int T, int H, int W, int wt, int wh, int ww, bool shifted,
                  std::vector<int>* dims) {
  const auto ti = axis_intervals(T, wt, shifted);
  const auto hi = axis_intervals(H, wh, shifted);
  const auto wi = axis_intervals(W, ww, shifted);
  dims->clear();
  dims->reserve(ti.size() * hi.size() * wi.size() * 6);
  for (const auto& a : wi)
    for (const auto& b : hi)
      for (const auto& c : ti) {
        const int box[6] = {c.first, c.second, b.first, b.second, a.first, a.second};
        dims->insert(dims->end(), box, box + 6);
      }
}

// Work items of `rows` query rows per item, in LPT order: heaviest first
// (query tiles x key tiles), ties by (window, q_start) -- the ordering rule of
// the note's "Planner" section applied to kernel work units.  A window's
// full items are therefore consecutive and its partial last item comes late,
// with the other light items.  (Keeping every item with its window, partial
// one included, cuts the tensor-core kernel's DRAM traffic from 1.43x to
// 0.97x of its algorithmic bytes, but measured 1-4% slower with canonical
// rows: DRAM is far from busy, and the coarser tail of the list costs more
// than the re-reads it saves.)
std::vector<WorkItem> make_items(const std::vector<int>& offsets, int rows, int tile) {
  struct Keyed {
    long long cost;
    WorkItem it;
  };
  std::vector<Keyed> v;
  const int nwin = static_cast<int>(offsets.size()) - 1;
  for (int w = 0; w < nwin; ++w) {
    const int n = offsets[w + 1] - offsets[w];
    const long long kv_tiles = ceil_div(n, tile);
    for (int q0 = 0; q0 < n; q0 += rows) {
      const long long q_tiles = ceil_div(std::min(rows, n - q0), tile);
      v.push_back({q_tiles * kv_tiles, {w, q0}});
    }
  }
  std::stable_sort(v.begin(), v.end(), [](const Keyed& a, const Keyed& b) {
    if (a.cost != b.cost) return a.cost > b.cost;
    return std::make_pair(a.it.window, a.it.q_start) < std::make_pair(b.it.window, b.it.q_start);
  });
  std::vector<WorkItem> out;
  out.reserve(v.size());
  for (const auto& k : v) out.push_back(k.it);
  return out;
}

namespace {

// One thread per packed position: find the window by binary search on the
// offsets, decode the row-major (dt, dh, dw) inside its box, write the
// canonical id and its inverse.
__global__ void plan_tables_kernel(const int* __restrict__ offsets, const int* __restrict__ dims,
                                   int num_windows, int H, int W, int N, int* __restrict__ ids,
                                   int* __restrict__ pos) {
  // 64-bit loop index: p + stride must not overflow for N close to 2^31
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long pp = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; pp < N; pp += stride) {
    const int p = static_cast<int>(pp);
    int lo = 0, hi = num_windows - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(offsets + mid) <= p) lo = mid; else hi = mid - 1;
    }
    const int* d = dims + 6 * lo;
    const int t0 = __ldg(d + 0), h0 = __ldg(d + 2), h1 = __ldg(d + 3);
    const int w0 = __ldg(d + 4), w1 = __ldg(d + 5);
    const int bw = w1 - w0, plane = (h1 - h0) * bw;
    const int local = p - __ldg(offsets + lo);
    const int dt = local / plane;
    const int r = local - dt * plane;
    const int dh = r / bw;
    const int dw = r - dh * bw;
    const int id = ((t0 + dt) * H + (h0 + dh)) * W + (w0 + dw);
    ids[p] = id;
    pos[id] = p;
  }
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

cudaError_t launch_plan_tables(const wsa_plan_s& p, cudaStream_t s) {
  const int threads = 256;
  const int sms = std::max(1, sm_count());
  const int blocks = static_cast<int>(std::min<long long>(ceil_div(p.num_tokens, threads), 8LL * sms));
  plan_tables_kernel<<<blocks, threads, 0, s>>>(p.d_offsets, p.d_dims, p.num_windows, p.H, p.W,
                                                p.num_tokens, p.d_ids, p.d_pos);
  return cudaGetLastError();
}

namespace {
// Test hook: the next g_fail_allocations plan allocations fail as if the
// device were out of memory (wsa_debug_fail_allocations).
std::atomic<int> g_fail_allocations{0};

bool take_forced_failure() {
  for (int n = g_fail_allocations.load(); n > 0;)
    if (g_fail_allocations.compare_exchange_weak(n, n - 1)) return true;
  return false;
}
}  // namespace

}  // namespace wsa

using namespace wsa;

extern "C" {

int wsa_version(void) { return 100; }

int wsa_bounds_checked(void) { return kBoundsCheck ? 1 : 0; }

wsa_status wsa_debug_fail_allocations(int count) {
  g_fail_allocations.store(count < 0 ? 0 : count);
  return WSA_OK;
}

const char* wsa_last_error(void) { return g_last_error.c_str(); }

wsa_status wsa_window_size(int T, int H, int W, int nt, int nh, int nw, int max_temporal,
                           int* wt, int* wh, int* ww) {
  if (!wt || !wh || !ww) return fail(WSA_ERR_INVALID_ARG, "null output pointer");
  return window_size(T, H, W, nt, nh, nw, max_temporal, wt, wh, ww);
}

wsa_status wsa_layout_windows(int T, int H, int W, int nt, int nh, int nw, wsa_layout layout,
                              int max_temporal, int* dims, int capacity, int* num_windows) {
  if (!num_windows) return fail(WSA_ERR_INVALID_ARG, "num_windows is null");
  if (layout != WSA_REGULAR && layout != WSA_SHIFTED)
    return fail(WSA_ERR_INVALID_ARG, "layout must be WSA_REGULAR or WSA_SHIFTED");
  int wt, wh, ww;
  wsa_status st = window_size(T, H, W, nt, nh, nw, max_temporal, &wt, &wh, &ww);
  if (st != WSA_OK) return st;
  std::vector<int> d;
  layout_boxes(T, H, W, wt, wh, ww, layout == WSA_SHIFTED, &d);
  const int n = static_cast<int>(d.size() / 6);
  *num_windows = n;
  if (dims) {
    if (capacity < n) return fail(WSA_ERR_INVALID_ARG, "dims capacity is smaller than the window count");
    std::memcpy(dims, d.data(), d.size() * sizeof(int));
  }
  return WSA_OK;
}

wsa_status wsa_plan_create(int T, int H, int W, int nt, int nh, int nw, wsa_layout layout,
                           int max_temporal, void* stream, wsa_plan_t* out) {
  if (!out) return fail(WSA_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  if (layout != WSA_REGULAR && layout != WSA_SHIFTED)
    return fail(WSA_ERR_INVALID_ARG, "layout must be WSA_REGULAR or WSA_SHIFTED");
  int wt, wh, ww;
  wsa_status st = window_size(T, H, W, nt, nh, nw, max_temporal, &wt, &wh, &ww);
  if (st != WSA_OK) return st;
  const long long N = static_cast<long long>(T) * H * W;
  if (N >= (1LL << 31)) return fail(WSA_ERR_UNSUPPORTED, "T*H*W must be < 2^31");

  auto* p = new wsa_plan_s();
  p->T = T; p->H = H; p->W = W;
  p->wt = wt; p->wh = wh; p->ww = ww;
  p->layout = layout;
  p->num_tokens = static_cast<int>(N);
  layout_boxes(T, H, W, wt, wh, ww, layout == WSA_SHIFTED, &p->h_dims);
  p->num_windows = static_cast<int>(p->h_dims.size() / 6);
  p->h_offsets.assign(p->num_windows + 1, 0);
  for (int k = 0; k < p->num_windows; ++k) {
    const int* b = &p->h_dims[6 * k];
    const int n = (b[1] - b[0]) * (b[3] - b[2]) * (b[5] - b[4]);
    p->h_offsets[k + 1] = p->h_offsets[k] + n;
    p->max_window_tokens = std::max(p->max_window_tokens, n);
  }
  const std::vector<WorkItem> tc = make_items(p->h_offsets, kTcItemRows, 128);
  const std::vector<WorkItem> simt = make_items(p->h_offsets, kSimtItemRows, kSimtItemRows);
  p->num_tc_items = static_cast<int>(tc.size());
  p->num_simt_items = static_cast<int>(simt.size());

  // one device block: offsets | dims | ids | pos | tc items | simt items | workspace
  const size_t a = 256;
  size_t off_offsets = 0;
  size_t off_dims = align_up(off_offsets + p->h_offsets.size() * sizeof(int), a);
  size_t off_ids = align_up(off_dims + p->h_dims.size() * sizeof(int), a);
  size_t off_pos = align_up(off_ids + N * sizeof(int), a);
  size_t off_tc = align_up(off_pos + N * sizeof(int), a);
  size_t off_simt = align_up(off_tc + tc.size() * sizeof(WorkItem), a);
  size_t off_work = align_up(off_simt + simt.size() * sizeof(WorkItem), a);
  size_t total = align_up(off_work + WS_WORDS * sizeof(int), a);

  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess && take_forced_failure()) {
    delete p;
    return fail(WSA_ERR_OOM, "wsa_plan_create: device allocation failed (forced by wsa_debug_fail_allocations)");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p->stream = s;
  // stream-ordered: no device-wide synchronisation, ready in stream order
  if (e == cudaSuccess) e = cudaMallocAsync(&p->d_block, total, s);
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "wsa_plan_create: cudaMallocAsync");
  }
  char* base = static_cast<char*>(p->d_block);
  p->d_offsets = reinterpret_cast<int*>(base + off_offsets);
  p->d_dims = reinterpret_cast<int*>(base + off_dims);
  p->d_ids = reinterpret_cast<int*>(base + off_ids);
  p->d_pos = reinterpret_cast<int*>(base + off_pos);
  p->d_tc_items = reinterpret_cast<WorkItem*>(base + off_tc);
  p->d_simt_items = reinterpret_cast<WorkItem*>(base + off_simt);
  p->d_work = reinterpret_cast<int*>(base + off_work);

  // Host sources are pageable vectors: cudaMemcpyAsync from pageable memory
  // copies out of them before returning, so they may go out of scope.
  e = cudaMemcpyAsync(p->d_offsets, p->h_offsets.data(), p->h_offsets.size() * sizeof(int),
                      cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p->d_dims, p->h_dims.data(), p->h_dims.size() * sizeof(int),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p->d_tc_items, tc.data(), tc.size() * sizeof(WorkItem), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p->d_simt_items, simt.data(), simt.size() * sizeof(WorkItem),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->d_work, 0, WS_WORDS * sizeof(int), s);
  if (e == cudaSuccess) e = launch_plan_tables(*p, s);
  if (e != cudaSuccess) {
    cudaFreeAsync(p->d_block, s);
    delete p;
    return cuda_fail(e, "wsa_plan_create: upload / plan kernel");
  }
  *out = p;
  return WSA_OK;
}

wsa_status wsa_plan_destroy(wsa_plan_t plan) {
  if (!plan) return fail(WSA_ERR_INVALID_ARG, "plan is null");
  cudaError_t e = cudaSuccess;
  // released in the order of the plan's latest call: later work on that
  // stream may reuse the memory, earlier work has finished with it
  if (plan->d_block) e = cudaFreeAsync(plan->d_block, plan->stream);
  delete plan;
  if (e != cudaSuccess) return cuda_fail(e, "wsa_plan_destroy: cudaFreeAsync");
  return WSA_OK;
}

wsa_status wsa_plan_info(wsa_plan_t plan, int* num_windows, int* num_tokens, int* max_window_tokens,
                         int* wt, int* wh, int* ww, int* layout) {
  if (!plan) return fail(WSA_ERR_INVALID_ARG, "plan is null");
  if (num_windows) *num_windows = plan->num_windows;
  if (num_tokens) *num_tokens = plan->num_tokens;
  if (max_window_tokens) *max_window_tokens = plan->max_window_tokens;
  if (wt) *wt = plan->wt;
  if (wh) *wh = plan->wh;
  if (ww) *ww = plan->ww;
  if (layout) *layout = plan->layout;
  return WSA_OK;
}

wsa_status wsa_plan_tables(wsa_plan_t plan, const int** offsets, const int** dims, const int** ids,
                           const int** pos) {
  if (!plan) return fail(WSA_ERR_INVALID_ARG, "plan is null");
  if (offsets) *offsets = plan->d_offsets;
  if (dims) *dims = plan->d_dims;
  if (ids) *ids = plan->d_ids;
  if (pos) *pos = plan->d_pos;
  return WSA_OK;
}

wsa_status wsa_plan_device_status(wsa_plan_t plan, int* code) {
  if (!plan || !code) return fail(WSA_ERR_INVALID_ARG, "plan or code is null");
  // Every launch that can record an error in this plan ran on the stream of
  // the plan's latest call or was ordered before it (one stream per plan).
  const cudaStream_t s = plan->stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_plan_device_status: synchronize");
  // WS_ERROR and WS_BOUNDS are adjacent words: read and clear both.
  static_assert(WS_BOUNDS == WS_ERROR + 1, "error words must be adjacent");
  int words[2] = {0, 0};
  e = cudaMemcpyAsync(words, plan->d_work + WS_ERROR, sizeof(words), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_plan_device_status: read");
  *code = words[0] != 0 ? words[0] : words[1];
  if (*code != 0) {
    const int zero[2] = {0, 0};
    e = cudaMemcpyAsync(plan->d_work + WS_ERROR, zero, sizeof(zero), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "wsa_plan_device_status: clear");
    if (words[0] != 0)
      return fail(WSA_ERR_DEVICE_CHECK, "a kernel recorded device error code " + std::to_string(words[0]));
    return fail(WSA_ERR_DEVICE_CHECK, "a plan table held a row index out of range (device code " +
                                          std::to_string(words[1]) + ", bounds-checked build)");
  }
  return WSA_OK;
}

}  // extern "C"
