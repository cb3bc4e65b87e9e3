// wsa_attention_noalloc: the bf16 tensor-core window attention for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not an option -- a host
// application whose device memory is entirely owned by another framework's
// pool, or a latency-critical serving loop that must not take the implicit
// device synchronisation of cudaMalloc/cudaFree.  Those callers cannot create
// a plan (wsa_plan_create allocates the plan's tables), so this entry point
// takes the grid and layout directly and keeps everything the kernels need
// beyond the caller's tensors -- window offsets and boxes,
// the ids/pos tables, the work list and the scheduler words -- in one
// file-scope device array of fixed size.
//
// It reuses the library's plan-table kernel and tensor-core attention kernel
// unchanged; only the memory they are pointed at differs.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "wsa_internal.h"

namespace wsa {
namespace {

// Limits of the static scratch.
constexpr int kNoAllocMaxTokens = 1 << 19;  // 524,288 tokens (T*H*W)
constexpr int kNoAllocMaxWindows = 8192;
constexpr int kNoAllocMaxItems = 16384;     // work items of 256 query rows

constexpr size_t pad64(size_t words) { return (words + 63) / 64 * 64; }  // 256-byte sub-buffers

constexpr size_t kOffWork = 0;
constexpr size_t kOffOffsets = kOffWork + pad64(WS_WORDS);
constexpr size_t kOffDims = kOffOffsets + pad64(kNoAllocMaxWindows + 1);
constexpr size_t kOffIds = kOffDims + pad64(6 * static_cast<size_t>(kNoAllocMaxWindows));
constexpr size_t kOffPos = kOffIds + pad64(kNoAllocMaxTokens);
constexpr size_t kOffItems = kOffPos + pad64(kNoAllocMaxTokens);
constexpr size_t kItemWords = sizeof(WorkItem) / sizeof(int);
constexpr size_t kScratchWords = kOffItems + pad64(kItemWords * kNoAllocMaxItems);  // ~4.6 MB

// Every device that loads the library holds this array until the process exits.
static __device__ __align__(256) int g_noalloc_scratch[kScratchWords];

// Device address of the scratch array on the current device.  The array's
// name in host code is only a host-side stand-in, so the address is looked up
// once per device with that device current and cached for the life of the
// process (a device reset, which destroys the array, ends that life).
wsa_status scratch_address(int device, int** out) {
  static std::mutex mu;
  static std::vector<int*> cache;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= device) cache.resize(device + 1, nullptr);
  if (cache[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "wsa_attention_noalloc: cudaGetSymbolAddress");
    cache[device] = static_cast<int*>(p);
  }
  *out = cache[device];
  return WSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const auto x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace wsa

using namespace wsa;

extern "C" wsa_status wsa_attention_noalloc(int T, int H, int W, int nt, int nh, int nw, wsa_layout layout,
                                            int max_temporal, const void* q, const void* k, const void* v,
                                            void* o, int heads, int in_order_canonical, float softmax_scale,
                                            void* stream) {
  if (layout != WSA_REGULAR && layout != WSA_SHIFTED)
    return fail(WSA_ERR_INVALID_ARG, "layout must be WSA_REGULAR or WSA_SHIFTED");
  if (!q || !k || !v || !o) return fail(WSA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (heads <= 0) return fail(WSA_ERR_INVALID_ARG, "heads must be > 0");
  if (heads > 65535) return fail(WSA_ERR_UNSUPPORTED, "at most 65535 heads");
  if (in_order_canonical != 0 && in_order_canonical != 1)
    return fail(WSA_ERR_INVALID_ARG, "in_order_canonical must be 0 or 1");
  if (!std::isfinite(softmax_scale)) return fail(WSA_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(WSA_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  int wt, wh, ww;
  wsa_status st = window_size(T, H, W, nt, nh, nw, max_temporal, &wt, &wh, &ww);
  if (st != WSA_OK) return st;
  const long long N = static_cast<long long>(T) * H * W;
  if (N > kNoAllocMaxTokens)
    return fail(WSA_ERR_UNSUPPORTED, "wsa_attention_noalloc: T*H*W = " + std::to_string(N) +
                                         " exceeds its static scratch limit of " +
                                         std::to_string(kNoAllocMaxTokens) + " tokens; use wsa_attention");
  const size_t bytes = static_cast<size_t>(N) * heads * 128 * 2;
  if (overlap(o, bytes, q, bytes) || overlap(o, bytes, k, bytes) || overlap(o, bytes, v, bytes))
    return fail(WSA_ERR_INVALID_ARG, "o must not overlap q, k or v");

  // Host geometry, exactly as wsa_plan_create computes it.
  wsa_plan_s view;
  view.T = T; view.H = H; view.W = W;
  view.wt = wt; view.wh = wh; view.ww = ww;
  view.layout = layout;
  view.num_tokens = static_cast<int>(N);
  layout_boxes(T, H, W, wt, wh, ww, layout == WSA_SHIFTED, &view.h_dims);
  view.num_windows = static_cast<int>(view.h_dims.size() / 6);
  if (view.num_windows > kNoAllocMaxWindows)
    return fail(WSA_ERR_UNSUPPORTED, "wsa_attention_noalloc: " + std::to_string(view.num_windows) +
                                         " windows exceed its static scratch limit of " +
                                         std::to_string(kNoAllocMaxWindows));
  view.h_offsets.assign(view.num_windows + 1, 0);
  for (int w = 0; w < view.num_windows; ++w) {
    const int* b = &view.h_dims[6 * w];
    view.h_offsets[w + 1] = view.h_offsets[w] + (b[1] - b[0]) * (b[3] - b[2]) * (b[5] - b[4]);
  }
  const std::vector<WorkItem> items = make_items(view.h_offsets, kTcItemRows, 128);
  view.num_tc_items = static_cast<int>(items.size());
  if (view.num_tc_items > kNoAllocMaxItems)
    return fail(WSA_ERR_UNSUPPORTED, "wsa_attention_noalloc: " + std::to_string(view.num_tc_items) +
                                         " work items exceed its static scratch limit of " +
                                         std::to_string(kNoAllocMaxItems));
  if (static_cast<long long>(view.num_tc_items) * heads >= (1LL << 31))
    return fail(WSA_ERR_UNSUPPORTED, "too many work units (windows x heads)");

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_attention_noalloc: cudaGetDevice");
  int* base = nullptr;
  st = scratch_address(dev, &base);
  if (st != WSA_OK) return st;
  view.device = dev;
  view.d_work = base + kOffWork;
  view.d_offsets = base + kOffOffsets;
  view.d_dims = base + kOffDims;
  view.d_ids = base + kOffIds;
  view.d_pos = base + kOffPos;
  view.d_tc_items = reinterpret_cast<WorkItem*>(base + kOffItems);

  // The array keeps the previous call's contents: the scheduler and error
  // words are cleared, every table entry the kernels read is rewritten.
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(128.0f);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(view.d_work, 0, WS_WORDS * sizeof(int), s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(view.d_offsets, view.h_offsets.data(), view.h_offsets.size() * sizeof(int),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(view.d_dims, view.h_dims.data(), view.h_dims.size() * sizeof(int),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(view.d_tc_items, items.data(), items.size() * sizeof(WorkItem), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = launch_plan_tables(view, s);
  if (e == cudaSuccess)
    e = launch_attention_bf16_tc(view, q, k, v, o, heads, in_order_canonical == 1, scale, s);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_attention_noalloc: launch");
  return WSA_OK;
}

extern "C" wsa_status wsa_noalloc_device_status(int* code) {
  if (!code) return fail(WSA_ERR_INVALID_ARG, "code is null");
  *code = 0;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_noalloc_device_status: cudaGetDevice");
  int* base = nullptr;
  wsa_status st = scratch_address(dev, &base);
  if (st != WSA_OK) return st;
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "wsa_noalloc_device_status: synchronize");
  // WS_ERROR and WS_BOUNDS are adjacent words of the array: read and clear both.
  static_assert(WS_BOUNDS == WS_ERROR + 1, "error words must be adjacent");
  int words[2] = {0, 0};
  int* err = base + kOffWork + WS_ERROR;
  e = cudaMemcpy(words, err, sizeof(words), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_noalloc_device_status: read");
  *code = words[0] != 0 ? words[0] : words[1];
  if (*code == 0) return WSA_OK;
  const int zero[2] = {0, 0};
  e = cudaMemcpy(err, zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_noalloc_device_status: clear");
  if (words[0] != 0)
    return fail(WSA_ERR_DEVICE_CHECK, "a kernel recorded device error code " + std::to_string(words[0]));
  return fail(WSA_ERR_DEVICE_CHECK, "a table held a row index out of range (device code " +
                                        std::to_string(words[1]) + ", bounds-checked build)");
}
