// Layout transition: the local permutation between two window layouts.
//
// "Window-Aligned Sequence Parallelism (SeedVR2)", sections "Motivation" and
// "Plan A redistribution": with one rank, moving the activations from one
// layout to the next is a permutation of rows.  Destination row p holds the
// token at packed position p of the destination plan, which the source plan
// stores at row pos_src[ids_dst[p]].
//
// The same kernel serves the row gather of the Plan A exchange (pack and
// unpack: y[i] = x[index[i]], one table level).  A table entry outside the
// table or tensor it indexes is skipped (its destination row is left
// unwritten), so a bad table cannot make the kernel read out of bounds; in
// bounds-checked builds the skip is also recorded in the plan's WS_BOUNDS word.
//
// The kernel is pure data movement and HBM-bound: every byte is read once and
// written once.  One warp moves one row at a time with 16-byte vector loads,
// keeping up to kVecPerLane loads in flight per lane before it stores them;
// the two table lookups per row hit L2.  Loads and stores use the streaming
// cache hints since neither side is reused.

#include <algorithm>

#include "wsa_internal.h"

namespace wsa {
namespace {

constexpr int kVecPerLane = 12;      // 12 x 16 B x 32 lanes = one 6 KB row per pass
constexpr int kThreads = 256;

template <typename Vec>
__global__ void __launch_bounds__(kThreads)
transition_rows_kernel(const Vec* __restrict__ src, Vec* __restrict__ dst,
                       const int* __restrict__ first, const int* __restrict__ second,
                       int n_rows, int vec_per_row, int src_rows, int* __restrict__ bounds) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = kThreads / 32;
  const long long warp0 = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
  const long long nwarps = static_cast<long long>(gridDim.x) * warps_per_block;
  for (long long row = warp0; row < n_rows; row += nwarps) {
    int g = __ldg(first + row);  // transition: ids_dst[row]; gather: index[row]
    // transition: pos_src[...] (pos_src has src_rows entries, like x_src)
    if (second && static_cast<unsigned>(g) < static_cast<unsigned>(src_rows)) g = __ldg(second + g);
    if (static_cast<unsigned>(g) >= static_cast<unsigned>(src_rows)) {
      if (kBoundsCheck && bounds && lane == 0) atomicCAS(bounds, 0, kErrBounds);
      continue;
    }
    const Vec* s = src + static_cast<long long>(g) * vec_per_row;
    Vec* d = dst + row * vec_per_row;
    for (int base = 0; base < vec_per_row; base += 32 * kVecPerLane) {
      Vec buf[kVecPerLane];
#pragma unroll
      for (int i = 0; i < kVecPerLane; ++i) {
        const int c = base + i * 32 + lane;
        if (c < vec_per_row) buf[i] = __ldcs(s + c);
      }
#pragma unroll
      for (int i = 0; i < kVecPerLane; ++i) {
        const int c = base + i * 32 + lane;
        if (c < vec_per_row) __stcs(d + c, buf[i]);
      }
    }
  }
}

template <typename Vec>
cudaError_t launch_rows(const void* x_src, void* x_dst, const int* first, const int* second, int n_rows,
                        int src_rows, size_t row_bytes, int* bounds, cudaStream_t s) {
  const int vec_per_row = static_cast<int>(row_bytes / sizeof(Vec));
  const int sms = std::max(1, sm_count());
  // 8 resident blocks of 256 threads per SM: 64 warps, the SM's limit.
  const long long want = (static_cast<long long>(n_rows) + 7) / 8;
  const int blocks = static_cast<int>(std::max(1LL, std::min<long long>(want, 8LL * sms)));
  transition_rows_kernel<Vec><<<blocks, kThreads, 0, s>>>(
      static_cast<const Vec*>(x_src), static_cast<Vec*>(x_dst), first, second, n_rows, vec_per_row, src_rows,
      bounds);
  return cudaGetLastError();
}

cudaError_t launch_any(const void* x_src, void* x_dst, const int* first, const int* second, int n_rows,
                       int src_rows, size_t row_bytes, int* bounds, cudaStream_t s) {
  const auto a = reinterpret_cast<uintptr_t>(x_src) | reinterpret_cast<uintptr_t>(x_dst);
  if (row_bytes % 16 == 0 && a % 16 == 0)
    return launch_rows<uint4>(x_src, x_dst, first, second, n_rows, src_rows, row_bytes, bounds, s);
  if (row_bytes % 4 == 0 && a % 4 == 0)
    return launch_rows<unsigned int>(x_src, x_dst, first, second, n_rows, src_rows, row_bytes, bounds, s);
  return launch_rows<unsigned short>(x_src, x_dst, first, second, n_rows, src_rows, row_bytes, bounds, s);
}

}  // namespace

cudaError_t launch_transition(const wsa_plan_s& src, const wsa_plan_s& dst, const void* x_src,
                              void* x_dst, size_t row_bytes, cudaStream_t s) {
  return launch_any(x_src, x_dst, dst.d_ids, src.d_pos, dst.num_tokens, src.num_tokens, row_bytes,
                    dst.d_work + WS_BOUNDS, s);
}

cudaError_t launch_gather_rows(const void* x, int x_rows, const int* index, void* y, int rows, size_t row_bytes,
                               cudaStream_t s) {
  return launch_any(x, y, index, nullptr, rows, x_rows, row_bytes, nullptr, s);
}

}  // namespace wsa
