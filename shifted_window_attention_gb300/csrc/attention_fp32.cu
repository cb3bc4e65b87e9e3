// fp32 window attention on CUDA cores.
//
// "Window-Aligned Sequence Parallelism (SeedVR2)", section "Motivation":
// attention only inside each window.  For window w and head h,
// O = softmax(Q K^T * scale) V over the window's tokens, in fp32 throughout
// (fp32 inputs and outputs; TF32 tensor cores would not keep the fp32
// tolerance, so this path uses FFMA).
//
// One block of 64 threads owns 64 query rows of one (window, head); thread i
// owns query row i.  Key/value tiles of 64 rows are gathered through the
// plan's ids table into shared memory; each thread scores the tile, keeps a
// running max and sum (online softmax, rescaling its accumulator when the max
// grows) and accumulates P V in registers.  Output rows are scattered back
// through the same table.

#include <algorithm>
#include <cmath>

#include "wsa_internal.h"

namespace wsa {
namespace {

constexpr int kRows = kSimtItemRows;  // 64 query rows per block
constexpr int kKv = 64;               // key rows per tile

template <int D>
__global__ void __launch_bounds__(kRows)
attention_fp32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                      const float* __restrict__ v, float* __restrict__ o,
                      const int* __restrict__ row_map, const int* __restrict__ offsets,
                      const WorkItem* __restrict__ items, int heads, float scale, int n_tokens,
                      int* __restrict__ bounds) {
  extern __shared__ float smem[];
  float* q_s = smem;                       // [kRows][D + 1] (padded: conflict-free row reads)
  float* k_s = q_s + kRows * (D + 1);      // [kKv][D]
  float* v_s = k_s + kKv * D;              // [kKv][D]
  float* s_s = v_s + kKv * D;              // [kKv][kRows]

  const WorkItem it = items[blockIdx.x];
  const int head = blockIdx.y;
  const int off = offsets[it.window];
  const int n = offsets[it.window + 1] - off;
  const int tid = threadIdx.x;
  const size_t stride = static_cast<size_t>(heads) * D;
  // Token of window row r; -1 (bounds-checked builds) when the table entry is
  // out of range: the row then reads as zeros and is not written.
  auto token = [&](int r) -> long long {
    const long long t = row_map ? row_map[off + r] : off + r;
    if (kBoundsCheck && static_cast<unsigned long long>(t) >= static_cast<unsigned long long>(n_tokens)) {
      atomicCAS(bounds, 0, kErrBounds);
      return -1;
    }
    return t;
  };

  const int qr = it.q_start + tid;
  long long q_tok = qr < n ? token(qr) : -1;
  const bool q_valid = q_tok >= 0;
  if (!q_valid) q_tok = 0;
  for (int c = 0; c < D; ++c)
    q_s[tid * (D + 1) + c] = q_valid ? q[q_tok * stride + head * D + c] : 0.f;

  float acc[D];
#pragma unroll
  for (int c = 0; c < D; ++c) acc[c] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int kv0 = 0; kv0 < n; kv0 += kKv) {
    const int kv_n = min(kKv, n - kv0);
    __syncthreads();  // previous tile fully consumed
    if (tid < kv_n) {
      const long long t = token(kv0 + tid);
      float4* kd = reinterpret_cast<float4*>(k_s + tid * D);
      float4* vd = reinterpret_cast<float4*>(v_s + tid * D);
      if (t >= 0) {
        const float4* ks = reinterpret_cast<const float4*>(k + t * stride + head * D);
        const float4* vs = reinterpret_cast<const float4*>(v + t * stride + head * D);
        for (int c = 0; c < D / 4; ++c) {
          kd[c] = ks[c];
          vd[c] = vs[c];
        }
      } else {
        for (int c = 0; c < D / 4; ++c) kd[c] = vd[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncthreads();
    float tmax = -INFINITY;
    for (int j = 0; j < kv_n; ++j) {
      float s = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; ++c) s = fmaf(q_s[tid * (D + 1) + c], k_s[j * D + c], s);
      s *= scale;
      s_s[j * kRows + tid] = s;
      tmax = fmaxf(tmax, s);
    }
    const float m_new = fmaxf(m, tmax);
    const float alpha = expf(m - m_new);  // 0 on the first tile (m = -inf)
    l *= alpha;
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] *= alpha;
    for (int j = 0; j < kv_n; ++j) {
      const float p = expf(s_s[j * kRows + tid] - m_new);
      l += p;
#pragma unroll
      for (int c = 0; c < D; ++c) acc[c] = fmaf(p, v_s[j * D + c], acc[c]);
    }
    m = m_new;
  }
  if (q_valid) {
    const float inv = 1.f / l;
    float* dst = o + q_tok * stride + head * D;
#pragma unroll
    for (int c = 0; c < D; ++c) dst[c] = acc[c] * inv;
  }
}

template <int D>
cudaError_t launch(const wsa_plan_s& p, const float* q, const float* k, const float* v, float* o,
                   int heads, bool canonical, float scale, cudaStream_t s) {
  const size_t smem = sizeof(float) * (kRows * (D + 1) + 2 * kKv * D + kKv * kRows);
  cudaError_t e = cudaFuncSetAttribute(attention_fp32_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_simt_items, heads);
  attention_fp32_kernel<D><<<grid, kRows, smem, s>>>(q, k, v, o, canonical ? p.d_ids : nullptr,
                                                     p.d_offsets, p.d_simt_items, heads, scale, p.num_tokens,
                                                     p.d_work + WS_BOUNDS);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_fp32(const wsa_plan_s& p, const float* q, const float* k,
                                  const float* v, float* o, int heads, int head_dim,
                                  bool canonical, float scale, cudaStream_t s) {
  if (head_dim == 64) return launch<64>(p, q, k, v, o, heads, canonical, scale, s);
  return launch<128>(p, q, k, v, o, heads, canonical, scale, s);
}

}  // namespace wsa
