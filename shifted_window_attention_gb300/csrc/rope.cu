// Window-local 3D rotary position embedding of Q and K rows.
//
// "Window-Aligned Sequence Parallelism (SeedVR2)", section "Reference quirks
// reproduced on purpose": positions are window-local, so a video token at
// (dt, dh, dw) inside its window takes the axial indices
// (text_len + dt, dh, dw), and every window restarts at 0.  The rotary span
// is 3 * (rope_dim // 3) channels.  Text token i takes (i, i, i).  Axis a of
// (t, h, w) owns channels [a*da, (a+1)*da) with da = rope_dim // 3.  Within
// an axis, channels (2j, 2j+1) turn by pos_a * theta^(-2j/da).
//
// Window-local coordinates need no table: windows are products of axis
// intervals, so the coordinate on an axis is the token's coordinate minus
// the start of its interval.  With cuts at 0, s, s + w, s + 2w, ... (s = 0
// for the regular layout; s = floor(w/2) for the shifted one on an axis
// longer than its window), the start is 0 when x < s and
// s + floor((x - s)/w) * w otherwise.  Rows in canonical order are streamed
// in order; packed rows read their canonical id from the plan.
//
// The kernel is pure streaming and HBM-bound.  One warp owns one token row
// (all heads) at a time and reads and writes it once, with 16-byte vectors.
// A head's row spans 8, 16 or 32 vectors, which divides the 32 lanes, so
// every lane sees the same channel slice in every head.  Each lane therefore
// computes the sines and cosines of its 2 or 4 rotation pairs once per row
// and applies them to all heads.  The angle is formed as a float pair: the
// frequency is split into hi + lo on the host and the product pos * hi is
// made exact with an fma.  This keeps the fp32 rotation accurate at positions
// of several hundred.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "wsa_internal.h"

namespace wsa {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPairs = 32;  // per axis
constexpr int kBatch = 8;      // 16-byte vectors per lane and tensor loaded before any store

struct RopeParams {
  const char* x[2];
  char* y[2];
  int ntensors;
  int video;            // 1: video rows of a plan; 0: text rows
  const int* ids;       // packed rows: canonical id of row p (null: canonical or text rows)
  int H, W;             // grid (decoding a canonical id)
  int win[3], shift[3]; // window size and first interior cut per axis (t, h, w)
  int n_rows;
  int text_len;
  int da;               // channels per axis (even)
  int vec_per_row;      // 16-byte vectors per token row
  int vec_per_head;
  float2 freq[kMaxPairs];  // theta^(-2j/da) as hi + lo
};

__device__ __forceinline__ int local_coord(int x, int w, int s) {
  return x < s ? x : (x - s) % w;
}

// Window-local axial position of canonical token id.
__device__ __forceinline__ void video_position(const RopeParams& P, int id, float (&pos)[3]) {
  const int x = id % P.W, th = id / P.W;
  const int y = th % P.H, t = th / P.H;
  pos[0] = static_cast<float>(P.text_len + local_coord(t, P.win[0], P.shift[0]));
  pos[1] = static_cast<float>(local_coord(y, P.win[1], P.shift[1]));
  pos[2] = static_cast<float>(local_coord(x, P.win[2], P.shift[2]));
}

__device__ __forceinline__ void rotate_pair(float& x0, float& x1, float c, float s) {
  const float a = x0 * c - x1 * s;
  const float b = x0 * s + x1 * c;
  x0 = a;
  x1 = b;
}

template <typename T>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static void load(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static uint4 store(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Vec16<float> {
  static constexpr int kElems = 4;
  __device__ static void load(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 store(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) rope_kernel(const RopeParams P) {
  using V = Vec16<T>;
  constexpr int E = V::kElems, NP = E / 2;
  const int lane = threadIdx.x & 31;
  const long long warp0 = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  const long long nwarps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  const int c0 = (lane % P.vec_per_head) * E;  // first channel of this lane's slice in every head
  for (long long p = warp0; p < P.n_rows; p += nwarps) {
    float pos[3];
    const int id = P.ids ? __ldg(P.ids + p) : static_cast<int>(p);
    if (P.video) {
      video_position(P, id, pos);
    } else {
      pos[0] = pos[1] = pos[2] = static_cast<float>(p);
    }
    float cs[NP], sn[NP];
    bool rot[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int c = c0 + 2 * i;
      rot[i] = c < 3 * P.da;
      cs[i] = 1.f;
      sn[i] = 0.f;
      if (rot[i]) {
        const int a = c / P.da;
        const float2 f = P.freq[(c - a * P.da) >> 1];
        const float hi = pos[a] * f.x;
        const float lo = fmaf(pos[a], f.x, -hi) + pos[a] * f.y;  // angle = hi + lo
        float s, k;
        sincosf(hi, &s, &k);
        cs[i] = k - lo * s;  // cos(hi + lo), |lo| << 1
        sn[i] = s + lo * k;  // sin(hi + lo)
      }
    }
    const long long row = p;  // canonical rows are processed in canonical order
    // Loads of a batch are issued before its stores: an output may be its own
    // input, so the compiler cannot move later loads above earlier stores.
    for (int base = lane; base < P.vec_per_row; base += 32 * kBatch) {
      uint4 buf[2][kBatch];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint4* src = reinterpret_cast<const uint4*>(P.x[t]) + row * P.vec_per_row;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int v = base + 32 * b;
          if (t < P.ntensors && v < P.vec_per_row) buf[t][b] = __ldcs(src + v);
        }
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint4* dst = reinterpret_cast<uint4*>(P.y[t]) + row * P.vec_per_row;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int v = base + 32 * b;
          if (t < P.ntensors && v < P.vec_per_row) {
            float f[E];
            V::load(buf[t][b], f);
#pragma unroll
            for (int i = 0; i < NP; ++i)
              if (rot[i]) rotate_pair(f[2 * i], f[2 * i + 1], cs[i], sn[i]);
            __stcs(dst + v, V::store(f));
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_rope(const wsa_plan_s* plan, bool canonical, const void* const x[2], void* const y[2],
                        int ntensors, int n_rows, int heads, int head_dim, bool bf16, int text_len, int rope_dim,
                        double theta, cudaStream_t s) {
  RopeParams P{};
  for (int t = 0; t < 2; ++t) {
    P.x[t] = static_cast<const char*>(x[t]);
    P.y[t] = static_cast<char*>(y[t]);
  }
  P.ntensors = ntensors;
  P.video = plan ? 1 : 0;
  P.ids = plan && !canonical ? plan->d_ids : nullptr;
  if (plan) {
    P.H = plan->H;
    P.W = plan->W;
    const int size[3] = {plan->T, plan->H, plan->W}, win[3] = {plan->wt, plan->wh, plan->ww};
    for (int a = 0; a < 3; ++a) {
      P.win[a] = win[a];
      // the shifted layout moves the cuts of an axis longer than its window
      P.shift[a] = plan->layout == WSA_SHIFTED && size[a] > win[a] ? win[a] / 2 : 0;
    }
  }
  P.n_rows = n_rows;
  P.text_len = text_len;
  P.da = rope_dim / 3;
  const int elt = bf16 ? 2 : 4;
  P.vec_per_head = head_dim * elt / 16;
  P.vec_per_row = heads * P.vec_per_head;
  for (int j = 0; j < P.da / 2 && j < kMaxPairs; ++j) {
    const double f = std::pow(theta, -2.0 * j / P.da);
    const float hi = static_cast<float>(f);
    P.freq[j] = make_float2(hi, static_cast<float>(f - static_cast<double>(hi)));
  }
  if (n_rows == 0) return cudaSuccess;
  const int sms = std::max(1, sm_count());
  // two resident blocks of 256 threads per SM (about 110 registers a thread)
  const long long want = (static_cast<long long>(n_rows) + 7) / 8;
  const int blocks = static_cast<int>(std::max(1LL, std::min<long long>(want, 2LL * sms)));
  if (bf16)
    rope_kernel<__nv_bfloat16><<<blocks, kThreads, 0, s>>>(P);
  else
    rope_kernel<float><<<blocks, kThreads, 0, s>>>(P);
  return cudaGetLastError();
}

}  // namespace wsa
