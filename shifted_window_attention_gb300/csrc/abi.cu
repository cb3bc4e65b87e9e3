// C-ABI entry points for attention and the layout transition: argument
// validation on the host, then one kernel launch each.  Each dtype has exactly
// one kernel; nothing falls back to another implementation.

#include <cmath>
#include <cstdint>

#include "wsa_internal.h"

using namespace wsa;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const auto x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

wsa_status wsa_debug_withhold_units(int launches) {
  withhold_attention_units(launches);
  return WSA_OK;
}

wsa_status wsa_attention(wsa_plan_t plan, const void* q, const void* k, const void* v, void* o,
                         int heads, int head_dim, wsa_dtype dtype, int in_order_canonical,
                         float softmax_scale, void* stream) {
  if (!plan) return fail(WSA_ERR_INVALID_ARG, "plan is null");
  if (!q || !k || !v || !o) return fail(WSA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (heads <= 0) return fail(WSA_ERR_INVALID_ARG, "heads must be > 0");
  if (dtype != WSA_BF16 && dtype != WSA_FP32) return fail(WSA_ERR_INVALID_ARG, "unknown dtype");
  if (in_order_canonical != 0 && in_order_canonical != 1)
    return fail(WSA_ERR_INVALID_ARG, "in_order_canonical must be 0 or 1");
  if (!std::isfinite(softmax_scale)) return fail(WSA_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (dtype == WSA_BF16 && head_dim != 128)
    return fail(WSA_ERR_UNSUPPORTED, "bf16 attention supports head_dim 128 only");
  if (dtype == WSA_FP32 && head_dim != 64 && head_dim != 128)
    return fail(WSA_ERR_UNSUPPORTED, "fp32 attention supports head_dim 64 or 128");
  const size_t elt = dtype == WSA_BF16 ? 2 : 4;
  const size_t bytes = static_cast<size_t>(plan->num_tokens) * heads * head_dim * elt;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(WSA_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (overlap(o, bytes, q, bytes) || overlap(o, bytes, k, bytes) || overlap(o, bytes, v, bytes))
    return fail(WSA_ERR_INVALID_ARG, "o must not overlap q, k or v");
  if (static_cast<long long>(plan->num_tc_items) * heads >= (1LL << 31))
    return fail(WSA_ERR_UNSUPPORTED, "too many work units (windows x heads)");
  if (dtype == WSA_BF16 && (heads > 65535 || plan->num_windows > 65535))
    return fail(WSA_ERR_UNSUPPORTED, "bf16 attention supports at most 65535 heads and 65535 windows");
  if (heads > 65535 && dtype == WSA_FP32)
    return fail(WSA_ERR_UNSUPPORTED, "fp32 attention supports at most 65535 heads");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_attention: cudaGetDevice");
  if (dev != plan->device) return fail(WSA_ERR_INVALID_ARG, "plan was created on another device");

  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  plan->stream = s;
  if (dtype == WSA_FP32) {
    e = launch_attention_fp32(*plan, static_cast<const float*>(q), static_cast<const float*>(k),
                              static_cast<const float*>(v), static_cast<float*>(o), heads, head_dim,
                              in_order_canonical == 1, scale, s);
  } else {
    e = launch_attention_bf16_tc(*plan, q, k, v, o, heads, in_order_canonical == 1, scale, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "wsa_attention: launch");
  return WSA_OK;
}

wsa_status wsa_attention_text_workspace(wsa_plan_t plan, int n_text, int heads, int head_dim, wsa_dtype dtype,
                                        size_t* bytes) {
  if (!plan || !bytes) return fail(WSA_ERR_INVALID_ARG, "plan and bytes must be non-null");
  if (n_text <= 0 || heads <= 0) return fail(WSA_ERR_INVALID_ARG, "n_text and heads must be > 0");
  if (dtype != WSA_BF16 || head_dim != 128)
    return fail(WSA_ERR_UNSUPPORTED, "the text segment is implemented for bf16, head_dim 128");
  *bytes = attention_text_workspace_bytes(*plan, n_text, heads, nullptr);
  return WSA_OK;
}

wsa_status wsa_attention_text(wsa_plan_t plan, const void* q, const void* k, const void* v, void* o,
                              const void* q_txt, const void* k_txt, const void* v_txt, void* o_txt, int n_text,
                              int heads, int head_dim, wsa_dtype dtype, int in_order_canonical, float softmax_scale,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan) return fail(WSA_ERR_INVALID_ARG, "plan is null");
  if (!q || !k || !v || !o || !q_txt || !k_txt || !v_txt || !o_txt || !workspace)
    return fail(WSA_ERR_INVALID_ARG, "tensors and workspace must be non-null");
  if (n_text <= 0 || heads <= 0) return fail(WSA_ERR_INVALID_ARG, "n_text and heads must be > 0");
  if (in_order_canonical != 0 && in_order_canonical != 1)
    return fail(WSA_ERR_INVALID_ARG, "in_order_canonical must be 0 or 1");
  if (!std::isfinite(softmax_scale)) return fail(WSA_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (dtype != WSA_BF16 || head_dim != 128)
    return fail(WSA_ERR_UNSUPPORTED, "the text segment is implemented for bf16, head_dim 128");
  if (heads > 65535 || plan->num_windows > 65535)
    return fail(WSA_ERR_UNSUPPORTED, "at most 65535 heads and 65535 windows");
  if (static_cast<long long>(plan->max_window_tokens) + n_text >= (1LL << 30))
    return fail(WSA_ERR_UNSUPPORTED, "segment too long");
  const void* ins[] = {q, k, v, q_txt, k_txt, v_txt, o, o_txt};
  for (const void* ptr : ins)
    if (!aligned16(ptr)) return fail(WSA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(WSA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = attention_text_workspace_bytes(*plan, n_text, heads, nullptr);
  if (workspace_bytes < need)
    return fail(WSA_ERR_INVALID_ARG, "workspace too small: need " + std::to_string(need) + " bytes");
  const size_t vb = static_cast<size_t>(plan->num_tokens) * heads * head_dim * 2;
  const size_t tb = static_cast<size_t>(n_text) * heads * head_dim * 2;
  const void* inv[] = {q, k, v};
  const void* int_[] = {q_txt, k_txt, v_txt};
  for (const void* ptr : inv)
    if (overlap(o, vb, ptr, vb) || overlap(o_txt, tb, ptr, vb) || overlap(workspace, need, ptr, vb))
      return fail(WSA_ERR_INVALID_ARG, "outputs or workspace overlap an input");
  for (const void* ptr : int_)
    if (overlap(o, vb, ptr, tb) || overlap(o_txt, tb, ptr, tb) || overlap(workspace, need, ptr, tb))
      return fail(WSA_ERR_INVALID_ARG, "outputs or workspace overlap an input");
  if (overlap(o, vb, o_txt, tb) || overlap(workspace, need, o, vb) || overlap(workspace, need, o_txt, tb))
    return fail(WSA_ERR_INVALID_ARG, "outputs and workspace must not overlap");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_attention_text: cudaGetDevice");
  if (dev != plan->device) return fail(WSA_ERR_INVALID_ARG, "plan was created on another device");
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  plan->stream = static_cast<cudaStream_t>(stream);
  e = launch_attention_text_bf16_tc(*plan, q, k, v, o, q_txt, k_txt, v_txt, o_txt, n_text, heads,
                                    in_order_canonical == 1, scale, workspace, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wsa_attention_text: launch");
  return WSA_OK;
}

}  // extern "C"

namespace {

// Shared checks of wsa_rope and wsa_rope_text.  Outputs may alias their own
// input exactly (in place) but must not overlap anything else.
wsa_status check_rope(const void* q, const void* k, void* q_out, void* k_out, long long rows, int heads,
                      int head_dim, wsa_dtype dtype, int rope_dim, float theta, size_t* bytes) {
  if (!q || !q_out) return fail(WSA_ERR_INVALID_ARG, "q and q_out must be non-null");
  if ((k == nullptr) != (k_out == nullptr))
    return fail(WSA_ERR_INVALID_ARG, "k and k_out must both be set or both null");
  if (heads <= 0) return fail(WSA_ERR_INVALID_ARG, "heads must be > 0");
  if (dtype != WSA_BF16 && dtype != WSA_FP32) return fail(WSA_ERR_INVALID_ARG, "unknown dtype");
  if (head_dim != 64 && head_dim != 128) return fail(WSA_ERR_UNSUPPORTED, "rope supports head_dim 64 or 128");
  if (rope_dim <= 0 || rope_dim > head_dim) return fail(WSA_ERR_INVALID_ARG, "rope_dim must be in [1, head_dim]");
  if ((rope_dim / 3) % 2 != 0 || rope_dim / 3 < 2)
    return fail(WSA_ERR_UNSUPPORTED, "rope_dim / 3 (channels per axis) must be even and >= 2");
  if (!std::isfinite(theta)) return fail(WSA_ERR_INVALID_ARG, "theta is not finite");
  if (!aligned16(q) || !aligned16(q_out) || (k && (!aligned16(k) || !aligned16(k_out))))
    return fail(WSA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const size_t b = static_cast<size_t>(rows) * heads * head_dim * (dtype == WSA_BF16 ? 2 : 4);
  auto bad = [&](const void* out, const void* in) { return out != in && overlap(out, b, in, b); };
  if (bad(q_out, q) || (k && (bad(q_out, k) || bad(k_out, k) || bad(k_out, q) || overlap(q_out, b, k_out, b))))
    return fail(WSA_ERR_INVALID_ARG, "an output overlaps another tensor (only exact in-place is allowed)");
  *bytes = b;
  return WSA_OK;
}

}  // namespace

extern "C" {

wsa_status wsa_rope(wsa_plan_t plan, const void* q, const void* k, void* q_out, void* k_out, int heads,
                    int head_dim, wsa_dtype dtype, int in_order_canonical, int text_len, int rope_dim, float theta,
                    void* stream) {
  if (!plan) return fail(WSA_ERR_INVALID_ARG, "plan is null");
  if (in_order_canonical != 0 && in_order_canonical != 1)
    return fail(WSA_ERR_INVALID_ARG, "in_order_canonical must be 0 or 1");
  if (text_len < 0 || text_len > (1 << 20)) return fail(WSA_ERR_INVALID_ARG, "text_len must be in [0, 2^20]");
  size_t bytes = 0;
  wsa_status st = check_rope(q, k, q_out, k_out, plan->num_tokens, heads, head_dim, dtype, rope_dim, theta, &bytes);
  if (st != WSA_OK) return st;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_rope: cudaGetDevice");
  if (dev != plan->device) return fail(WSA_ERR_INVALID_ARG, "plan was created on another device");
  const void* x[2] = {q, k};
  void* y[2] = {q_out, k_out};
  plan->stream = static_cast<cudaStream_t>(stream);
  e = launch_rope(plan, in_order_canonical == 1, x, y, k ? 2 : 1, plan->num_tokens, heads, head_dim,
                  dtype == WSA_BF16, text_len, rope_dim, theta > 0.f ? theta : 10000.0,
                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wsa_rope: launch");
  return WSA_OK;
}

wsa_status wsa_rope_text(const void* q_txt, const void* k_txt, void* q_out, void* k_out, int n_text, int heads,
                         int head_dim, wsa_dtype dtype, int rope_dim, float theta, void* stream) {
  if (n_text < 0 || n_text > (1 << 20)) return fail(WSA_ERR_INVALID_ARG, "n_text must be in [0, 2^20]");
  size_t bytes = 0;
  wsa_status st = check_rope(q_txt, k_txt, q_out, k_out, n_text, heads, head_dim, dtype, rope_dim, theta, &bytes);
  if (st != WSA_OK) return st;
  const void* x[2] = {q_txt, k_txt};
  void* y[2] = {q_out, k_out};
  cudaError_t e = launch_rope(nullptr, false, x, y, k_txt ? 2 : 1, n_text, heads, head_dim, dtype == WSA_BF16, 0,
                              rope_dim, theta > 0.f ? theta : 10000.0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wsa_rope_text: launch");
  return WSA_OK;
}

wsa_status wsa_transition(wsa_plan_t src, wsa_plan_t dst, const void* x_src, void* x_dst, int channels,
                          wsa_dtype dtype, void* stream) {
  if (!src || !dst) return fail(WSA_ERR_INVALID_ARG, "plans must be non-null");
  if (!x_src || !x_dst) return fail(WSA_ERR_INVALID_ARG, "x_src and x_dst must be non-null");
  if (channels <= 0) return fail(WSA_ERR_INVALID_ARG, "channels must be > 0");
  if (dtype != WSA_BF16 && dtype != WSA_FP32) return fail(WSA_ERR_INVALID_ARG, "unknown dtype");
  if (src->T != dst->T || src->H != dst->H || src->W != dst->W)
    return fail(WSA_ERR_MISMATCH, "plans describe different grids");
  if (src->device != dst->device) return fail(WSA_ERR_INVALID_ARG, "plans live on different devices");
  const size_t elt = dtype == WSA_BF16 ? 2 : 4;
  const size_t row_bytes = static_cast<size_t>(channels) * elt;
  const size_t bytes = row_bytes * static_cast<size_t>(src->num_tokens);
  if (reinterpret_cast<uintptr_t>(x_src) % elt || reinterpret_cast<uintptr_t>(x_dst) % elt)
    return fail(WSA_ERR_INVALID_ARG, "x_src and x_dst must be aligned to the element size");
  if (overlap(x_src, bytes, x_dst, bytes)) return fail(WSA_ERR_INVALID_ARG, "x_src and x_dst overlap");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "wsa_transition: cudaGetDevice");
  if (dev != src->device) return fail(WSA_ERR_INVALID_ARG, "plans were created on another device");
  src->stream = dst->stream = static_cast<cudaStream_t>(stream);
  e = launch_transition(*src, *dst, x_src, x_dst, row_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wsa_transition: launch");
  return WSA_OK;
}

wsa_status wsa_ensure_layout(wsa_plan_t current, wsa_plan_t required, const void* x, void* x_out, int channels,
                             wsa_dtype dtype, void* stream, int* moved) {
  if (!current || !required || !moved) return fail(WSA_ERR_INVALID_ARG, "plans and moved must be non-null");
  *moved = 0;
  if (current->T != required->T || current->H != required->H || current->W != required->W)
    return fail(WSA_ERR_MISMATCH, "plans describe different grids");
  // The windows of a plan follow from the grid, the window size and the
  // layout, so equal triples mean identical packed orders.
  if (current->layout == required->layout && current->wt == required->wt && current->wh == required->wh &&
      current->ww == required->ww)
    return WSA_OK;
  if (!x_out) return fail(WSA_ERR_INVALID_ARG, "the layouts differ: x_out must be given");
  const wsa_status st = wsa_transition(current, required, x, x_out, channels, dtype, stream);
  if (st == WSA_OK) *moved = 1;
  return st;
}

}  // extern "C"
