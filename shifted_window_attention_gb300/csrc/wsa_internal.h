// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "wsa.h"

namespace wsa {

// Records `msg` as this thread's last error and returns `st`.
wsa_status fail(wsa_status st, const std::string& msg);
// Maps a CUDA error to WSA_ERR_CUDA (or WSA_ERR_OOM) with context.
wsa_status cuda_fail(cudaError_t e, const char* what);
void clear_error();

// Number of SMs of the current device (cached per device).
int sm_count();

// One unit of attention work: query rows [q_start, q_start + span) of a window.
struct WorkItem {
  int window;
  int q_start;
};

// Host geometry of a layout (plan.cu): window size, window boxes
// (t0,t1,h0,h1,w0,w1 per window, enumeration order) and the attention work
// items of `rows` query rows in heaviest-first order.
wsa_status window_size(int T, int H, int W, int nt, int nh, int nw, int max_temporal, int* wt, int* wh,
                       int* ww);
void layout_boxes(int T, int H, int W, int wt, int wh, int ww, bool shifted, std::vector<int>* dims);
std::vector<WorkItem> make_items(const std::vector<int>& offsets, int rows, int tile);

// Words of the per-plan device workspace (int32 each).
enum WorkspaceWord {
  WS_NEXT_UNIT = 0,   // dynamic scheduler: next unit to hand out
  WS_DONE_CTAS = 1,   // CTAs that finished (the last one resets both counters)
  WS_ERROR = 2,       // first error code recorded by a kernel (0 = none)
  WS_BOUNDS = 3,      // bounds-checked builds: a table index was out of range
  WS_WORDS = 8
};

// Bounds-checked builds (compiled with -DWSA_BOUNDS_CHECK, libwsa_checked.so):
// every row index read from a plan table is range-checked on the device
// before it addresses memory.  An index out of range skips its access (the
// row reads as zeros or is not written) and records kErrBounds in the plan's
// WS_BOUNDS word, which wsa_plan_device_status reports; the kernel itself
// runs to completion.
#ifdef WSA_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif
constexpr int kErrBounds = 0x401;

// Query rows covered by one work item of each attention kernel.
constexpr int kTcItemRows = 256;    // tensor-core kernel: two 128-row tiles
constexpr int kSimtItemRows = 64;   // fp32 CUDA-core kernel

}  // namespace wsa

struct wsa_plan_s {
  int T = 0, H = 0, W = 0;
  int wt = 0, wh = 0, ww = 0;
  int layout = 0;
  int num_windows = 0;
  int num_tokens = 0;
  int max_window_tokens = 0;
  int device = 0;
  std::vector<int> h_offsets;  // [num_windows + 1]
  std::vector<int> h_dims;     // [num_windows * 6]
  int num_tc_items = 0;
  int num_simt_items = 0;
  // Stream of the plan's latest call (creation, then every launch that uses
  // the plan): its status read and its release are ordered on it.
  cudaStream_t stream = nullptr;
  // device memory: one allocation carved into the tables below
  void* d_block = nullptr;
  int* d_offsets = nullptr;
  int* d_dims = nullptr;
  int* d_ids = nullptr;
  int* d_pos = nullptr;
  wsa::WorkItem* d_tc_items = nullptr;
  wsa::WorkItem* d_simt_items = nullptr;
  int* d_work = nullptr;       // WS_WORDS int32, zero-initialised
};

namespace wsa {

// Launchers (asynchronous; arguments already validated by the ABI layer).
cudaError_t launch_plan_tables(const wsa_plan_s& p, cudaStream_t s);
cudaError_t launch_transition(const wsa_plan_s& src, const wsa_plan_s& dst, const void* x_src,
                              void* x_dst, size_t row_bytes, cudaStream_t s);
// Window-local 3D RoPE of one or two [n_rows, heads, head_dim] tensors (x[t]
// -> y[t], in place allowed).  plan != null: video rows of the plan (canonical
// or packed order); plan == null: text rows, token i at (i, i, i).
cudaError_t launch_rope(const wsa_plan_s* plan, bool canonical, const void* const x[2], void* const y[2],
                        int ntensors, int n_rows, int heads, int head_dim, bool bf16, int text_len, int rope_dim,
                        double theta, cudaStream_t s);
// y[i] = x[index[i]] for i < rows; rows whose index is outside [0, x_rows)
// are skipped.
cudaError_t launch_gather_rows(const void* x, int x_rows, const int* index, void* y, int rows, size_t row_bytes,
                               cudaStream_t s);
cudaError_t launch_attention_fp32(const wsa_plan_s& p, const float* q, const float* k,
                                  const float* v, float* o, int heads, int head_dim,
                                  bool canonical, float scale, cudaStream_t s);
cudaError_t launch_attention_bf16_tc(const wsa_plan_s& p, const void* q, const void* k,
                                     const void* v, void* o, int heads, bool canonical,
                                     float scale, cudaStream_t s);
// General form: optional text segment (n_text > 0, text tensors and fp32
// partial buffer) and an explicit work list.
cudaError_t launch_attention_tc(const wsa_plan_s& p, const void* q, const void* k, const void* v, void* o,
                                int heads, bool canonical, float scale, cudaStream_t s, const void* qt,
                                const void* kt, const void* vt, float* text_part, int n_text,
                                const WorkItem* items, int n_items);
// Failure-path test hook: the next `launches` tensor-core attention launches
// hand out no work unit (wsa_debug_withhold_units).
void withhold_attention_units(int launches);
// Workspace of the text form: its work list, then W x n_text x heads x 128
// fp32 partials.  *items_bytes (optional) receives the work-list part.
size_t attention_text_workspace_bytes(const wsa_plan_s& p, int n_text, int heads, size_t* items_bytes);
cudaError_t launch_attention_text_bf16_tc(const wsa_plan_s& p, const void* q, const void* k, const void* v,
                                          void* o, const void* qt, const void* kt, const void* vt, void* ot,
                                          int n_text, int heads, bool canonical, float scale,
                                          void* workspace, cudaStream_t s);

}  // namespace wsa
