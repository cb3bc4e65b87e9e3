/*
 * wsa.h -- C ABI of the GB300 (sm_103a) window-attention library.
 *
 * NaDiT-style 3D window attention over a post-patch video token grid
 * (T, H, W) with alternating regular and shifted window layouts, as described
 * in the vllm-omni design note "Window-Aligned Sequence Parallelism (SeedVR2)".
 *
 * Conventions shared by every call
 * --------------------------------
 * - Plain C types only.  Device pointers are CUDA device addresses on the
 *   current device; host pointers are ordinary host memory.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every device call is asynchronous on that stream.
 * - The caller owns every tensor it passes.  A plan owns its device tables
 *   until wsa_plan_destroy().
 * - Argument errors are detected on the host before anything is launched; an
 *   argument error never leaves a partially written output.
 * - On failure a call returns a negative wsa_status and records a message that
 *   wsa_last_error() returns (per host thread).
 * - Non-finite inputs are not validated: they propagate as IEEE arithmetic
 *   does.
 * - Two builds export this same ABI.  libwsa.so is the product build.
 *   libwsa_checked.so (compiled with -DWSA_BOUNDS_CHECK) also range-checks on
 *   the device every row index it reads from a plan table before the index
 *   addresses memory: an out-of-range index skips its access (the row reads as
 *   zeros or is not written) and is reported by wsa_plan_device_status.  The
 *   checked build stands in for a memory checker; its results on valid
 *   tables are bit-identical to the product build's.
 */
#ifndef WSA_H_
#define WSA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct wsa_plan_s* wsa_plan_t; /* opaque; owned by the library */

typedef enum {
  WSA_OK = 0,
  WSA_ERR_INVALID_ARG = -1,  /* bad size, null pointer, misalignment */
  WSA_ERR_UNSUPPORTED = -2,  /* valid request this library does not implement */
  WSA_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
  WSA_ERR_OOM = -4,          /* device allocation failed */
  WSA_ERR_MISMATCH = -5,     /* plans of different grids */
  WSA_ERR_DEVICE_CHECK = -6  /* a kernel recorded an error word (see wsa_plan_device_status) */
} wsa_status;

typedef enum { WSA_BF16 = 0, WSA_FP32 = 1 } wsa_dtype;
typedef enum { WSA_REGULAR = 0, WSA_SHIFTED = 1 } wsa_layout;

/* Library ABI version (major*100 + minor). */
int wsa_version(void);

/* 1 in the bounds-checked build (libwsa_checked.so), 0 in libwsa.so. */
int wsa_bounds_checked(void);

/* Message of the last failed call on this host thread ("" if none). */
const char* wsa_last_error(void);

/*
 * wsa_window_size -- host only, needs no GPU.
 * Window size of "Window layouts": scale = sqrt(45*80/(H*W)),
 * wh = ceil(round(H*scale)/nh), ww = ceil(round(W*scale)/nw),
 * wt = ceil(min(T, max_temporal)/nt), round = round-half-to-even in fp64.
 * All of T,H,W,nt,nh,nw,max_temporal must be > 0 (max_temporal is 30 in the
 * note); a size that computes to 0 is WSA_ERR_INVALID_ARG.
 */
wsa_status wsa_window_size(int T, int H, int W, int nt, int nh, int nw,
                           int max_temporal, int* wt, int* wh, int* ww);

/*
 * wsa_layout_windows -- host only, needs no GPU.
 * Windows of one layout ("Window layouts": regular cuts at multiples of the
 * window size, shifted cuts moved by floor(w/2) and clipped to the grid, no
 * cyclic roll; an axis not longer than its window is not shifted; empty
 * intervals are dropped), enumerated w-outermost, t-innermost.
 * Writes *num_windows always; if dims != NULL and capacity >= *num_windows,
 * also writes dims[6*k .. 6*k+5] = (t0, t1, h0, h1, w0, w1) of window k
 * (half-open).  capacity too small with dims != NULL is WSA_ERR_INVALID_ARG.
 */
wsa_status wsa_layout_windows(int T, int H, int W, int nt, int nh, int nw,
                              wsa_layout layout, int max_temporal,
                              int* dims, int capacity, int* num_windows);

/*
 * wsa_plan_create -- builds one layout's plan on the current device.
 * Host: window size and cuts (as wsa_layout_windows), ragged window offsets
 * in the cu_seqlens convention (vLLM-Omni diffusion-runtime blog, section
 * 4.2: prefix sums from 0 to N), and the attention work lists.  Device: a
 * kernel writes ids[p] = canonical id (t*H + h)*W + w of packed position p
 * (windows in enumeration order, tokens row-major in (t, h, w) inside a
 * window -- "Window layouts") and pos[ids[p]] = p.
 * N = T*H*W must be < 2^31.  The plan allocates its tables stream-ordered
 * (cudaMallocAsync on `stream`, no device-wide synchronisation) and fills
 * them asynchronously on `stream`; work on another stream must be ordered
 * after that stream before it uses the plan.
 */
wsa_status wsa_plan_create(int T, int H, int W, int nt, int nh, int nw,
                           wsa_layout layout, int max_temporal, void* stream,
                           wsa_plan_t* out);

/*
 * Frees the plan and its device tables.  The tables are released
 * stream-ordered (cudaFreeAsync) on the stream of the plan's latest call --
 * its creation or the last launch that used it -- which must still exist;
 * work on other streams that uses the plan must be ordered before that
 * stream's release.  Does not synchronise the device.
 */
wsa_status wsa_plan_destroy(wsa_plan_t plan);

/* Sizes of a plan.  Any output pointer may be NULL. */
wsa_status wsa_plan_info(wsa_plan_t plan, int* num_windows, int* num_tokens,
                         int* max_window_tokens, int* wt, int* wh, int* ww,
                         int* layout);

/*
 * Device pointers to the plan's int32 tables, valid until wsa_plan_destroy:
 *   offsets [num_windows + 1], dims [num_windows * 6], ids [N], pos [N].
 * Read-only for the caller.  Any output pointer may be NULL.
 */
wsa_status wsa_plan_tables(wsa_plan_t plan, const int** offsets, const int** dims,
                           const int** ids, const int** pos);

/*
 * wsa_attention -- per-window softmax attention over all heads.
 * "Window-Aligned Sequence Parallelism (SeedVR2)", section "Motivation":
 * attention runs only inside each window; for window w and head h
 *     O[w,h] = softmax(Q[w,h] K[w,h]^T * softmax_scale) V[w,h]
 * with no mask inside a window and no term across windows.
 *
 * q, k, v, o: device, [N, heads, head_dim] contiguous (token-major, heads,
 *   then channels).  in_order_canonical = 1: row = canonical token id;
 *   0: row = packed position of the plan (what wsa_transition produces).
 *   The window gather and the output scatter go through the plan's ids table
 *   inside the kernel; no separate permutation pass runs.  With packed rows
 *   (bf16) a window's full 128-row tiles are plain strided blocks and arrive
 *   by TMA tile loads; its last partial tile is gathered with zero fill, so
 *   rows of another window never enter its tiles.  Both orders give
 *   bit-identical results.
 * dtype WSA_BF16: head_dim must be 128; tensor-core kernel (tcgen05, TMEM),
 *   fp32 accumulation and softmax, bf16 output; pointers 16-byte aligned.
 * dtype WSA_FP32: head_dim 64 or 128; fp32 CUDA-core kernel throughout.
 * softmax_scale <= 0 selects 1/sqrt(head_dim).
 * o must not alias q, k or v.  Calls that use the same plan must be ordered
 * on one stream (the plan holds the kernel's work counter).
 */
wsa_status wsa_attention(wsa_plan_t plan, const void* q, const void* k,
                         const void* v, void* o, int heads, int head_dim,
                         wsa_dtype dtype, int in_order_canonical,
                         float softmax_scale, void* stream);

/*
 * wsa_attention_text -- window attention over packed segments
 * [video window, replicated text] with the text output averaged over windows.
 * "Window-Aligned Sequence Parallelism (SeedVR2)", sections "SeedVR2
 * integration" (window attention is a packed call over [video window,
 * replicated text] segments) and "Text stream" (each window yields a text
 * output; the layer's text output is their sum divided by the global window
 * count, T = (sum_w T_w) / W, not a token-weighted mean).
 *
 * For window w and head h the segment is S_w = [video rows of w ; the n_text
 * text rows]; O_seg = softmax(Q_seg K_seg^T * scale) V_seg.  Video rows of O
 * go to `o` (layout of wsa_attention); text rows give T_w, and o_txt receives
 * (sum_w T_w) / W, summed in window order (deterministic).
 * q, k, v, o: [N, heads, 128] bf16 (canonical or packed rows as in
 * wsa_attention); q_txt, k_txt, v_txt, o_txt: [n_text, heads, 128] bf16.
 * workspace: device, 256-byte aligned, at least wsa_attention_text_workspace
 * bytes (the work list and W x n_text x heads x 128 fp32 partials); owned by
 * the caller, contents undefined after the call.  n_text > 0; bf16 and
 * head_dim 128 only (WSA_ERR_UNSUPPORTED otherwise); at most 65535 heads and
 * 65535 windows.  Outputs and workspace must not overlap inputs.
 */
wsa_status wsa_attention_text_workspace(wsa_plan_t plan, int n_text, int heads,
                                        int head_dim, wsa_dtype dtype, size_t* bytes);
wsa_status wsa_attention_text(wsa_plan_t plan, const void* q, const void* k,
                              const void* v, void* o, const void* q_txt,
                              const void* k_txt, const void* v_txt, void* o_txt,
                              int n_text, int heads, int head_dim, wsa_dtype dtype,
                              int in_order_canonical, float softmax_scale,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * wsa_transition -- the local-permutation layout change between layers.
 * "Window-Aligned Sequence Parallelism (SeedVR2)", sections "Motivation" and
 * "Plan A redistribution": with one rank a layout change is a permutation of
 * the activation rows.  x_src holds row p = token at packed position p of
 * `src`; x_dst receives row p = token at packed position p of `dst`, i.e.
 *     x_dst[p] = x_src[pos_src[ids_dst[p]]].
 * x_src, x_dst: device, [N, channels] contiguous of `dtype`, must not
 * overlap.  src and dst may be the same plan (plain copy).  Plans of
 * different grids: WSA_ERR_MISMATCH.  Bit-exact (pure data movement).
 * A table entry out of range at either level (possible only if a caller has
 * written into the plan tables) skips its row, which is left unwritten; the
 * bounds-checked build also reports it through wsa_plan_device_status(dst).
 */
wsa_status wsa_transition(wsa_plan_t src, wsa_plan_t dst, const void* x_src,
                          void* x_dst, int channels, wsa_dtype dtype, void* stream);

/*
 * wsa_ensure_layout -- brings the activations into the layout a layer needs.
 * "Window-Aligned Sequence Parallelism (SeedVR2)", section "Window layouts":
 * the number of layout transitions follows the model's actual layer
 * schedule; ensure_layout(current, required) derives each one before a layer
 * instead of assuming that layer l uses layout l % 2.
 *
 * x: device, [N, channels] of `dtype`, rows in the packed order of
 * `current`.  When `required` describes the same windows as `current` (same
 * grid, same window size, same layout) the rows are already in the required
 * order: nothing is launched and *moved = 0.  Otherwise the rows are
 * rearranged into x_out exactly as wsa_transition(current, required, x,
 * x_out, ...) does, and *moved = 1; the caller's activations then live in
 * x_out.  x_out may be null only when no transition is needed (the call
 * fails with WSA_ERR_INVALID_ARG otherwise).  Errors as wsa_transition.
 */
wsa_status wsa_ensure_layout(wsa_plan_t current, wsa_plan_t required, const void* x,
                             void* x_out, int channels, wsa_dtype dtype, void* stream,
                             int* moved);

/*
 * wsa_attention_noalloc -- the bf16 window attention of wsa_attention for
 * callers that cannot allocate device memory.  The pages have no counterpart:
 * this is a deployment convenience of this library.
 *
 * Some callers cannot call cudaMalloc: their device memory is owned by
 * another framework's pool, or their serving loop must not take the
 * device-wide synchronisation that cudaMalloc/cudaFree imply.  They cannot
 * create a plan, so this call takes the grid
 * (T, H, W, nt, nh, nw, layout, max_temporal as in wsa_plan_create) directly
 * and builds the plan tables itself in a fixed device array inside the
 * library, then runs the same tensor-core attention kernel.  It allocates no
 * device memory: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * q, k, v, o, heads, in_order_canonical, softmax_scale and stream as in
 * wsa_attention with dtype WSA_BF16 and head_dim 128 (fixed); at most 65535
 * heads (WSA_ERR_UNSUPPORTED beyond).
 *
 * Limits of the fixed array (about 4.4 MB, held by every GPU that loads the
 * library until the process exits): T*H*W <= 524288 tokens, at most 8192
 * windows and 16384 work items of 256 query rows; beyond them the call
 * returns WSA_ERR_UNSUPPORTED with a message naming the limit.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and keeps it for the life of the
 * process; make that first call before any stream capture, and make no call
 * after a reset of the device (cudaDeviceReset destroys the array).  Every
 * call reuses the same array and overwrites what the previous call left
 * there, so calls whose GPU work overlaps (other streams, other host
 * threads) race and must be ordered by the caller.  A device-side wait that
 * gives up records its code in the array instead of returning it:
 * wsa_noalloc_device_status reads it, and the next call clears it.
 */
wsa_status wsa_attention_noalloc(int T, int H, int W, int nt, int nh, int nw,
                                 wsa_layout layout, int max_temporal,
                                 const void* q, const void* k, const void* v,
                                 void* o, int heads, int in_order_canonical,
                                 float softmax_scale, void* stream);

/*
 * wsa_noalloc_device_status -- the device error words of the last
 * wsa_attention_noalloc call on the current device (no counterpart in the
 * pages, like the call it serves).  Synchronises the device, reads the error
 * word a kernel of that call recorded in the fixed array (a bounded wait that
 * gave up; in the bounds-checked build also an out-of-range table index),
 * clears it, and returns WSA_ERR_DEVICE_CHECK with the code in *code, or
 * WSA_OK with *code = 0.  The next wsa_attention_noalloc call clears the
 * words itself, so read them before it.  Allocates no device memory.
 */
wsa_status wsa_noalloc_device_status(int* code);

/*
 * wsa_rope -- window-local 3D rotary position embedding of Q and K.
 * "Window-Aligned Sequence Parallelism (SeedVR2)", section "Reference quirks
 * reproduced on purpose": RoPE positions are window-local.  A video token at
 * (dt, dh, dw) inside its window of `plan` takes the axial indices
 * (text_len + dt, dh, dw), and every window restarts at 0.  Only the first
 * 3 * (rope_dim // 3) channels of each head rotate (126 of 128 when
 * rope_dim = 128); the rest pass through.
 * Readings of what the note leaves open:
 *   - axis a of (t, h, w) owns channels [a*da, (a+1)*da), da = rope_dim / 3;
 *   - channels (2j, 2j+1) of an axis are rotation pair j, turned by
 *     pos_a * theta^(-2j/da): (x0, x1) -> (x0 c - x1 s, x0 s + x1 c);
 *   - theta <= 0 selects 10000.
 * q, k (inputs) and q_out, k_out (outputs): device, [N, heads, head_dim]
 *   contiguous of `dtype`, rows canonical (in_order_canonical = 1) or
 *   plan-packed (0), as in wsa_attention; 16-byte aligned.  k and k_out may
 *   both be NULL (rotate q only).  An output may be its own input (in place)
 *   but must not overlap anything else.
 * head_dim 64 or 128; 0 < rope_dim <= head_dim with rope_dim / 3 even
 *   (WSA_ERR_UNSUPPORTED otherwise); 0 <= text_len <= 2^20.
 * The rotation is computed in fp32 and rounded once to `dtype`.  The layout
 * fixes the positions, so Q and K are rotated for the layout the next
 * attention call uses.
 */
wsa_status wsa_rope(wsa_plan_t plan, const void* q, const void* k, void* q_out,
                    void* k_out, int heads, int head_dim, wsa_dtype dtype,
                    int in_order_canonical, int text_len, int rope_dim,
                    float theta, void* stream);

/*
 * wsa_rope_text -- the same rotation for the replicated text rows
 * [n_text, heads, head_dim].  Text token i takes the axial indices (i, i, i):
 * text occupies indices [0, text_len) of the first axis, which is why the
 * video's first index starts at text_len (reading of the same section).
 * Other arguments as in wsa_rope; n_text = 0 is a no-op.
 */
wsa_status wsa_rope_text(const void* q_txt, const void* k_txt, void* q_out,
                         void* k_out, int n_text, int heads, int head_dim,
                         wsa_dtype dtype, int rope_dim, float theta,
                         void* stream);

/*
 * Window-aligned sequence parallelism, Plan A ("Window-Aligned Sequence
 * Parallelism (SeedVR2)", sections "Planner" and "Plan A redistribution").
 * Whole windows are sharded over `ranks` ranks.  The LPT rule takes windows
 * by (-token count, window id) and gives each to the rank with the smallest
 * (assigned tokens, rank id).  A rank lists its windows in ascending id and
 * holds their rows (row-major in (t, h, w) inside a window) in that order;
 * this is its rank-local order.  The grid arguments are those of
 * wsa_plan_create.  These three calls run on the host only and need no GPU.
 * Each writes its counts always and fills an array only when the array is
 * non-NULL; a capacity smaller than the count is WSA_ERR_INVALID_ARG.
 *
 * wsa_sp_owners: owner[w] = rank holding window w of `layout`
 *   (num_windows entries).  ranks > 0.
 */
wsa_status wsa_sp_owners(int T, int H, int W, int nt, int nh, int nw,
                         wsa_layout layout, int max_temporal, int ranks,
                         int* owner, int capacity, int* num_windows);

/* wsa_sp_local_rows: ids[i] = canonical id of row i of `rank`'s rank-local
 * order in `layout` (*n_rows entries).  0 <= rank < ranks. */
wsa_status wsa_sp_local_rows(int T, int H, int W, int nt, int nh, int nw,
                             wsa_layout layout, int max_temporal, int ranks,
                             int rank, int* ids, int capacity, int* n_rows);

/*
 * wsa_sp_plan_a: the exchange of `rank` at the boundary src_layout ->
 * dst_layout.
 *   counts [ranks * ranks] (may be NULL): the global count matrix, with
 *     counts[s * ranks + d] the rows rank d needs from rank s.  Rank r's
 *     input split sizes are row r; its output split sizes are column r.
 *   send_index [*n_send]: send row i holds local source row send_index[i].
 *     Rows are grouped by destination rank, and within a group they are in
 *     the destination's rank-local order.
 *   recv_index [*n_recv]: destination-local row p is receive row
 *     recv_index[p], the argsort of the received rows' destination
 *     positions.  The receive buffer is the source ranks' segments
 *     concatenated in rank order.
 *   *network_exchange_required: 1 if any row changes rank.  It is computed
 *     from the global matrix, so every rank gets the same value.  When it is
 *     0, the exchange is the local permutation x[send_index[recv_index[p]]].
 *   local_index [*n_recv] (may be NULL): that composed index,
 *     local_index[p] = send_index[recv_index[p]], the one gather of the
 *     local-permutation fast path.  Written only when
 *     *network_exchange_required is 0 (then *n_send == *n_recv).
 * Every index table is int32 on the host; row counts fit in int.  A capacity
 * below the count it must hold is WSA_ERR_INVALID_ARG.
 */
wsa_status wsa_sp_plan_a(int T, int H, int W, int nt, int nh, int nw,
                         wsa_layout src_layout, wsa_layout dst_layout,
                         int max_temporal, int ranks, int rank,
                         long long* counts, int* send_index, int send_capacity,
                         int* recv_index, int recv_capacity, int* local_index,
                         int local_capacity, int* n_send, int* n_recv,
                         int* network_exchange_required);

/*
 * wsa_sp_plan_b -- host only: the counts of a Plan B halo exchange for one
 * regular/shifted layer pair, for the crossover evaluation against Plan A.
 * The note leaves Plan B to a follow-up ("Window-Aligned Sequence
 * Parallelism (SeedVR2)", section "Limitations"); this call reads it as:
 *   - hidden rows stay with the regular layout's LPT owners (as in
 *     wsa_sp_owners) for the whole network, so regular layers exchange
 *     nothing;
 *   - shifted window w is computed by the rank holding most of its rows
 *     (window_rank[w]; the lowest rank id on ties);
 *   - its other rows travel to that rank before the shifted layer (halo_in
 *     of the receiver, halo_out of each sender), and their outputs travel
 *     back after it (the same counts, mirrored).
 * Outputs (each may be NULL): window_rank [num_windows of the shifted
 * layout]; halo_in, halo_out, tokens (sum of n_w of the windows a rank
 * computes) and work (sum of n_w^2) [ranks each].  *num_windows is always
 * written.  A window_rank capacity below the count is WSA_ERR_INVALID_ARG.
 */
wsa_status wsa_sp_plan_b(int T, int H, int W, int nt, int nh, int nw,
                         int max_temporal, int ranks, int* window_rank,
                         int capacity, int* num_windows, long long* halo_in,
                         long long* halo_out, long long* tokens, double* work);

/*
 * wsa_sp_crossover -- host only: Plan A against Plan B for one regular +
 * shifted layer pair, the crossover evaluation that the note leaves open
 * ("Window-Aligned Sequence Parallelism (SeedVR2)", section "Limitations";
 * Plan B read as in wsa_sp_plan_b).  Rows are hidden-state rows of
 * `channels` elements of `bytes_per_elem` bytes.
 *   plan_a_bytes: rows that change rank at the regular -> shifted and the
 *     shifted -> regular boundary (off-diagonal counts of both matrices);
 *   plan_a_max_rank_bytes: per boundary the busiest rank's rows sent or
 *     received (whichever is larger), summed over the two boundaries; it
 *     bounds the all-to-all time;
 *   plan_b_bytes, plan_b_max_rank_bytes: the halo rows in plus their outputs
 *     back (twice the halo counts), total and for the busiest rank;
 *   plan_*_shifted_imbalance: the shifted layer's attention work (sum of
 *     n_w^2) on the busiest rank over the mean, Plan A under its LPT owners,
 *     Plan B under its computing ranks.
 * With shifted_ms > 0, the measured one-GPU time of the shifted attention
 * layer, each plan's busiest-rank attention time is estimated as shifted_ms
 * times its share of the total sum of n_w^2 (plan_*_shifted_ms_max_rank), and
 * crossover_link_gbs is the link bandwidth below which Plan B's smaller
 * exchange outweighs its imbalance: the difference of the busiest ranks'
 * bytes over the difference of their attention times.  Fields that do not
 * apply (no shifted_ms, or Plan B never wins) are -1.
 */
typedef struct {
  long long plan_a_bytes;
  long long plan_a_max_rank_bytes;
  long long plan_b_bytes;
  long long plan_b_max_rank_bytes;
  double plan_a_shifted_imbalance;
  double plan_b_shifted_imbalance;
  double plan_a_shifted_ms_max_rank;
  double plan_b_shifted_ms_max_rank;
  double crossover_link_gbs;
} wsa_sp_crossover_t;

wsa_status wsa_sp_crossover(int T, int H, int W, int nt, int nh, int nw,
                            int max_temporal, int ranks, int channels,
                            int bytes_per_elem, double shifted_ms,
                            wsa_sp_crossover_t* out);

/*
 * wsa_gather_rows -- y[i] = x[index[i]] for 0 <= i < rows: the pack
 * (index = send_index) and unpack (index = recv_index) steps of the Plan A
 * exchange, on the device.
 * x: device, [x_rows, channels]; y: device, [rows, channels]; both of
 * `dtype` and contiguous; they must not overlap.  index: device int32 [rows].
 * An index outside [0, x_rows) leaves its row of y unwritten; it is not
 * reported.  rows == 0 is a no-op.  Bit-exact (pure data movement).
 */
wsa_status wsa_gather_rows(const void* x, int x_rows, const int* index, void* y,
                           int rows, int channels, wsa_dtype dtype, void* stream);

/*
 * wsa_debug_withhold_units -- test hook for the failure path of the
 * tensor-core attention kernel.  The pages have no counterpart: their
 * coordination waits are bounded and report typed failures ("Window-Aligned
 * Sequence Parallelism (SeedVR2)" and the runtime pages' failure handling),
 * and this hook lets a test make such a wait run out on a GPU without a
 * fault.  The next `launches` launches of that kernel (wsa_attention with
 * bf16, wsa_attention_text, wsa_attention_noalloc) hand out no work unit:
 * every role of the kernel waits for a unit that never comes, each wait gives
 * up after about one second, the kernel records the code of the first wait
 * that gave up in the plan's error word and returns without writing any
 * output, and wsa_plan_device_status then reports WSA_ERR_DEVICE_CHECK.
 * launches <= 0 turns the hook off.  Process-wide; a test uses it with no
 * other attention launch in flight.
 */
wsa_status wsa_debug_withhold_units(int launches);

/*
 * wsa_debug_fail_allocations -- test hook for the allocation failure path.
 * The pages have no counterpart: their runtimes classify failures into typed
 * errors, and this hook lets a test see this library's out-of-memory error
 * without exhausting a GPU.  The next `count` device allocations of
 * wsa_plan_create fail: the call returns WSA_ERR_OOM with a message naming
 * the hook and creates nothing.  count <= 0 turns the hook off.  Process-wide.
 */
wsa_status wsa_debug_fail_allocations(int count);

/*
 * Reads and clears the plan's device error words.  Synchronises the stream
 * of the plan's latest call (not the whole device): calls that use one plan
 * are ordered on one stream, so every launch that can have recorded an
 * error in it has finished.
 * *code = 0 when no kernel recorded an error; otherwise the code of the first
 * bounded wait that gave up or, in the bounds-checked build, 0x401 when a
 * kernel met a row index out of range in this plan's tables, and the call
 * returns WSA_ERR_DEVICE_CHECK.
 */
wsa_status wsa_plan_device_status(wsa_plan_t plan, int* code);

#ifdef __cplusplus
}
#endif

#endif /* WSA_H_ */
