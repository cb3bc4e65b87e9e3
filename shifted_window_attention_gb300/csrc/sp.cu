// Window-aligned sequence parallelism, Plan A: the host planner of the
// per-rank exchange at a layout boundary, and the row gather that packs and
// unpacks the exchanged rows on the device.
//
// "Window-Aligned Sequence Parallelism (SeedVR2)":
// - section "Planner": whole windows go to ranks by a deterministic LPT rule.
//   Windows are taken by (-token count, window id), and each goes to the rank
//   with the smallest (assigned tokens, rank id).  A rank lists its windows in
//   ascending id and holds their rows in window order (its rank-local order).
// - section "Plan A redistribution": C[r, d] counts the rows rank d needs
//   from rank r.  Rank r's input split sizes are row r of C and its output
//   split sizes are column r.  Each peer segment is packed in
//   destination-local order, and the receiver puts the concatenated segments
//   in order with one argsort of their destination positions.  Whether any
//   row crosses ranks is decided from the global C.
//
// Plan B (wsa_sp_plan_b) is the halo-exchange alternative that the note
// leaves to a separate crossover evaluation ("Limitations").  This library
// reads it as follows.  Hidden rows stay with the regular layout's owners,
// and each shifted window is computed by the rank holding most of its rows.
// The other rows travel to that rank before the shifted layer, and their
// outputs travel back after it.  The call returns the counts that the
// evaluation compares with Plan A.
//
// The planner needs no GPU and costs O(N) per call.  The receiver's argsort
// is computed by counting: the destination positions are distinct, so
// argsort[p] is the receive-buffer row that holds destination position p.
// That row is the segment of the row's source rank plus the number of earlier
// positions from the same source.

#include <algorithm>
#include <cstring>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "wsa_internal.h"

namespace wsa {
namespace {

struct Layout {
  int T = 0, H = 0, W = 0;
  long long N = 0;
  std::vector<int> dims;  // 6 per window, enumeration order
  int num_windows() const { return static_cast<int>(dims.size() / 6); }
  long long window_tokens(int w) const {
    const int* d = &dims[6 * w];
    return static_cast<long long>(d[1] - d[0]) * (d[3] - d[2]) * (d[5] - d[4]);
  }
  // canonical ids of window w, row-major in (t, h, w)
  template <typename F>
  void for_each_id(int win, F&& f) const {
    const int* d = &dims[6 * win];
    for (int t = d[0]; t < d[1]; ++t)
      for (int h = d[2]; h < d[3]; ++h) {
        const int base = (t * H + h) * W;
        for (int x = d[4]; x < d[5]; ++x) f(base + x);
      }
  }
};

wsa_status make_layout(int T, int H, int W, int nt, int nh, int nw, wsa_layout layout, int max_temporal,
                       Layout* out) {
  if (layout != WSA_REGULAR && layout != WSA_SHIFTED)
    return fail(WSA_ERR_INVALID_ARG, "layout must be WSA_REGULAR or WSA_SHIFTED");
  int wt, wh, ww;
  wsa_status st = window_size(T, H, W, nt, nh, nw, max_temporal, &wt, &wh, &ww);
  if (st != WSA_OK) return st;
  out->T = T;
  out->H = H;
  out->W = W;
  out->N = static_cast<long long>(T) * H * W;
  if (out->N >= (1LL << 31)) return fail(WSA_ERR_UNSUPPORTED, "T*H*W must be < 2^31");
  layout_boxes(T, H, W, wt, wh, ww, layout == WSA_SHIFTED, &out->dims);
  return WSA_OK;
}

// owner[w] under the LPT rule of the planner section.
std::vector<int> lpt_owner(const Layout& L, int ranks) {
  const int nwin = L.num_windows();
  std::vector<int> order(nwin);
  for (int w = 0; w < nwin; ++w) order[w] = w;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    const long long na = L.window_tokens(a), nb = L.window_tokens(b);
    return na != nb ? na > nb : a < b;
  });
  using Load = std::pair<long long, int>;  // (assigned tokens, rank): smallest first
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int r = 0; r < ranks; ++r) heap.push({0, r});
  std::vector<int> owner(nwin, 0);
  for (int w : order) {
    Load top = heap.top();
    heap.pop();
    owner[w] = top.second;
    top.first += L.window_tokens(w);
    heap.push(top);
  }
  return owner;
}

// rank_of[id] and local_of[id] (row index in the holder's rank-local order).
void assign_rows(const Layout& L, const std::vector<int>& owner, int ranks, std::vector<int>* rank_of,
                 std::vector<int>* local_of, std::vector<long long>* held) {
  rank_of->assign(static_cast<size_t>(L.N), 0);
  local_of->assign(static_cast<size_t>(L.N), 0);
  held->assign(ranks, 0);
  for (int w = 0; w < L.num_windows(); ++w) {
    const int r = owner[w];
    long long& cnt = (*held)[r];
    L.for_each_id(w, [&](int id) {
      (*rank_of)[id] = r;
      (*local_of)[id] = static_cast<int>(cnt++);
    });
  }
}

// C[s * ranks + d] = rows that rank d holds in the destination layout and
// rank s holds in the source layout.
std::vector<long long> count_matrix(const std::vector<int>& src_rank, const std::vector<int>& dst_rank, int ranks) {
  std::vector<long long> C(static_cast<size_t>(ranks) * ranks, 0);
  for (size_t id = 0; id < src_rank.size(); ++id) ++C[static_cast<size_t>(src_rank[id]) * ranks + dst_rank[id]];
  return C;
}

bool crosses(const std::vector<long long>& C, int ranks) {
  for (int s = 0; s < ranks; ++s)
    for (int d = 0; d < ranks; ++d)
      if (s != d && C[static_cast<size_t>(s) * ranks + d] != 0) return true;
  return false;
}

// Plan B under this library's reading: hidden rows stay with the regular
// layout's owners; shifted window w runs on the rank holding most of its
// rows (lowest id on ties), which receives the others (halo) and sends
// their outputs back.
struct PlanBCounts {
  std::vector<int> window_rank;
  std::vector<long long> halo_in, halo_out, tokens;
  std::vector<double> work;  // sum of n_w^2 of the windows a rank computes
};

PlanBCounts plan_b_counts(const Layout& R, const Layout& S, int ranks) {
  const std::vector<int> own = lpt_owner(R, ranks);
  std::vector<int> holder, unused;
  std::vector<long long> held;
  assign_rows(R, own, ranks, &holder, &unused, &held);
  PlanBCounts b;
  b.window_rank.assign(S.num_windows(), 0);
  b.halo_in.assign(ranks, 0);
  b.halo_out.assign(ranks, 0);
  b.tokens.assign(ranks, 0);
  b.work.assign(ranks, 0.0);
  std::vector<long long> share(ranks, 0);
  for (int w = 0; w < S.num_windows(); ++w) {
    std::fill(share.begin(), share.end(), 0);
    S.for_each_id(w, [&](int id) { ++share[holder[id]]; });
    int best = 0;  // the rank holding most rows; the lowest id on ties
    for (int r = 1; r < ranks; ++r)
      if (share[r] > share[best]) best = r;
    const long long n = S.window_tokens(w);
    b.halo_in[best] += n - share[best];
    for (int r = 0; r < ranks; ++r)
      if (r != best) b.halo_out[r] += share[r];
    b.tokens[best] += n;
    b.work[best] += static_cast<double>(n) * static_cast<double>(n);
    b.window_rank[w] = best;
  }
  return b;
}

wsa_status check_ranks(int ranks, int rank) {
  if (ranks <= 0) return fail(WSA_ERR_INVALID_ARG, "ranks must be > 0");
  if (rank < 0 || rank >= ranks) return fail(WSA_ERR_INVALID_ARG, "rank must be in [0, ranks)");
  return WSA_OK;
}

}  // namespace
}  // namespace wsa

using namespace wsa;

extern "C" {

wsa_status wsa_sp_owners(int T, int H, int W, int nt, int nh, int nw, wsa_layout layout, int max_temporal,
                         int ranks, int* owner, int capacity, int* num_windows) {
  if (!num_windows) return fail(WSA_ERR_INVALID_ARG, "num_windows is null");
  if (ranks <= 0) return fail(WSA_ERR_INVALID_ARG, "ranks must be > 0");
  Layout L;
  wsa_status st = make_layout(T, H, W, nt, nh, nw, layout, max_temporal, &L);
  if (st != WSA_OK) return st;
  *num_windows = L.num_windows();
  if (owner) {
    if (capacity < L.num_windows()) return fail(WSA_ERR_INVALID_ARG, "owner capacity is smaller than the window count");
    const std::vector<int> o = lpt_owner(L, ranks);
    std::memcpy(owner, o.data(), o.size() * sizeof(int));
  }
  return WSA_OK;
}

wsa_status wsa_sp_local_rows(int T, int H, int W, int nt, int nh, int nw, wsa_layout layout, int max_temporal,
                             int ranks, int rank, int* ids, int capacity, int* n_rows) {
  if (!n_rows) return fail(WSA_ERR_INVALID_ARG, "n_rows is null");
  wsa_status st = check_ranks(ranks, rank);
  if (st != WSA_OK) return st;
  Layout L;
  st = make_layout(T, H, W, nt, nh, nw, layout, max_temporal, &L);
  if (st != WSA_OK) return st;
  const std::vector<int> owner = lpt_owner(L, ranks);
  long long n = 0;
  for (int w = 0; w < L.num_windows(); ++w)
    if (owner[w] == rank) n += L.window_tokens(w);
  *n_rows = static_cast<int>(n);
  if (ids) {
    if (capacity < n) return fail(WSA_ERR_INVALID_ARG, "ids capacity is smaller than the rank's row count");
    long long k = 0;
    for (int w = 0; w < L.num_windows(); ++w)
      if (owner[w] == rank) L.for_each_id(w, [&](int id) { ids[k++] = id; });
  }
  return WSA_OK;
}

wsa_status wsa_sp_plan_a(int T, int H, int W, int nt, int nh, int nw, wsa_layout src_layout,
                         wsa_layout dst_layout, int max_temporal, int ranks, int rank, long long* counts,
                         int* send_index, int send_capacity, int* recv_index, int recv_capacity, int* local_index,
                         int local_capacity, int* n_send, int* n_recv, int* network_exchange_required) {
  if (!n_send || !n_recv || !network_exchange_required)
    return fail(WSA_ERR_INVALID_ARG, "n_send, n_recv and network_exchange_required must be non-null");
  wsa_status st = check_ranks(ranks, rank);
  if (st != WSA_OK) return st;
  Layout S, D;
  st = make_layout(T, H, W, nt, nh, nw, src_layout, max_temporal, &S);
  if (st != WSA_OK) return st;
  st = make_layout(T, H, W, nt, nh, nw, dst_layout, max_temporal, &D);
  if (st != WSA_OK) return st;
  const std::vector<int> own_s = lpt_owner(S, ranks), own_d = lpt_owner(D, ranks);
  std::vector<int> src_rank, src_local, dst_rank, dst_local;
  std::vector<long long> src_held, dst_held;
  assign_rows(S, own_s, ranks, &src_rank, &src_local, &src_held);
  assign_rows(D, own_d, ranks, &dst_rank, &dst_local, &dst_held);

  const std::vector<long long> C = count_matrix(src_rank, dst_rank, ranks);
  const bool cross = crosses(C, ranks);
  *network_exchange_required = cross ? 1 : 0;
  *n_send = static_cast<int>(src_held[rank]);
  *n_recv = static_cast<int>(dst_held[rank]);
  if (counts) std::memcpy(counts, C.data(), C.size() * sizeof(long long));
  if (send_index && send_capacity < *n_send)
    return fail(WSA_ERR_INVALID_ARG, "send_index capacity is smaller than the rank's source row count");
  if (recv_index && recv_capacity < *n_recv)
    return fail(WSA_ERR_INVALID_ARG, "recv_index capacity is smaller than the rank's destination row count");
  if (local_index && !cross && local_capacity < *n_recv)
    return fail(WSA_ERR_INVALID_ARG, "local_index capacity is smaller than the rank's destination row count");
  if (!send_index && !recv_index && !local_index) return WSA_OK;

  // segments by destination rank; inside one, destination-local order:
  // walk each destination rank's rows in its order, keep those held here
  std::vector<int> send(static_cast<size_t>(*n_send));
  {
    long long k = 0;
    for (int d = 0; d < ranks; ++d)
      for (int w = 0; w < D.num_windows(); ++w)
        if (own_d[w] == d)
          D.for_each_id(w, [&](int id) {
            if (src_rank[id] == rank) send[k++] = src_local[id];
          });
  }
  std::vector<int> recv(static_cast<size_t>(*n_recv));
  {
    std::vector<long long> next(ranks, 0);  // next receive row of each source segment
    for (int s = 1; s < ranks; ++s) next[s] = next[s - 1] + C[static_cast<size_t>(s - 1) * ranks + rank];
    long long p = 0;
    for (int w = 0; w < D.num_windows(); ++w)
      if (own_d[w] == rank) D.for_each_id(w, [&](int id) { recv[p++] = static_cast<int>(next[src_rank[id]]++); });
  }
  if (send_index) std::copy(send.begin(), send.end(), send_index);
  if (recv_index) std::copy(recv.begin(), recv.end(), recv_index);
  // No row changes rank: every receive row comes from this rank's own send
  // buffer, so the two gathers compose into one through send[recv[p]].
  if (local_index && !cross)
    for (size_t p = 0; p < recv.size(); ++p) local_index[p] = send[static_cast<size_t>(recv[p])];
  return WSA_OK;
}

wsa_status wsa_sp_plan_b(int T, int H, int W, int nt, int nh, int nw, int max_temporal, int ranks,
                         int* window_rank, int capacity, int* num_windows, long long* halo_in, long long* halo_out,
                         long long* tokens, double* work) {
  if (!num_windows) return fail(WSA_ERR_INVALID_ARG, "num_windows is null");
  if (ranks <= 0) return fail(WSA_ERR_INVALID_ARG, "ranks must be > 0");
  Layout R, S;
  wsa_status st = make_layout(T, H, W, nt, nh, nw, WSA_REGULAR, max_temporal, &R);
  if (st != WSA_OK) return st;
  st = make_layout(T, H, W, nt, nh, nw, WSA_SHIFTED, max_temporal, &S);
  if (st != WSA_OK) return st;
  *num_windows = S.num_windows();
  if (window_rank && capacity < S.num_windows())
    return fail(WSA_ERR_INVALID_ARG, "window_rank capacity is smaller than the shifted window count");
  const PlanBCounts b = plan_b_counts(R, S, ranks);
  if (window_rank) std::copy(b.window_rank.begin(), b.window_rank.end(), window_rank);
  for (int r = 0; r < ranks; ++r) {
    if (halo_in) halo_in[r] = b.halo_in[r];
    if (halo_out) halo_out[r] = b.halo_out[r];
    if (tokens) tokens[r] = b.tokens[r];
    if (work) work[r] = b.work[r];
  }
  return WSA_OK;
}

wsa_status wsa_sp_crossover(int T, int H, int W, int nt, int nh, int nw, int max_temporal, int ranks, int channels,
                            int bytes_per_elem, double shifted_ms, wsa_sp_crossover_t* out) {
  if (!out) return fail(WSA_ERR_INVALID_ARG, "out is null");
  if (ranks <= 0) return fail(WSA_ERR_INVALID_ARG, "ranks must be > 0");
  if (channels <= 0 || bytes_per_elem <= 0) return fail(WSA_ERR_INVALID_ARG, "channels and bytes_per_elem must be > 0");
  if (!(shifted_ms == shifted_ms)) return fail(WSA_ERR_INVALID_ARG, "shifted_ms is NaN");
  Layout R, S;
  wsa_status st = make_layout(T, H, W, nt, nh, nw, WSA_REGULAR, max_temporal, &R);
  if (st != WSA_OK) return st;
  st = make_layout(T, H, W, nt, nh, nw, WSA_SHIFTED, max_temporal, &S);
  if (st != WSA_OK) return st;
  const long long row = static_cast<long long>(channels) * bytes_per_elem;
  const std::vector<int> own_r = lpt_owner(R, ranks), own_s = lpt_owner(S, ranks);
  std::vector<int> rank_r, rank_s, local_unused;
  std::vector<long long> held_unused;
  assign_rows(R, own_r, ranks, &rank_r, &local_unused, &held_unused);
  assign_rows(S, own_s, ranks, &rank_s, &local_unused, &held_unused);
  // Plan A: the rows that change rank at the regular -> shifted and the
  // shifted -> regular boundary (off-diagonal counts); the busiest rank is
  // the larger of its rows sent and its rows received.
  long long a_rows = 0, a_max = 0;
  for (int dir = 0; dir < 2; ++dir) {
    const std::vector<long long> C = dir == 0 ? count_matrix(rank_r, rank_s, ranks) : count_matrix(rank_s, rank_r, ranks);
    long long busiest = 0;
    for (int r = 0; r < ranks; ++r) {
      long long sent = 0, recv = 0;
      for (int q = 0; q < ranks; ++q)
        if (q != r) {
          sent += C[static_cast<size_t>(r) * ranks + q];
          recv += C[static_cast<size_t>(q) * ranks + r];
        }
      a_rows += sent;
      busiest = std::max(busiest, std::max(sent, recv));
    }
    a_max += busiest;
  }
  // Plan B: halo rows in before the shifted layer and their outputs back after it.
  const PlanBCounts b = plan_b_counts(R, S, ranks);
  long long b_in = 0, b_busiest = 0;
  for (int r = 0; r < ranks; ++r) {
    b_in += b.halo_in[r];
    b_busiest = std::max(b_busiest, std::max(b.halo_in[r], b.halo_out[r]));
  }
  // shifted-layer attention work per rank: Plan A's LPT owners against Plan B's computing ranks
  std::vector<double> a_work(ranks, 0.0);
  double total = 0.0;
  for (int w = 0; w < S.num_windows(); ++w) {
    const double n = static_cast<double>(S.window_tokens(w));
    a_work[own_s[w]] += n * n;
    total += n * n;
  }
  const double a_peak = *std::max_element(a_work.begin(), a_work.end());
  const double b_peak = *std::max_element(b.work.begin(), b.work.end());
  const double mean = total / ranks;
  out->plan_a_bytes = a_rows * row;
  out->plan_a_max_rank_bytes = a_max * row;
  out->plan_b_bytes = 2 * b_in * row;
  out->plan_b_max_rank_bytes = 2 * b_busiest * row;
  out->plan_a_shifted_imbalance = mean > 0 ? a_peak / mean : 1.0;
  out->plan_b_shifted_imbalance = mean > 0 ? b_peak / mean : 1.0;
  out->plan_a_shifted_ms_max_rank = -1.0;
  out->plan_b_shifted_ms_max_rank = -1.0;
  out->crossover_link_gbs = -1.0;
  if (shifted_ms > 0 && total > 0) {
    // each plan's busiest-rank attention time as its share of the one-GPU time
    const double ta = shifted_ms * a_peak / total, tb = shifted_ms * b_peak / total;
    out->plan_a_shifted_ms_max_rank = ta;
    out->plan_b_shifted_ms_max_rank = tb;
    const double dbytes = static_cast<double>(out->plan_a_max_rank_bytes - out->plan_b_max_rank_bytes);
    if (tb > ta && dbytes > 0) out->crossover_link_gbs = dbytes / ((tb - ta) * 1e-3) / 1e9;
  }
  return WSA_OK;
}

wsa_status wsa_gather_rows(const void* x, int x_rows, const int* index, void* y, int rows, int channels,
                           wsa_dtype dtype, void* stream) {
  if (rows < 0 || x_rows < 0) return fail(WSA_ERR_INVALID_ARG, "rows and x_rows must be >= 0");
  if (channels <= 0) return fail(WSA_ERR_INVALID_ARG, "channels must be > 0");
  if (dtype != WSA_BF16 && dtype != WSA_FP32) return fail(WSA_ERR_INVALID_ARG, "unknown dtype");
  if (rows == 0) return WSA_OK;
  if (!x || !index || !y) return fail(WSA_ERR_INVALID_ARG, "x, index and y must be non-null");
  const size_t row_bytes = static_cast<size_t>(channels) * (dtype == WSA_BF16 ? 2 : 4);
  const auto a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(y);
  const size_t nx = row_bytes * static_cast<size_t>(x_rows), ny = row_bytes * static_cast<size_t>(rows);
  if (a < b + ny && b < a + nx) return fail(WSA_ERR_INVALID_ARG, "x and y must not overlap");
  cudaError_t e = launch_gather_rows(x, x_rows, index, y, rows, row_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wsa_gather_rows: launch");
  return WSA_OK;
}

}  // extern "C"
