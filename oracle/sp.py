"""Window-aligned sequence parallelism, Plan A redistribution (host logic).

"Window-Aligned Sequence Parallelism (SeedVR2)", sections "Planner" and
"Plan A redistribution":

* whole windows are assigned to ranks by the deterministic LPT rule
  (windows by (-token count, window id); each to the rank with the smallest
  (assigned tokens, rank id)); a rank lists its windows in ascending id and
  holds their tokens in window order -- its rank-local order;
* at a layout boundary, C[r, d] is the number of rows rank d needs from rank
  r; rank r's input split sizes are row r of C and its output split sizes are
  column r;
* each peer segment is packed in destination-local order, so the receiver
  reorders the concatenated segments with a single argsort of their
  destination positions;
* network_exchange_required is computed from the global count matrix, so
  every rank takes the same branch.
"""

import numpy as np

from .planner import lpt_assign


def owners(plan, ranks):
    """owner[w]: the rank holding window w (LPT on window token counts)."""
    owned, _ = lpt_assign(np.diff(plan.offsets).tolist(), ranks)
    owner = np.empty(plan.num_windows, dtype=np.int64)
    for r, ws in enumerate(owned):
        owner[ws] = r
    return owner


def local_rows(plan, ranks, rank, owner=None):
    """Canonical ids held by `rank`, in rank-local order."""
    owner = owners(plan, ranks) if owner is None else owner
    parts = [plan.ids[plan.offsets[w]:plan.offsets[w + 1]] for w in range(plan.num_windows) if owner[w] == rank]
    return np.concatenate(parts).astype(np.int64) if parts else np.zeros(0, dtype=np.int64)


def plan_a(src, dst, ranks):
    """Exchange schedule of every rank for the src -> dst layout change.

    Returns a dict with the global count matrix C [ranks, ranks] and, per
    rank r: send_index (local src row placed at each send position; segments
    by destination rank, each in destination-local order), recv_index (the
    single argsort that puts the received rows into dst-local order), and
    network_exchange_required."""
    own_s, own_d = owners(src, ranks), owners(dst, ranks)
    n = src.num_tokens
    # destination rank and destination-local position of every canonical id
    dest_rank = np.empty(n, dtype=np.int64)
    dest_pos = np.empty(n, dtype=np.int64)
    for d in range(ranks):
        rows = local_rows(dst, ranks, d, own_d)
        dest_rank[rows] = d
        dest_pos[rows] = np.arange(rows.size)
    src_rows = [local_rows(src, ranks, r, own_s) for r in range(ranks)]
    counts = np.zeros((ranks, ranks), dtype=np.int64)
    send_index, recv_positions = [], [[] for _ in range(ranks)]
    for r in range(ranks):
        ids = src_rows[r]
        order = []
        for d in range(ranks):
            sel = np.nonzero(dest_rank[ids] == d)[0]
            sel = sel[np.argsort(dest_pos[ids[sel]], kind="stable")]
            counts[r, d] = sel.size
            order.append(sel)
            recv_positions[d].append(dest_pos[ids[sel]])
        send_index.append(np.concatenate(order) if order else np.zeros(0, dtype=np.int64))
    recv_index = [np.argsort(np.concatenate(p), kind="stable") if p else np.zeros(0, dtype=np.int64)
                  for p in recv_positions]
    off_diag = counts.sum() - np.trace(counts)
    return {"counts": counts, "send_index": send_index, "recv_index": recv_index,
            "src_rows": src_rows, "dst_rows": [local_rows(dst, ranks, d, own_d) for d in range(ranks)],
            "network_exchange_required": bool(off_diag > 0)}


def simulate(x_canonical, src, dst, ranks):
    """Run the Plan A exchange among `ranks` simulated ranks on one host
    (each rank's rows in rank-local order); returns every rank's dst rows."""
    sched = plan_a(src, dst, ranks)
    x = np.asarray(x_canonical)
    local = [x[rows] for rows in sched["src_rows"]]
    send = [local[r][sched["send_index"][r]] for r in range(ranks)]
    bounds = [np.concatenate([[0], np.cumsum(sched["counts"][r])]) for r in range(ranks)]
    out = []
    for d in range(ranks):
        recv = np.concatenate([send[r][bounds[r][d]:bounds[r][d + 1]] for r in range(ranks)])
        out.append(recv[sched["recv_index"][d]])
    return out, sched


def plan_b(regular, shifted, ranks):
    """Plan B (halo exchange) counts for one regular/shifted layer pair.

    The pages name Plan B only as the follow-up to Plan A ("Limitations":
    Plan A re-shards the full activation at every boundary; a halo exchange
    needs its own crossover evaluation).  Reading used here:
    * hidden rows stay with the regular layout's LPT owners for the whole
      network, so regular layers exchange nothing;
    * shifted window w is computed by the rank that holds most of its rows
      (ties: lowest rank id); its other rows travel to that rank (halo in)
      and their attention outputs travel back to their owners (halo out).

    Returns a dict: owner of every shifted window, per-rank rows received
    (halo_in) and sent (halo_out) before a shifted layer (the return trip
    mirrors them), and per-rank shifted-layer work (sum of n_w and n_w^2)."""
    own_r = owners(regular, ranks)
    holder = np.empty(regular.num_tokens, dtype=np.int64)
    for w in range(regular.num_windows):
        holder[regular.ids[regular.offsets[w]:regular.offsets[w + 1]]] = own_r[w]
    comp = np.empty(shifted.num_windows, dtype=np.int64)
    halo_in = np.zeros(ranks, dtype=np.int64)
    halo_out = np.zeros(ranks, dtype=np.int64)
    tokens = np.zeros(ranks, dtype=np.int64)
    work = np.zeros(ranks, dtype=np.float64)
    for w in range(shifted.num_windows):
        rows = shifted.ids[shifted.offsets[w]:shifted.offsets[w + 1]]
        share = np.bincount(holder[rows], minlength=ranks)
        r = int(np.argmax(share))  # first maximum: lowest rank id on ties
        comp[w] = r
        n = rows.size
        halo_in[r] += n - share[r]
        halo_out += share
        halo_out[r] -= share[r]
        tokens[r] += n
        work[r] += float(n) * n
    return {"owner": comp, "halo_in": halo_in, "halo_out": halo_out, "tokens": tokens, "work": work}


def plan_a_rows_moved(src, dst, ranks):
    """Rows that change rank at one Plan A boundary (off-diagonal sum of C)."""
    c = plan_a(src, dst, ranks)["counts"]
    return int(c.sum() - np.trace(c))
