"""Window-aligned sequence parallelism, Plan A (binding of wsa_sp_* and the
exchange built on wsa_gather_rows).

"Window-Aligned Sequence Parallelism (SeedVR2)", sections "Planner" and
"Plan A redistribution".  Each rank holds whole windows (LPT on token
counts) in rank-local order.  At a layout boundary, rank r sends row r of
the global count matrix and receives column r.  Every peer segment is
packed in destination-local order, and one argsort puts the received rows
in place.

The library's host planner produces the schedule.  On the device, a
boundary is one ``wsa_gather_rows`` pack, one variable-split
``all_to_all_single`` and one ``wsa_gather_rows`` unpack.  If no row changes
rank, it is a single gather through the composed index (the
local-permutation fast path, which includes the one-rank case).
"""

import ctypes

import numpy as np
import torch
import torch.distributed as dist

from . import WsaError, _check, gather_rows, lib


def owners(T, H, W, nt, nh, nw, layout, ranks, max_temporal=30):
    """owner[w]: the rank holding window w of ``layout`` (host only)."""
    n = ctypes.c_int()
    _check(lib.wsa_sp_owners(T, H, W, nt, nh, nw, layout, max_temporal, ranks, None, 0, ctypes.byref(n)))
    out = np.zeros(n.value, dtype=np.int32)
    _check(lib.wsa_sp_owners(T, H, W, nt, nh, nw, layout, max_temporal, ranks,
                             out.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n.value, ctypes.byref(n)))
    return out


def local_rows(T, H, W, nt, nh, nw, layout, ranks, rank, max_temporal=30):
    """Canonical ids held by ``rank`` in ``layout``, in rank-local order (host only)."""
    n = ctypes.c_int()
    _check(lib.wsa_sp_local_rows(T, H, W, nt, nh, nw, layout, max_temporal, ranks, rank, None, 0,
                                 ctypes.byref(n)))
    out = np.zeros(n.value, dtype=np.int32)
    _check(lib.wsa_sp_local_rows(T, H, W, nt, nh, nw, layout, max_temporal, ranks, rank,
                                 out.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n.value, ctypes.byref(n)))
    return out


class PlanA:
    """The Plan A exchange of one rank at the boundary src_layout -> dst_layout.

    Host attributes (from the library's planner): ``counts`` [ranks, ranks]
    (rows rank d needs from rank s at [s, d]), ``input_split_sizes`` (row
    ``rank``), ``output_split_sizes`` (column ``rank``), ``send_index``,
    ``recv_index`` and ``network_exchange_required``."""

    def __init__(self, T, H, W, nt, nh, nw, src_layout, dst_layout, ranks, rank, max_temporal=30):
        self.grid = (T, H, W, nt, nh, nw)
        self.src_layout, self.dst_layout = src_layout, dst_layout
        self.ranks, self.rank = ranks, rank
        counts = np.zeros((ranks, ranks), dtype=np.int64)
        n_send, n_recv, cross = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        args = (T, H, W, nt, nh, nw, src_layout, dst_layout, max_temporal, ranks, rank)
        cp = counts.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong))
        _check(lib.wsa_sp_plan_a(*args, cp, None, 0, None, 0, None, 0, ctypes.byref(n_send), ctypes.byref(n_recv),
                                 ctypes.byref(cross)))
        self.send_index = np.zeros(n_send.value, dtype=np.int32)
        self.recv_index = np.zeros(n_recv.value, dtype=np.int32)
        # the fast path's composed index (filled by the planner when no row changes rank)
        self.local_index = np.zeros(0 if cross.value else n_recv.value, dtype=np.int32)
        ip = ctypes.POINTER(ctypes.c_int)
        _check(lib.wsa_sp_plan_a(*args, cp, self.send_index.ctypes.data_as(ip), n_send.value,
                                 self.recv_index.ctypes.data_as(ip), n_recv.value,
                                 self.local_index.ctypes.data_as(ip) if not cross.value else None,
                                 self.local_index.size, ctypes.byref(n_send), ctypes.byref(n_recv),
                                 ctypes.byref(cross)))
        self.counts = counts
        self.network_exchange_required = bool(cross.value)
        self.input_split_sizes = [int(c) for c in counts[rank]]
        self.output_split_sizes = [int(c) for c in counts[:, rank]]
        self.n_send, self.n_recv = n_send.value, n_recv.value
        self._dev = {}

    def device_tables(self, device):
        """(send_index, recv_index, local_index) as int32 tensors on ``device``;
        local_index is the planner's composed index of the fast path (empty
        when rows change rank)."""
        key = torch.device(device)
        if key not in self._dev:
            self._dev[key] = tuple(torch.from_numpy(a).to(key)
                                   for a in (self.send_index, self.recv_index, self.local_index))
        return self._dev[key]

    def pack(self, x_local, out=None, stream=None):
        """Send buffer: this rank's source rows, grouped by destination rank,
        each group in destination-local order."""
        self._check_rows(x_local, self.n_send)
        return gather_rows(x_local, self.device_tables(x_local.device)[0], out=out, stream=stream)

    def unpack(self, recv, out=None, stream=None):
        """Destination-local rows from the receive buffer (source segments in rank order)."""
        self._check_rows(recv, self.n_recv)
        return gather_rows(recv, self.device_tables(recv.device)[1], out=out, stream=stream)

    def exchange(self, x_local, group=None, out=None, stream=None):
        """The whole boundary for this rank: returns its rows in the destination
        layout's rank-local order.  Every rank of ``group`` must call it (the
        collective runs whenever any rank exchanges rows)."""
        self._check_rows(x_local, self.n_send)
        if not self.network_exchange_required:
            return gather_rows(x_local, self.device_tables(x_local.device)[2], out=out, stream=stream)
        send = self.pack(x_local, stream=stream)
        recv = torch.empty((self.n_recv, x_local.shape[1]), dtype=x_local.dtype, device=x_local.device)
        dist.all_to_all_single(recv, send, output_split_sizes=self.output_split_sizes,
                               input_split_sizes=self.input_split_sizes, group=group)
        return self.unpack(recv, out=out, stream=stream)

    @staticmethod
    def _check_rows(x, n):
        if x.dim() != 2 or x.shape[0] != n:
            raise WsaError(-1, f"expected [{n}, channels] rows, got {tuple(x.shape)}")


__all__ = ["owners", "local_rows", "PlanA", "plan_b", "crossover"]


def plan_b(T, H, W, nt, nh, nw, ranks, max_temporal=30):
    """wsa_sp_plan_b: Plan B halo-exchange counts for one regular/shifted
    layer pair (host only).  Returns a dict of numpy arrays: ``window_rank``
    (computing rank of every shifted window), ``halo_in``, ``halo_out``,
    ``tokens`` and ``work`` per rank."""
    n = ctypes.c_int()
    _check(lib.wsa_sp_plan_b(T, H, W, nt, nh, nw, max_temporal, ranks, None, 0, ctypes.byref(n),
                             None, None, None, None))
    wr = np.zeros(n.value, dtype=np.int32)
    arrs = {k: np.zeros(ranks, dtype=np.int64) for k in ("halo_in", "halo_out", "tokens")}
    work = np.zeros(ranks, dtype=np.float64)
    ll = ctypes.POINTER(ctypes.c_longlong)
    _check(lib.wsa_sp_plan_b(T, H, W, nt, nh, nw, max_temporal, ranks,
                             wr.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n.value, ctypes.byref(n),
                             arrs["halo_in"].ctypes.data_as(ll), arrs["halo_out"].ctypes.data_as(ll),
                             arrs["tokens"].ctypes.data_as(ll), work.ctypes.data_as(ctypes.POINTER(ctypes.c_double))))
    return {"window_rank": wr, "work": work, **arrs}


class _Crossover(ctypes.Structure):
    _fields_ = [("plan_a_bytes", ctypes.c_longlong), ("plan_a_max_rank_bytes", ctypes.c_longlong),
                ("plan_b_bytes", ctypes.c_longlong), ("plan_b_max_rank_bytes", ctypes.c_longlong),
                ("plan_a_shifted_imbalance", ctypes.c_double), ("plan_b_shifted_imbalance", ctypes.c_double),
                ("plan_a_shifted_ms_max_rank", ctypes.c_double), ("plan_b_shifted_ms_max_rank", ctypes.c_double),
                ("crossover_link_gbs", ctypes.c_double)]


def crossover(T, H, W, nt, nh, nw, ranks, channels, bytes_per_elem=2, max_temporal=30, shifted_ms=None):
    """wsa_sp_crossover: Plan A against Plan B for one regular + shifted
    layer pair (host only), as a dict of the library's figures.  With
    ``shifted_ms`` (the measured one-GPU shifted-layer time) it also holds
    each plan's busiest-rank attention time and ``crossover_link_gbs`` (None
    when Plan B never wins)."""
    c = _Crossover()
    _check(lib.wsa_sp_crossover(T, H, W, nt, nh, nw, max_temporal, ranks, channels, bytes_per_elem,
                                float(shifted_ms) if shifted_ms is not None else 0.0, ctypes.byref(c)))
    out = {"ranks": ranks}
    out.update({name: getattr(c, name) for name, _ in _Crossover._fields_[:6]})
    if shifted_ms is not None:
        out["plan_a_shifted_ms_max_rank"] = c.plan_a_shifted_ms_max_rank
        out["plan_b_shifted_ms_max_rank"] = c.plan_b_shifted_ms_max_rank
        out["crossover_link_gbs"] = c.crossover_link_gbs if c.crossover_link_gbs >= 0 else None
    return out


def _main():
    import argparse
    ap = argparse.ArgumentParser(description="Plan A / Plan B exchange comparison for one layer pair")
    ap.add_argument("grid", type=int, nargs=6, metavar=("T", "H", "W", "nt", "nh", "nw"))
    ap.add_argument("--channels", type=int, default=3072)
    ap.add_argument("--ranks", type=int, nargs="+", default=[2, 4, 8])
    ap.add_argument("--shifted-ms", type=float, default=None,
                    help="measured one-GPU time of the shifted attention layer (ms)")
    args = ap.parse_args()
    for r in args.ranks:
        c = crossover(*args.grid, r, args.channels, shifted_ms=args.shifted_ms)
        line = (f"ranks {r}: Plan A {c['plan_a_bytes'] / 1e6:.1f} MB (busiest rank "
                f"{c['plan_a_max_rank_bytes'] / 1e6:.1f}), Plan B {c['plan_b_bytes'] / 1e6:.1f} MB (busiest rank "
                f"{c['plan_b_max_rank_bytes'] / 1e6:.1f}); shifted-layer work imbalance A "
                f"{c['plan_a_shifted_imbalance']:.3f}, B {c['plan_b_shifted_imbalance']:.3f}")
        if args.shifted_ms is not None:
            x = c["crossover_link_gbs"]
            line += (f"; Plan B wins only on links slower than {x:.0f} GB/s" if x
                     else "; Plan B never wins (its busiest rank also moves more bytes)")
        print(line)


if __name__ == "__main__":
    _main()
