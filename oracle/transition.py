"""Layout transition between two plans of the same grid.

"Window-Aligned Sequence Parallelism (SeedVR2)", sections "Motivation" and
"Plan A redistribution": with one rank the change from one layout to the next
is a local permutation of the activation rows.  Rows stored in the source
layout's packed order are rearranged into the destination layout's packed
order: destination row p holds canonical token ids_dst[p], which sits at
source row pos_src[ids_dst[p]].
"""

import numpy as np


def gather_table(plan_src, plan_dst):
    """g[p] = source row feeding destination row p."""
    if (plan_src.T, plan_src.H, plan_src.W) != (plan_dst.T, plan_dst.H, plan_dst.W):
        raise ValueError("plans describe different grids")
    return plan_src.pos.astype(np.int64)[plan_dst.ids.astype(np.int64)]


def transition(x_src, plan_src, plan_dst):
    """Return x_dst with x_dst[p] = x_src[g[p]] (rows of any width, any dtype)."""
    x_src = np.asarray(x_src)
    if x_src.shape[0] != plan_src.num_tokens:
        raise ValueError("row count does not match the plan")
    return x_src[gather_table(plan_src, plan_dst)]
