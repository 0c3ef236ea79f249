"""Ring Attention across real ranks (torch.distributed over gloo, CPU), float64.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): used by the multi-rank tests to check
the ring's communication pattern and its failure behaviour on the host; the product library never
imports it.

Follows the page's "Ring Attention" section (Figure 3): every rank keeps its query block and
starts with its own KV block; at each of the P - 1 ring steps it passes the KV block it holds to
the next rank, receives the previous rank's, and updates its running output with the attention
of its queries over the block just received (here: the log-sum-exp merge of the two partials).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from .cp_attention import attention, lse_merge, to_f64


def _exchange(t: np.ndarray, dst: int, src: int) -> np.ndarray:
    """Send `t` to rank dst while receiving the array rank src sends (shape first, then data)."""
    shape_out = torch.tensor(list(t.shape), dtype=torch.int64)
    shape_in = torch.empty_like(shape_out)
    reqs = [dist.isend(shape_out, dst), dist.irecv(shape_in, src)]
    for r in reqs:
        r.wait()
    data_out = torch.from_numpy(np.ascontiguousarray(t))
    data_in = torch.empty(tuple(shape_in.tolist()), dtype=torch.float64)
    reqs = [dist.isend(data_out, dst), dist.irecv(data_in, src)]
    for r in reqs:
        r.wait()
    return data_in.numpy()


def ring_attention_ranks(q_local, k_local, v_local, scale: float | None = None):
    """This rank's O and LSE (float64) for its queries q_local [..., Sq_r, D] after P - 1 ring
    steps over the ranks' KV blocks k_local, v_local [..., Skv_r, D].  Raises if a peer
    disappears (the process group's timeout bounds every receive)."""
    world, rank = dist.get_world_size(), dist.get_rank()
    q = to_f64(q_local)
    k_cur, v_cur = to_f64(k_local), to_f64(v_local)
    o_run, lse_run = attention(q, k_cur, v_cur, scale)
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    for _ in range(world - 1):
        k_cur = _exchange(k_cur, nxt, prv)
        v_cur = _exchange(v_cur, nxt, prv)
        o_c, lse_c = attention(q, k_cur, v_cur, scale)
        o_run, lse_run = lse_merge(np.stack([o_run, o_c]), np.stack([lse_run, lse_c]))
    return o_run, lse_run
