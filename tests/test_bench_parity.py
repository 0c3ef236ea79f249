"""CPU check of the bench's oracle check on the timed step's output: a bf16 rounding of the exact
result passes, a wrong value or a wrong LSE fails."""
import importlib.util
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_bench_parity_decision():
    b = _bench()
    rng = np.random.default_rng(0)
    o_ref = rng.standard_normal((1, 2, 50, 16)) * 0.3
    lse_ref = rng.standard_normal((1, 2, 50)) * 3
    o_gpu = torch.from_numpy(o_ref).to(torch.bfloat16)
    l_gpu = torch.from_numpy(lse_ref).float()
    assert b._parity(o_ref, lse_ref, (o_gpu, l_gpu))["ok"]
    bad = o_gpu.clone()
    bad[0, 1, 7, 3] += 0.02
    assert not b._parity(o_ref, lse_ref, (bad, l_gpu))["ok"]
    assert not b._parity(o_ref, lse_ref, (o_gpu, l_gpu + 2e-3))["ok"]
    # the GPU copy may hold more rows than the oracle sample: only the common rows count
    more = torch.cat([o_gpu, torch.zeros(1, 2, 10, 16, dtype=torch.bfloat16)], dim=2)
    lmore = torch.cat([l_gpu, torch.zeros(1, 2, 10)], dim=2)
    r = b._parity(o_ref, lse_ref, (more, lmore))
    assert r["ok"] and r["rows_per_head"] == 50
