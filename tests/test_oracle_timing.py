"""The CPU-baseline timing harness (oracle/timing.py) on a tiny workload: its
worker processes run the oracle and the returned throughput accounts for every
finished step (CPU only)."""
from __future__ import annotations

import numpy as np

from oracle import timing
from ragged_attention_token_gb300 import workloads as W


def test_host_cores_is_positive():
    assert timing.host_cores() >= 1


def test_two_workers_time_the_oracle():
    case = W.make_tiny()
    keep = case.keep.numpy()
    q, k, v = (x.double().numpy() for x in (case.q, case.k, case.v))
    r = timing.time_pipeline(keep, q, k, v, 0.125, budget_s=0.2, workers=2, max_steps_per_worker=3)
    assert r["workers"] == 2
    assert 2 <= r["steps"] <= 6                          # every worker finished at least one step
    T = int((keep != 0).sum())
    assert np.isclose(r["tokens_per_s"], T * r["steps"] / r["window_s"], rtol=1e-9)
