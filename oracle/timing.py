"""Timing of the CPU oracle on this host's cores (benchmark baseline only).

TEST INFRASTRUCTURE, like the rest of this package: only the benchmark's
CPU-baseline leg and its reference arm use this module.  It runs the oracle
as it stands, ``pipeline`` over the whole workload, in worker processes: one
worker per core, each repeating full steps of the same inputs (independent
replicas of the step, as the GPU side replays independent steps), with the
BLAS thread count pinned to one per worker.  Throughput is the kept tokens of
every finished step over the wall-clock window from the first worker's start
to the last worker's end.

Each worker is a fresh interpreter (``python -m oracle.timing``) that imports
numpy and the oracle only, and reads its inputs from a temporary .npz file.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def host_cores() -> int:
    """Cores this process may run on (its CPU affinity mask)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:   # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _worker(path: str, start_at: float, budget_s: float, max_steps: int) -> None:
    from oracle.ragged_attention import pipeline

    z = np.load(path)
    keep, q, k, v, scale = z["keep"], z["q"], z["k"], z["v"], float(z["scale"])
    pipeline(keep, q, k, v, scale)                 # warm: page in the code and the arrays
    while time.time() < start_at:
        time.sleep(0.001)
    t0 = time.time()
    steps = 0
    while steps < max_steps:
        pipeline(keep, q, k, v, scale)
        steps += 1
        if time.time() - t0 >= budget_s:
            break
    print(json.dumps({"steps": steps, "t0": t0, "t1": time.time()}), flush=True)


def time_pipeline(keep, q, k, v, scale: float, budget_s: float, workers: int,
                  max_steps_per_worker: int = 1 << 30) -> dict:
    """Run ``workers`` concurrent replicas of oracle.pipeline for about ``budget_s``
    seconds each; returns tokens/s over all of them and what was run."""
    keep = np.asarray(keep)
    T = int((keep != 0).sum())
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "inputs.npz")
        np.savez(path, keep=keep, q=np.asarray(q, dtype=np.float64), k=np.asarray(k, dtype=np.float64),
                 v=np.asarray(v, dtype=np.float64), scale=np.float64(scale))
        start_at = time.time() + 2.0 + 0.1 * workers
        cmd = [sys.executable, "-m", "oracle.timing", path, repr(start_at), repr(budget_s),
               str(max_steps_per_worker)]
        procs = [subprocess.Popen(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
                 for _ in range(workers)]
        rows = []
        for p in procs:
            out, err = p.communicate()
            if p.returncode != 0:
                raise RuntimeError(f"oracle timing worker failed ({p.returncode}): {err.strip()[-400:]}")
            rows.append(json.loads(out.strip().splitlines()[-1]))
    steps = sum(r["steps"] for r in rows)
    window = max(r["t1"] for r in rows) - min(r["t0"] for r in rows)
    return {"tokens_per_s": T * steps / window, "steps": steps, "window_s": window, "workers": workers,
            "kept_tokens_per_step": T}


if __name__ == "__main__":
    _worker(sys.argv[1], float(sys.argv[2]), float(sys.argv[3]), int(sys.argv[4]))
