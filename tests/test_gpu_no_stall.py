"""Every decode route finishes in milliseconds on the benchmark workloads.

A pipeline wait that gives up, or an exit drain that waits on a phase the
barrier has already passed twice, costs at least a second per launch
without changing a single output (the drained exit keeps the results); the
parity tests cannot see that.  These tests time each route's call and bound
it far below one second, and check the status word stays clean."""
import pytest
import torch

import mla_decode_attention_04_gb300 as mla
from mla_decode_attention_04_gb300 import pipeline, workloads as wl

pytestmark = pytest.mark.gpu

BOUND_MS = 200.0  # the slowest route here takes about 1 ms; one stalled wait takes 1000 ms


def _time_ms(fn, reps=3):
    fn()
    torch.cuda.synchronize()
    worst = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        worst = max(worst, e0.elapsed_time(e1))
    return worst


ROUTES = [
    ("plain_decode_d1", "shards"), ("plain_decode_d2", "shards"), ("plain_decode_d2", "fused"),
    ("plain_decode_d2", "fp8"), ("mtp", "shards"), ("mtp", "fused"), ("mtp", "fp8"),
    ("long_context", "fused"), ("sparse_mixed", "shards"), ("sparse_mixed", "fused"),
]


@pytest.mark.parametrize("name,route", ROUTES, ids=[f"{n}-{r}" for n, r in ROUTES])
def test_route_has_no_stalled_wait(name, route):
    w = wl.NAMED[name](device="cuda")
    if route == "fp8":
        _, views = wl.fp8_cache(w, 0.25)
        step = pipeline.fused_step_for_workload(w, fp8_caches=views, kv_scale=0.25)
    elif route == "fused":
        step = pipeline.fused_step_for_workload(w)
    else:
        step = pipeline.step_for_workload(w)
    ms = _time_ms(step.run)
    rc, detail = mla.workspace_status(step.workspace)
    assert rc == mla.MLA_OK, f"device check {detail}"
    assert ms < BOUND_MS, f"{name} {route}: {ms:.1f} ms per step"
