"""blkattn_fwd_static_scratch: the entry point for callers that must not
allocate device memory at call time (a framework owning all device memory
through its own pool, a latency-critical loop that cannot take cudaMalloc's
synchronisation, a runtime that forbids allocation after start-up).

It must give blkattn_fwd's results, within the parity tolerances, on calls in
a row (the fixed scratch array is reused and keeps the previous call's
contents), and refuse problems whose split states exceed the array.
Collected last on purpose; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_blocked_attention_gb300 import blkattn, workloads
from exact_blocked_attention_gb300 import build as libbuild

pytestmark = pytest.mark.gpu

TOL_O, TOL_L = 2e-3, 1e-3  # the bf16 parity tolerances of the other GPU tests
# the array's last 256 KiB hold the per-unit counters; plans get the rest
PLAN_BYTES = blkattn.STATIC_SCRATCH_BYTES - 256 * 1024


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    blkattn.load()


def on_device(name):
    s = workloads.spec(name, small=True)
    inp = workloads.generate(s)
    return s, {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def both_paths(s, g):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = blkattn.debug_plan(s.B, s.Hq, s.Hkv, s.Tq, s.Tmax, s.d, torch.bfloat16, sms)
    assert plan["n_splits"] > 1, "the case must use the split scratch"
    assert 0 < plan["workspace_bytes"] <= PLAN_BYTES
    ref_o, ref_l = blkattn.attention(g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], g["bias"], g["scale"])
    out = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_l, float("nan"))
    blkattn.fwd_static_scratch(g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], g["bias"], g["scale"], out, lse)
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    return ref_o, ref_l, out, lse


def assert_close(ref_o, ref_l, out, lse):
    masked = torch.isneginf(ref_l)
    assert torch.equal(torch.isneginf(lse), masked)
    assert torch.all(out[masked] == 0)
    live = ~masked
    bound = TOL_O * (1 + ref_o[live].abs())
    assert torch.all((out[live] - ref_o[live]).abs() <= bound)
    assert torch.all((lse[live] - ref_l[live]).abs() <= TOL_L)


def test_static_scratch_matches_blkattn_fwd_on_consecutive_calls():
    # two different problems back to back: the second reuses the array the
    # first left behind
    for name in ("decode_gqa", "spec_verify", "decode_gqa"):
        s, g = on_device(name)
        assert_close(*both_paths(s, g))


def test_static_scratch_refuses_problems_beyond_its_size():
    # 32 packed query rows per KV head (8 grouped heads x 4 rows) for a batch
    # large enough that the per-CTA / per-unit states outgrow the static array
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hq, Hkv, Tq, d, Tmax = 64, 8, 4, 128, 256
    B = 16
    while True:
        plan = blkattn.debug_plan(B, Hq, Hkv, Tq, Tmax, d, torch.bfloat16, sms)
        if plan["n_splits"] > 1 and plan["workspace_bytes"] > blkattn.STATIC_SCRATCH_BYTES:
            break
        B *= 2
        assert B <= 1024, "no over-limit split plan found"
    g = torch.Generator().manual_seed(0)
    q = torch.randn(B, Hq, Tq, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, Hkv, Tmax, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, Hkv, Tmax, d, generator=g).to(torch.bfloat16).cuda()
    sl = torch.full((B,), Tmax, dtype=torch.int32).cuda()
    qp = torch.full((B, Tq), Tmax - 1, dtype=torch.int32).cuda()
    out = torch.full((B, Hq, Tq, d), 7.0, device="cuda")
    lse = torch.full((B, Hq, Tq), 7.0, device="cuda")
    with pytest.raises(blkattn.BlkattnError) as e:
        blkattn.fwd_static_scratch(q, k, v, sl, qp, None, d ** -0.5, out, lse)
    assert e.value.status == blkattn.ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)  # nothing was enqueued
    # the allocating entry point still serves it
    blkattn.fwd(q, k, v, sl, qp, None, d ** -0.5, out, lse)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()


def test_static_scratch_refuses_plans_in_the_counter_region():
    """A plan larger than the 15.75 MiB the split states may use, though not
    larger than the whole 16 MiB array, is refused too (the last 256 KiB hold
    the unit counters).  (The 65536-unit counter limit is never the binding
    one: that many units need more than 16 MiB of split states.)"""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hq, Hkv, Tq, d, Tmax = 32, 8, 1, 128, 256
    for B in range(1, 1025):
        plan = blkattn.debug_plan(B, Hq, Hkv, Tq, Tmax, d, torch.bfloat16, sms)
        if PLAN_BYTES < plan["workspace_bytes"] <= blkattn.STATIC_SCRATCH_BYTES:
            break
    else:
        pytest.fail("no plan between 15.75 and 16 MiB")
    assert plan["kernel"] == 3 and plan["n_splits"] > 1
    g = torch.Generator().manual_seed(1)
    q = torch.randn(B, Hq, Tq, d, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, Hkv, Tmax, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, Hkv, Tmax, d, generator=g).to(torch.bfloat16).cuda()
    sl = torch.full((B,), Tmax, dtype=torch.int32).cuda()
    qp = torch.full((B, Tq), Tmax - 1, dtype=torch.int32).cuda()
    out = torch.full((B, Hq, Tq, d), 7.0, device="cuda")
    lse = torch.full((B, Hq, Tq), 7.0, device="cuda")
    with pytest.raises(blkattn.BlkattnError) as e:
        blkattn.fwd_static_scratch(q, k, v, sl, qp, None, d ** -0.5, out, lse)
    assert e.value.status == blkattn.ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)  # nothing was enqueued
