"""Host checks of the work counts bench.py divides by (no GPU): the FLOPs of
the tensor-bound workloads, windowed or not, against closed forms, and the
algorithmic bytes of the windowed decode."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from exact_blocked_attention_gb300 import workloads  # noqa: E402


def test_causal_flops_closed_form():
    s = workloads.spec("prefill")
    inp = workloads.generate(s)
    T = s.Tq
    pairs = T * (T + 1) // 2  # row i sees keys 0..i
    assert bench.causal_flops(s, inp) == pairs * s.B * s.Hq * 4 * s.d


def test_window_flops_closed_form():
    s = workloads.spec("window_prefill")
    inp = workloads.generate(s)
    T, W = s.Tq, s.window
    pairs = sum(min(i + 1, W) for i in range(T))  # row i sees keys i-W+1..i
    assert bench.causal_flops(s, inp) == pairs * s.B * s.Hq * 4 * s.d
    assert bench.tensor_bound(s) and bench.tensor_bound(workloads.spec("prefill"))
    assert not bench.tensor_bound(workloads.spec("window_decode"))


def test_window_decode_bytes_count_only_the_window():
    s = workloads.spec("window_decode")
    inp = workloads.generate(s)
    lens = np.minimum(inp["seqlens"].numpy().astype(np.int64), s.Tmax)
    want = int(np.minimum(lens, s.window).sum()) * s.Hkv * s.d * 2 * 2
    assert workloads.kv_bytes(s, inp["seqlens"].numpy()) == want
    # a windowed prefill still reads every cache row (some row sees each key)
    sp = workloads.spec("window_prefill", small=True)
    ip = workloads.generate(sp)
    assert workloads.kv_bytes(sp, ip["seqlens"].numpy()) == sp.B * sp.Tq * sp.Hkv * sp.d * 2 * 2
