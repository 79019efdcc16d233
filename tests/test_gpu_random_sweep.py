"""Randomised GPU parity sweep: seeded random problems across every kernel
path and visibility feature of the forward (dtype, head dim, grouping, row
count including prefill shapes, lengths, positions including negative and
beyond-length ones, bias, sliding window, token tree, output dtype) and of
the backward, each compared with the fp64 oracle under the same tolerances
as the targeted tests ("Chapter 33: inference compute optimisation" eqs.
33.2-33.8)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import backward as obwd
from exact_blocked_attention_gb300 import blkattn

pytestmark = pytest.mark.gpu

F32_TOL = 1e-5
BF16_TOL_O, BF16_TOL_L = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    blkattn.load()


def random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    dtype = "f32" if rng.random() < 0.2 else "bf16"
    d = 64 if rng.random() < 0.3 else 128
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    Hq = Hkv * G
    B = int(rng.integers(1, 4))
    Tq = int(rng.choice([1, 2, 3, 5, 8, 13, 64, 80]))
    Tmax = int(rng.integers(max(Tq, 1), 1400))
    lens = rng.integers(0, Tmax + 40, size=B)
    feature = rng.choice(["none", "bias", "window", "tree"], p=[0.4, 0.25, 0.2, 0.15])
    kind = rng.choice(["causal_tail", "random", "last"])
    qpos = np.zeros((B, Tq), dtype=np.int64)
    for b in range(B):
        ln = int(min(lens[b], Tmax))
        if kind == "causal_tail":
            qpos[b] = ln - Tq + np.arange(Tq)
        elif kind == "last":
            qpos[b] = ln - 1
        else:
            qpos[b] = rng.integers(-3, ln + 5, size=Tq)
    if feature == "tree":
        Tq = min(Tq, 64)
        qpos = np.repeat(np.minimum(lens, Tmax)[:, None] - 1, Tq, axis=1)
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    c = {"q": torch.randn(B, Hq, Tq, d, generator=g).to(dt),
         "k": torch.randn(B, Hkv, Tmax, d, generator=g).to(dt),
         "v": torch.randn(B, Hkv, Tmax, d, generator=g).to(dt),
         "seqlens": torch.tensor(lens, dtype=torch.int32),
         "qpos": torch.tensor(qpos, dtype=torch.int32), "bias": None, "tree": None, "window": 0,
         "scale": d ** -0.5, "dtype": dtype}
    if feature == "bias":
        heads = Hq if rng.random() < 0.5 else 1
        bias = torch.randn(B, heads, Tq, Tmax, generator=g)
        bias[torch.rand(B, heads, Tq, Tmax, generator=g) < 0.2] = -math.inf
        c["bias"] = bias
    elif feature == "window":
        c["window"] = int(rng.integers(1, Tmax + 10))
    elif feature == "tree":
        masks = []
        for b in range(B):
            row = []
            parents = [-1] + [int(rng.integers(0, k)) for k in range(1, Tq)]
            for i in range(Tq):
                m, node = 0, i
                while node >= 0:
                    m |= 1 << node
                    node = parents[node]
                row.append(m - (1 << 64) if m >= 1 << 63 else m)
            masks.append(row)
        c["tree"] = torch.tensor(masks, dtype=torch.int64)
    return c


@pytest.mark.parametrize("seed", range(500))
def test_random_forward(seed):
    c = random_case(seed)
    dev = lambda t: None if t is None else t.cuda()
    out_dtype = torch.bfloat16 if (c["dtype"] == "bf16" and seed % 5 == 0) else torch.float32
    out, lse = blkattn.attention(dev(c["q"]), dev(c["k"]), dev(c["v"]), dev(c["seqlens"]), dev(c["qpos"]),
                                 dev(c["bias"]), c["scale"], out_dtype=out_dtype, tree=dev(c["tree"]),
                                 window=c["window"])
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    ref = oracle.attention(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], bias=c["bias"],
                           tree=c["tree"], window=c["window"])
    d = c["q"].shape[-1]
    o = out.double().cpu().numpy().reshape(-1, d)
    l = lse.double().cpu().numpy().reshape(-1)
    masked = ref["n_visible"] == 0
    np.testing.assert_array_equal(np.isneginf(l), masked)
    assert np.all(o[masked] == 0.0)
    live = ~masked
    if live.any():
        tol_o, tol_l = (F32_TOL, F32_TOL) if c["dtype"] == "f32" else (BF16_TOL_O, BF16_TOL_L)
        ro = ref["out"][live]
        bound = tol_o * (1 + np.abs(ro))
        if out_dtype == torch.bfloat16:
            bound = bound + np.abs(ro) * 2.0 ** -8
        assert np.all(np.abs(o[live] - ro) <= bound)
        assert np.abs(l[live] - ref["lse"][live]).max() <= tol_l


def random_bwd_case(seed):
    rng = np.random.default_rng(5000 + seed)
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    Tq = int(rng.choice([1, 5, 64, 130, 257]))
    Tmax = int(rng.integers(Tq, Tq + 300))
    lens = rng.integers(max(1, Tq // 2), Tmax + 1, size=B)
    causal = rng.random() < 0.6
    qpos = np.zeros((B, Tq), dtype=np.int64)
    for b in range(B):
        qpos[b] = (lens[b] - Tq + np.arange(Tq)) if causal else rng.integers(-2, lens[b] + 3, size=Tq)
    g = torch.Generator().manual_seed(seed)
    c = {"q": torch.randn(B, Hkv * G, Tq, 128, generator=g).to(torch.bfloat16),
         "k": torch.randn(B, Hkv, Tmax, 128, generator=g).to(torch.bfloat16),
         "v": torch.randn(B, Hkv, Tmax, 128, generator=g).to(torch.bfloat16),
         "go": torch.randn(B, Hkv * G, Tq, 128, generator=g).to(torch.bfloat16),
         "seqlens": torch.tensor(lens, dtype=torch.int32), "qpos": torch.tensor(qpos, dtype=torch.int32),
         "bias": None, "scale": 128 ** -0.5}
    if rng.random() < 0.3:
        bias = torch.randn(B, 1, Tq, Tmax, generator=g)
        bias[torch.rand(B, 1, Tq, Tmax, generator=g) < 0.2] = -math.inf
        c["bias"] = bias
    c["window"] = int(rng.integers(1, Tmax + 20)) if rng.random() < 0.35 else 0
    return c


@pytest.mark.parametrize("seed", range(150))
def test_random_backward(seed):
    c = random_bwd_case(seed)
    ref = obwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                                  bias=c["bias"], window=c["window"])
    dev = lambda t: None if t is None else t.cuda()
    o = torch.from_numpy(ref["o"]).float()
    lse = torch.from_numpy(ref["lse"]).float()
    dq, dk, dv = blkattn.attention_backward(dev(c["q"]), dev(c["k"]), dev(c["v"]), dev(c["seqlens"]),
                                            dev(c["qpos"]), dev(o), dev(lse), dev(c["go"]),
                                            mask_bias=dev(c["bias"]), scale=c["scale"], window=c["window"])
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        got = t.double().cpu().numpy()
        scale_abs = ref[name + "_abs"]
        bound = 2.0 ** -7 * scale_abs + 1e-6 * max(float(scale_abs.max()), 1e-30)
        assert np.all(np.abs(got - ref[name]) <= bound), name
        np.testing.assert_array_equal(got[scale_abs == 0], 0.0)
