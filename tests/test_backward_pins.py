"""Pins of the backward oracle (oracle/backward.py) to facts outside itself:
central finite differences of the forward oracle (the C statement of
eq. 33.2), fp64 autograd of a separately written dense formulation, the
row-sum identity of Exercise 33.4 and the shift invariance it implies, and
closed-form special cases ("Chapter 33: inference compute optimisation",
eqs. 33.6–33.8)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import backward as bwd


def tiny_case(seed=0, G=2, bias=True):
    rng = np.random.default_rng(seed)
    B, Hkv, Tq, Tmax, d = 2, 2, 4, 6, 4
    Hq = Hkv * G
    q = rng.standard_normal((B, Hq, Tq, d))
    k = rng.standard_normal((B, Hkv, Tmax, d))
    v = rng.standard_normal((B, Hkv, Tmax, d))
    go = rng.standard_normal((B, Hq, Tq, d))
    seqlens = np.array([6, 4], dtype=np.int32)
    # pos < 0 (an empty row), 0 (one key), middle, beyond the length
    qpos = np.array([[-1, 0, 3, 5], [2, 1, 9, 3]], dtype=np.int32)
    M = None
    if bias:
        M = rng.standard_normal((B, Hq, Tq, Tmax))
        M[rng.random(M.shape) < 0.25] = -np.inf
        M[1, 0, 3, :] = -np.inf  # one more fully masked row
    return dict(q=q, k=k, v=v, go=go, seqlens=seqlens, qpos=qpos, bias=M, scale=0.7)


def loss(c, q=None, k=None, v=None):
    """L = sum(G_O * O) with O from the C forward oracle."""
    q = c["q"] if q is None else q
    k = c["k"] if k is None else k
    v = c["v"] if v is None else v
    r = oracle.attention(q, k, v, c["seqlens"], c["qpos"], c["scale"], bias=c["bias"], window=c.get("window", 0))
    return float((r["out"].reshape(c["go"].shape) * c["go"]).sum())


@pytest.mark.parametrize("G,bias,window", [(1, False, 0), (2, True, 0), (3, True, 0), (2, False, 2), (1, True, 3)])
def test_gradients_match_finite_differences_of_the_forward_oracle(G, bias, window):
    c = tiny_case(seed=G + 7 * window, G=G, bias=bias)
    c["window"] = window
    g = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                               bias=c["bias"], window=window)
    h = 1e-6
    for name, key in (("dq", "q"), ("dk", "k"), ("dv", "v")):
        x = c[key]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            num[idx] = (loss(c, **{key: xp}) - loss(c, **{key: xm})) / (2 * h)
        np.testing.assert_allclose(g[name], num, rtol=1e-6, atol=1e-7, err_msg=name)


def test_forward_quantities_match_the_forward_oracle():
    c = tiny_case(seed=5, G=2)
    g = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                               bias=c["bias"])
    r = oracle.attention(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], bias=c["bias"])
    np.testing.assert_allclose(g["o"].reshape(r["out"].shape), r["out"], rtol=0, atol=1e-13)
    lse = g["lse"].reshape(-1)
    np.testing.assert_array_equal(np.isneginf(lse), r["n_visible"] == 0)
    live = r["n_visible"] > 0
    np.testing.assert_allclose(lse[live], r["lse"][live], rtol=0, atol=1e-13)


def dense_autograd(c):
    """Separate dense formulation: scores with a -inf-free mask, torch
    autograd in fp64."""
    q = torch.tensor(c["q"], requires_grad=True)
    k = torch.tensor(c["k"], requires_grad=True)
    v = torch.tensor(c["v"], requires_grad=True)
    B, Hq, Tq, d = q.shape
    Hkv, Tmax = k.shape[1], k.shape[2]
    G = Hq // Hkv
    kk = k.repeat_interleave(G, dim=1)
    vv = v.repeat_interleave(G, dim=1)
    j = torch.arange(Tmax)
    vis = (j[None, None, :] < torch.tensor(c["seqlens"], dtype=torch.int64)[:, None, None]) & \
          (j[None, None, :] <= torch.tensor(c["qpos"], dtype=torch.int64)[:, :, None])
    vis = vis[:, None].expand(B, Hq, Tq, Tmax)
    s = c["scale"] * q @ kk.transpose(-1, -2)
    if c["bias"] is not None:
        M = torch.tensor(c["bias"])
        vis = vis & ~torch.isneginf(M)
        s = s + torch.where(vis, M, torch.zeros_like(M))
    m = torch.where(vis, s, torch.full_like(s, -1e300)).amax(-1, keepdim=True).detach()
    w = torch.where(vis, torch.exp(torch.where(vis, s, m) - m), torch.zeros_like(s))
    ell = w.sum(-1, keepdim=True)
    o = (w / torch.where(ell > 0, ell, torch.ones_like(ell))) @ vv
    (o * torch.tensor(c["go"])).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gradients_match_fp64_autograd(seed):
    c = tiny_case(seed=10 + seed, G=2)
    rng = np.random.default_rng(seed)
    # a larger shape too: 3 query rows x 40 keys per head
    c2 = dict(c)
    c2["q"] = rng.standard_normal((1, 4, 3, 8)); c2["k"] = rng.standard_normal((1, 2, 40, 8))
    c2["v"] = rng.standard_normal((1, 2, 40, 8)); c2["go"] = rng.standard_normal((1, 4, 3, 8))
    c2["seqlens"] = np.array([37], dtype=np.int32); c2["qpos"] = np.array([[36, 20, 5]], dtype=np.int32)
    c2["bias"] = None
    for cc in (c, c2):
        g = bwd.attention_backward(cc["q"], cc["k"], cc["v"], cc["seqlens"], cc["qpos"], cc["scale"], cc["go"],
                                   bias=cc["bias"])
        dq, dk, dv = dense_autograd(cc)
        np.testing.assert_allclose(g["dq"], dq, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dk"], dk, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dv"], dv, rtol=1e-12, atol=1e-13)


def test_row_sum_identity_and_shift_invariance():
    """Exercise 33.4: sum_k P_ik (G_P)_ik = g_o . o for every row, and the
    gradient along a common shift of a row's scores is zero, so the key
    gradients of each KV head sum to zero: sum_j G_K[j] = scale sum_i q_i
    sum_j (G_S)_ij = 0."""
    for seed in range(4):
        c = tiny_case(seed=20 + seed, G=2)
        g = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                                   bias=c["bias"])
        np.testing.assert_allclose(g["D"], (c["go"] * g["o"]).sum(-1), rtol=0, atol=1e-13)
        np.testing.assert_allclose(g["dk"].sum(axis=2), 0.0, atol=1e-13)


def test_special_cases():
    c = tiny_case(seed=7, G=2, bias=False)
    g = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"])
    # a row with one visible key (pos = 0): softmax is constant, no score gradient
    np.testing.assert_array_equal(g["dq"][0, :, 1], 0.0)
    # the empty row (pos < 0): nothing
    np.testing.assert_array_equal(g["dq"][0, :, 0], 0.0)
    # keys never visible (beyond the length of sequence 1) take no gradient
    np.testing.assert_array_equal(g["dk"][1, :, 4:], 0.0)
    np.testing.assert_array_equal(g["dv"][1, :, 4:], 0.0)
    # equal value rows: G_P is constant along each row, so G_S = 0
    c2 = dict(c)
    c2["v"] = np.broadcast_to(c["v"][:, :, :1], c["v"].shape).copy()
    g2 = bwd.attention_backward(c2["q"], c2["k"], c2["v"], c2["seqlens"], c2["qpos"], c2["scale"], c2["go"])
    np.testing.assert_allclose(g2["dq"], 0.0, atol=1e-14)
    np.testing.assert_allclose(g2["dk"], 0.0, atol=1e-14)
    assert np.abs(g2["dv"]).max() > 0.1
    # equal scores (q = 0): P uniform over the n visible keys, so
    # G_V[j] = sum over the rows that see j of G_O[i] / n_i
    c3 = dict(c)
    c3["q"] = np.zeros_like(c["q"])
    g3 = bwd.attention_backward(c3["q"], c3["k"], c3["v"], c3["seqlens"], c3["qpos"], c3["scale"], c3["go"])
    B, Hq, Tq, d = c["q"].shape
    G = Hq // c["k"].shape[1]
    want = np.zeros_like(c["v"])
    for b in range(B):
        for h in range(Hq):
            for i in range(Tq):
                n = min(int(c["qpos"][b, i]) + 1, int(c["seqlens"][b]))
                for j in range(max(n, 0)):
                    want[b, h // G, j] += c["go"][b, h, i] / n
    np.testing.assert_allclose(g3["dv"], want, rtol=1e-13, atol=1e-14)


def test_units_select_kv_heads():
    c = tiny_case(seed=9, G=2)
    full = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                                  bias=c["bias"])
    part = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                                  bias=c["bias"], units=[(1, 0)])
    np.testing.assert_array_equal(part["dk"][1, 0], full["dk"][1, 0])
    np.testing.assert_array_equal(part["dq"][1, 0:2], full["dq"][1, 0:2])
    assert not part["dk"][0].any() and not part["dq"][1, 2:].any()


def test_error_scales_dominate_the_gradients():
    """The error scales are sums of the absolute values of the terms each
    gradient adds up, so they bound the gradients (triangle inequality)."""
    c = tiny_case(seed=11, G=2)
    g = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                               bias=c["bias"])
    for name in ("dq", "dk", "dv"):
        assert np.all(g[name + "_abs"] >= 0)
        assert np.all(np.abs(g[name]) <= g[name + "_abs"] + 1e-12)


def test_window_gradients_match_fp64_autograd():
    """Sliding window (keys pos - W < j <= pos): the dense autograd
    formulation with the window folded into its bias as -inf."""
    c = tiny_case(seed=31, G=2, bias=False)
    W = 2
    B, Hq, Tq, d = c["q"].shape
    Tmax = c["k"].shape[2]
    j = np.arange(Tmax)
    M = np.where(j[None, None, :] > c["qpos"][:, :, None] - W, 0.0, -np.inf)[:, None].repeat(Hq, axis=1)
    dense = dict(c, bias=M)
    dq, dk, dv = dense_autograd(dense)
    g = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"], window=W)
    np.testing.assert_allclose(g["dq"], dq, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dk"], dk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dv"], dv, rtol=1e-12, atol=1e-13)
    # W = 1: one visible key per row, so no score gradient at all
    g1 = bwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"], window=1)
    np.testing.assert_array_equal(g1["dq"], 0.0)
    np.testing.assert_array_equal(g1["dk"], 0.0)
