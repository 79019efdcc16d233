"""Pins for the fp64 oracle: values, closed forms and exact brute force that do
not come from the oracle itself.

Sources: "Chapter 33: inference compute optimisation" §33.2 (eqs. 33.2–33.5,
Example 25.1, Algorithm 33.1) and its workbook (Exercises 33.1–33.3);
"Generation and Caching with the Same Model" (logical-position alignment and
its incremental-cache check).  Each golden file under tests/golden/ names the
passage its numbers come from.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import states

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def run(q, k, v, seqlens, qpos, scale, bias=None, rows=None):
    return oracle.attention(np.asarray(q, np.float64), np.asarray(k, np.float64),
                            np.asarray(v, np.float64), np.asarray(seqlens, np.int32),
                            np.asarray(qpos, np.int32), scale, bias=bias, rows=rows)


# ---------------------------------------------------------------- Example 25.1

def test_example_25_1_block_states_and_merge():
    g = golden("example_25_1.json")
    z = np.log(np.array(g["scores_are_natural_logs_of"], dtype=np.float64))
    v = np.array(g["values"], dtype=np.float64)[:, None]
    a_idx, b_idx = g["blocks"]
    sa = states.block_state(z[a_idx], v[a_idx])
    sb = states.block_state(z[b_idx], v[b_idx])
    assert sa[0] == pytest.approx(math.log(g["state_A"]["m_is_log_of"]), abs=1e-15)
    assert sa[1] == pytest.approx(g["state_A"]["l"], abs=1e-15)
    assert sa[2][0] == pytest.approx(g["state_A"]["u"], abs=1e-15)
    assert sb[0] == pytest.approx(math.log(g["state_B"]["m_is_log_of"]), abs=1e-15)
    assert sb[1] == pytest.approx(g["state_B"]["l"], abs=1e-15)
    assert sb[2][0] == pytest.approx(g["state_B"]["u"], abs=1e-15)
    # the rescale factor of A against the common maximum
    assert math.exp(sa[0] - max(sa[0], sb[0])) == pytest.approx(g["scale_factor_of_A"], abs=1e-15)
    m, l, u = states.merge(sa, sb)
    assert m == pytest.approx(math.log(g["merged"]["m_is_log_of"]), abs=1e-15)
    assert l == pytest.approx(g["merged"]["l"], abs=1e-14)
    assert u[0] == pytest.approx(g["merged"]["u"], abs=1e-14)
    assert u[0] / l == pytest.approx(g["o"], abs=1e-14)
    # merge is symmetric
    m2, l2, u2 = states.merge(sb, sa)
    assert (m2, l2) == (m, l) and u2[0] == u[0]
    # exponential masses of the two blocks in the global denominator
    assert sa[1] * math.exp(sa[0]) == pytest.approx(g["exponential_masses"][0], abs=1e-14)
    assert sb[1] * math.exp(sb[0]) == pytest.approx(g["exponential_masses"][1], abs=1e-14)


def test_example_25_1_negative_controls():
    g = golden("example_25_1.json")
    z = np.log(np.array(g["scores_are_natural_logs_of"], dtype=np.float64))
    v = np.array(g["values"], dtype=np.float64)[:, None]
    local = [states.finish(states.block_state(z[idx], v[idx]), 1)[0][0] for idx in g["blocks"]]
    assert local == pytest.approx(g["local_outputs"], abs=1e-14)
    assert sum(local) == pytest.approx(g["wrong_sum_of_local_outputs"])
    assert np.mean(local) == pytest.approx(g["wrong_equal_weight_average"])
    o, _, _ = states.blocked_attention(z, v, None, g["blocks"])
    assert o[0] == pytest.approx(g["o"], abs=1e-14)
    assert abs(o[0] - g["wrong_sum_of_local_outputs"]) > 1
    assert abs(o[0] - g["wrong_equal_weight_average"]) > 0.4


def test_example_25_1_through_explicit_oracle():
    """Same numbers through the explicit C oracle: d=1, q=1, scale=1, k_j=z_j."""
    g = golden("example_25_1.json")
    z = np.log(np.array(g["scores_are_natural_logs_of"], dtype=np.float64))
    q = np.ones((1, 1, 1, 1))
    k = z.reshape(1, 1, 3, 1)
    v = np.array(g["values"], dtype=np.float64).reshape(1, 1, 3, 1)
    r = run(q, k, v, [3], [[2]], 1.0)
    assert r["out"][0, 0] == pytest.approx(g["o"], abs=1e-14)
    assert r["lse"][0] == pytest.approx(math.log(sum(g["scores_are_natural_logs_of"])), abs=1e-14)
    assert (r["n_visible"][0], r["first"][0], r["last"][0]) == (3, 0, 2)


# ---------------------------------------------------------------- workbook

def test_exercise_33_2_mass_weighted_merge():
    g = golden("exercise_33_2.json")
    ma, mb = g["masses"]
    sa = states.block_state([math.log(ma)], [[g["values"][0]]])
    sb = states.block_state([math.log(mb)], [[g["values"][1]]])
    o, _ = states.finish(states.merge(sa, sb), 1)
    assert o[0] == pytest.approx(g["o"], abs=1e-14)
    assert abs(o[0] - g["wrong_equal_weight_average"]) > 0.5
    r = run(np.ones((1, 1, 1, 1)), np.log(np.array(g["masses"], float)).reshape(1, 1, 2, 1),
            np.array(g["values"], float).reshape(1, 1, 2, 1), [2], [[1]], 1.0)
    assert r["out"][0, 0] == pytest.approx(g["o"], abs=1e-14)


def _partition(rng, n):
    perm = rng.permutation(n)
    cuts = np.sort(rng.choice(np.arange(1, n), size=rng.integers(0, min(n - 1, 12) + 1), replace=False))
    blocks = np.split(perm, cuts)
    order = rng.permutation(len(blocks))
    return [blocks[i] for i in order]


def test_exercise_33_1_three_block_form():
    """m = max of three, l and u rescaled by e^{m_i - m}, equal the full sums."""
    rng = np.random.default_rng(7)
    z = rng.normal(size=9) * 3
    v = rng.normal(size=(9, 4))
    blocks = [[0, 1, 2], [3, 4], [5, 6, 7, 8]]
    st = [states.block_state(z[b], v[b]) for b in blocks]
    m = max(s[0] for s in st)
    l = sum(math.exp(s[0] - m) * s[1] for s in st)
    u = sum(math.exp(s[0] - m) * s[2] for s in st)
    assert m == z.max()
    assert l == pytest.approx(np.exp(z - z.max()).sum(), rel=1e-14)
    np.testing.assert_allclose(u, (np.exp(z - z.max())[:, None] * v).sum(0), rtol=1e-13, atol=1e-14)
    for perm in itertools.permutations(range(3)):
        s = states.EMPTY
        for i in perm:
            s = states.merge(s, st[i])
        assert s[0] == m
        assert s[1] == pytest.approx(l, rel=1e-14)
        np.testing.assert_allclose(s[2], u, rtol=1e-13, atol=1e-14)


def test_random_partitions_match_explicit_oracle():
    """Any blocking, any order, gives the explicit result (exact up to rounding):
    100 random partitions of the 1000 keys of the tiny fp32 workload."""
    from exact_blocked_attention_gb300 import workloads
    inp = workloads.generate(workloads.spec("tiny_fp32"))
    q = inp["q"].double().numpy()
    k = inp["k"].double().numpy()
    v = inp["v"].double().numpy()
    scale = inp["scale"]
    ref = oracle.attention(q, k, v, inp["seqlens"], inp["qpos"], scale)
    z = scale * (k[0, 0] @ q[0, 0, 0])
    rng = np.random.default_rng(0)
    for _ in range(100):
        o, lse, _ = states.blocked_attention(z, v[0, 0], None, _partition(rng, z.size))
        np.testing.assert_allclose(o, ref["out"][0], rtol=1e-12, atol=1e-13)
        assert lse == pytest.approx(ref["lse"][0], rel=1e-13, abs=1e-13)


def test_exercise_33_3_masked_block_versus_masked_row():
    rng = np.random.default_rng(3)
    z = rng.normal(size=12)
    v = rng.normal(size=(12, 3))
    valid = np.ones(12, bool)
    valid[4:8] = False  # one whole block masked
    with np.errstate(invalid="raise", over="raise"):
        o, lse, _ = states.blocked_attention(z, v, valid, [[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, 11]])
        # masked block first: the first NON-EMPTY block initialises the state
        o2, lse2, _ = states.blocked_attention(z, v, valid, [[4, 5, 6, 7], [8, 9, 10, 11], [0, 1, 2, 3]])
        # fully masked row: the defined output, no -inf - (-inf)
        o3, lse3, st3 = states.blocked_attention(z, v, np.zeros(12, bool), [[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, 11]])
    w = np.exp(z[valid] - z[valid].max())
    np.testing.assert_allclose(o, (w[:, None] * v[valid]).sum(0) / w.sum(), rtol=1e-13)
    np.testing.assert_allclose(o2, o, rtol=1e-13)
    assert lse2 == pytest.approx(lse, rel=1e-14)
    assert st3 is states.EMPTY and lse3 == -math.inf and np.all(o3 == 0)


# ---------------------------------------------------------------- exact brute force

def _rational_problem(rng, B, Hq, Hkv, Tq, Tmax, dv, with_bias):
    """Scores whose exponentials are exact rationals: q = (c, 0), scale = 1/c,
    k_j = (ln r_j, noise), bias = ln s_j or -inf, so e^{z_j} = r_j * s_j."""
    r = [[[Fraction(int(rng.integers(1, 9)), int(rng.integers(1, 5))) for _ in range(Tmax)]
          for _ in range(Hkv)] for _ in range(B)]
    vals = rng.integers(-4, 5, size=(B, Hkv, Tmax, dv)).astype(np.float64)
    c = 2.0
    q = np.zeros((B, Hq, Tq, 2))
    q[..., 0] = c
    k = rng.normal(size=(B, Hkv, Tmax, 2))  # the second dim must not leak in
    for b, h, j in itertools.product(range(B), range(Hkv), range(Tmax)):
        k[b, h, j, 0] = math.log(r[b][h][j])
    sfrac = None
    bias = None
    if with_bias:
        sfrac = [[[[None if rng.random() < 0.3 else Fraction(int(rng.integers(1, 4)), 1)
                    for _ in range(Tmax)] for _ in range(Tq)] for _ in range(Hq)] for _ in range(B)]
        bias = np.zeros((B, Hq, Tq, Tmax))
        for b, h, i, j in itertools.product(range(B), range(Hq), range(Tq), range(Tmax)):
            s = sfrac[b][h][i][j]
            bias[b, h, i, j] = -math.inf if s is None else math.log(s)
    return q, k, vals, r, sfrac, bias, 1.0 / c


def test_brute_force_exact_rationals_gqa_positions_bias():
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Tq, Tmax, dv = 2, 4, 2, 3, 6, 3
    for trial in range(6):
        with_bias = trial % 2 == 1
        q, k, vals, r, sfrac, bias, scale = _rational_problem(rng, B, Hq, Hkv, Tq, Tmax, dv, with_bias)
        seqlens = rng.integers(-1, Tmax + 2, size=B).astype(np.int32)
        qpos = rng.integers(-2, Tmax + 1, size=(B, Tq)).astype(np.int32)
        res = run(q, k, vals, seqlens, qpos, scale, bias=bias)
        G = Hq // Hkv
        for b, h, i in itertools.product(range(B), range(Hq), range(Tq)):
            row = (b * Hq + h) * Tq + i
            hk = h // G  # contiguous groups of query heads share a KV head
            num = [Fraction(0)] * dv
            den = Fraction(0)
            seen = []
            for j in range(Tmax):
                if not (j < seqlens[b] and j <= qpos[b, i]):
                    continue
                w = r[b][hk][j]
                if with_bias:
                    s = sfrac[b][h][i][j]
                    if s is None:
                        continue
                    w = w * s
                seen.append(j)
                den += w
                for t in range(dv):
                    num[t] += w * Fraction(vals[b, hk, j, t])
            assert res["n_visible"][row] == len(seen)
            assert res["first"][row] == (seen[0] if seen else -1)
            assert res["last"][row] == (seen[-1] if seen else -1)
            if not seen:
                assert res["lse"][row] == -math.inf
                assert np.all(res["out"][row] == 0.0)
                continue
            exact = np.array([float(x / den) for x in num])
            np.testing.assert_allclose(res["out"][row], exact, rtol=1e-13, atol=1e-13)
            assert res["lse"][row] == pytest.approx(math.log(den), abs=1e-13)


def test_brute_force_every_mask_over_three_keys():
    """All 8 visibility patterns over 3 keys, including the empty one."""
    rng = np.random.default_rng(5)
    q, k, vals, r, _, _, scale = _rational_problem(rng, 1, 1, 1, 1, 3, 2, False)
    for pattern in itertools.product([False, True], repeat=3):
        bias = np.where(np.array(pattern), 0.0, -math.inf).reshape(1, 1, 1, 3)
        res = run(q, k, vals, [3], [[2]], scale, bias=bias)
        keep = [j for j in range(3) if pattern[j]]
        if not keep:
            assert res["lse"][0] == -math.inf and np.all(res["out"][0] == 0)
            continue
        den = sum(r[0][0][j] for j in keep)
        exact = [float(sum(r[0][0][j] * Fraction(vals[0, 0, j, t]) for j in keep) / den) for t in range(2)]
        np.testing.assert_allclose(res["out"][0], exact, rtol=1e-13, atol=1e-13)
        assert res["n_visible"][0] == len(keep)


def test_out_of_contract_bias_is_rejected():
    q = np.ones((1, 1, 1, 1)); k = np.zeros((1, 1, 2, 1)); v = np.zeros((1, 1, 2, 1))
    for bad in (math.inf, math.nan):
        with pytest.raises(ValueError):
            run(q, k, v, [2], [[1]], 1.0, bias=np.array([0.0, bad]).reshape(1, 1, 1, 2))


# ---------------------------------------------------------------- closed forms

def test_constant_values_give_the_constant():
    rng = np.random.default_rng(2)
    q = rng.normal(size=(1, 2, 3, 8)); k = rng.normal(size=(1, 1, 50, 8)) * 4
    v = np.full((1, 1, 50, 5), -1.625)
    res = run(q, k, v, [37], [[0, 20, 100]], 0.7)
    np.testing.assert_allclose(res["out"], -1.625, rtol=0, atol=1e-15)


def test_zero_query_gives_mean_and_log_count():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, Tq, Tmax = 2, 2, 1, 4, 40
    q = np.zeros((B, Hq, Tq, 16)); k = rng.normal(size=(B, Hkv, Tmax, 16))
    v = rng.normal(size=(B, Hkv, Tmax, 3))
    seqlens = np.array([33, 40], np.int32)
    qpos = np.array([[0, 5, 32, 39], [-1, 0, 17, 60]], np.int32)
    res = run(q, k, v, seqlens, qpos, 0.125)
    for b, h, i in itertools.product(range(B), range(Hq), range(Tq)):
        row = (b * Hq + h) * Tq + i
        n = max(0, min(int(seqlens[b]), int(qpos[b, i]) + 1))
        if n == 0:
            assert res["lse"][row] == -math.inf
            continue
        np.testing.assert_allclose(res["out"][row], v[b, 0, :n].mean(0), rtol=1e-13, atol=1e-14)
        assert res["lse"][row] == pytest.approx(math.log(n), abs=1e-14)


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(6)
    q = rng.normal(size=(1, 1, 1, 8)); k = rng.normal(size=(1, 1, 9, 8)); v = rng.normal(size=(1, 1, 9, 4))
    res = run(q, k, v, [9], [[0]], 0.3)
    np.testing.assert_array_equal(res["out"][0], v[0, 0, 0])
    assert res["lse"][0] == pytest.approx(0.3 * float(q[0, 0, 0] @ k[0, 0, 0]), abs=1e-14)


def test_one_hot_values_expose_probabilities():
    """V = I: out[j] is the probability of key j; invisible keys give exactly 0."""
    rng = np.random.default_rng(8)
    Tmax = 12
    q = rng.normal(size=(1, 1, 3, 8)); k = rng.normal(size=(1, 1, Tmax, 8))
    v = np.eye(Tmax).reshape(1, 1, Tmax, Tmax)
    res = run(q, k, v, [10], [[3, 9, 11]], 0.5)
    for i, pos in enumerate([3, 9, 11]):
        n = min(10, pos + 1)
        assert np.all(res["out"][i, n:] == 0.0)
        assert np.all(res["out"][i, :n] > 0.0)
        assert res["out"][i].sum() == pytest.approx(1.0, abs=1e-14)
        z = 0.5 * (k[0, 0, :n] @ q[0, 0, i])
        assert res["out"][i, 0] / res["out"][i, 1] == pytest.approx(math.exp(z[0] - z[1]), rel=1e-13)


# ---------------------------------------------------------------- cache alignment

def test_logical_position_alignment_example():
    g = golden("cache_alignment.json")
    t, r = g["cache_length_before"], g["new_tokens"]
    rng = np.random.default_rng(9)
    q = rng.normal(size=(1, 1, r, 4)); k = rng.normal(size=(1, 1, t + r, 4)); v = rng.normal(size=(1, 1, t + r, 2))
    res = run(q, k, v, [t + r], [g["query_positions"]], 0.5)
    for i, keys in enumerate(g["visible_keys"]):
        assert res["n_visible"][i] == len(keys)
        assert (res["first"][i], res["last"][i]) == (keys[0], keys[-1])
    # the misaligned reading (positions from zero) is a different, wrong result
    bad = run(q, k, v, [t + r], [[0, 1]], 0.5)
    assert bad["n_visible"][0] == len(g["misaligned_control"]["visible_keys"])
    assert not np.allclose(bad["out"], res["out"])


def test_incremental_cache_equals_full_prefix():
    g = golden("cache_alignment.json")["incremental_check"]
    vec = np.array(g["vectors"])
    n = len(vec)
    x = vec.reshape(1, 1, n, 2)
    scale = 1 / math.sqrt(2)
    full = run(x, x, x, [n], [list(range(n))], scale)  # all rows in one call
    for end in range(1, n + 1):
        step = run(x[:, :, end - 1:end], x[:, :, :end], x[:, :, :end], [end], [[end - 1]], scale)
        np.testing.assert_allclose(step["out"][0], full["out"][end - 1], rtol=0, atol=g["tolerance"])
        # and each equals the plain softmax-weighted mean over the prefix
        z = scale * (vec[:end] @ vec[end - 1])
        w = np.exp(z - z.max()); w /= w.sum()
        np.testing.assert_allclose(step["out"][0], w @ vec[:end], rtol=0, atol=g["tolerance"])


def test_row_subset_matches_full_run():
    rng = np.random.default_rng(12)
    q = rng.normal(size=(2, 4, 3, 8)); k = rng.normal(size=(2, 2, 30, 8)); v = rng.normal(size=(2, 2, 30, 5))
    full = run(q, k, v, [30, 17], [[5, 10, 29], [0, 16, 40]], 0.4)
    rows = [23, 0, 7, 11]
    sub = run(q, k, v, [30, 17], [[5, 10, 29], [0, 16, 40]], 0.4, rows=rows)
    np.testing.assert_array_equal(sub["out"], full["out"][rows])
    np.testing.assert_array_equal(sub["lse"], full["lse"][rows])


# ---------------------------------------------------------------- token-tree verification
# "推理加速算法" (inference acceleration algorithms) §7.2.2 Medusa, tree
# attention verification: the T_q rows of a sequence are the nodes of a
# candidate tree; the last T_q cache entries hold their keys (node k at key
# len - T_q + k); a node sees the earlier cache and, in the tree, only its
# ancestors and itself.  The pins below take the ancestry from parent arrays
# (never from the bit masks the oracle reads).

def _ancestor_masks(parents):
    """Bit masks (int64) from a parent array: bit k of mask[i] = node k is i or
    an ancestor of i.  parents[0] = -1 (root); parents[k] < k."""
    masks = []
    for i in range(len(parents)):
        m, node = 0, i
        while node >= 0:
            m |= 1 << node
            node = parents[node]
        masks.append(m - (1 << 64) if m >= 1 << 63 else m)
    return np.array(masks, dtype=np.int64)


def _random_parents(rng, n):
    return [-1] + [int(rng.integers(0, k)) for k in range(1, n)]


def _is_ancestor_or_self(parents, k, i):
    node = i
    while node >= 0:
        if node == k:
            return True
        node = parents[node]
    return False


def run_tree(q, k, v, seqlens, qpos, scale, tree, bias=None):
    return oracle.attention(np.asarray(q, np.float64), np.asarray(k, np.float64),
                            np.asarray(v, np.float64), np.asarray(seqlens, np.int32),
                            np.asarray(qpos, np.int32), scale, bias=bias, tree=tree)


def test_tree_brute_force_exact_rationals():
    rng = np.random.default_rng(21)
    B, Hq, Hkv, Tq, Tmax, dv = 2, 4, 2, 5, 9, 3
    for trial in range(8):
        with_bias = trial % 2 == 1
        q, k, vals, r, sfrac, bias, scale = _rational_problem(rng, B, Hq, Hkv, Tq, Tmax, dv, with_bias)
        parents = [_random_parents(rng, Tq) for _ in range(B)]
        tree = np.stack([_ancestor_masks(p) for p in parents])
        # lengths include ones shorter than the tree (its first nodes then
        # have no cache entry) and positions that cut into the tree
        seqlens = rng.integers(2, Tmax + 2, size=B).astype(np.int32)
        qpos = np.where(rng.random((B, Tq)) < 0.7, Tmax + 5,
                        rng.integers(-1, Tmax, size=(B, Tq))).astype(np.int32)
        res = run_tree(q, k, vals, seqlens, qpos, scale, tree, bias=bias)
        G = Hq // Hkv
        for b, h, i in itertools.product(range(B), range(Hq), range(Tq)):
            row = (b * Hq + h) * Tq + i
            hk = h // G
            length = min(int(seqlens[b]), Tmax)
            num = [Fraction(0)] * dv
            den = Fraction(0)
            seen = []
            for j in range(Tmax):
                if not (j < length and j <= qpos[b, i]):
                    continue
                node = j - (length - Tq)
                if node >= 0 and not _is_ancestor_or_self(parents[b], node, i):
                    continue
                w = r[b][hk][j]
                if with_bias:
                    s = sfrac[b][h][i][j]
                    if s is None:
                        continue
                    w = w * s
                seen.append(j)
                den += w
                for t in range(dv):
                    num[t] += w * Fraction(vals[b, hk, j, t])
            assert res["n_visible"][row] == len(seen)
            assert res["first"][row] == (seen[0] if seen else -1)
            assert res["last"][row] == (seen[-1] if seen else -1)
            if not seen:
                assert res["lse"][row] == -math.inf
                assert np.all(res["out"][row] == 0.0)
                continue
            exact = np.array([float(x / den) for x in num])
            np.testing.assert_allclose(res["out"][row], exact, rtol=1e-13, atol=1e-13)
            assert res["lse"][row] == pytest.approx(math.log(den), abs=1e-13)


def test_tree_chain_equals_causal_positions():
    """A chain (every node the child of the one before) is ordinary causal
    verification: node i at logical position len - T_q + i."""
    rng = np.random.default_rng(22)
    B, Hq, Hkv, Tq, Tmax, d = 3, 4, 2, 7, 40, 8
    q = rng.normal(size=(B, Hq, Tq, d)); k = rng.normal(size=(B, Hkv, Tmax, d)); v = rng.normal(size=(B, Hkv, Tmax, d))
    seqlens = np.array([40, 23, 7], dtype=np.int32)
    chain = np.stack([_ancestor_masks([-1] + list(range(Tq - 1)))] * B)
    full = np.broadcast_to((seqlens - 1)[:, None], (B, Tq)).astype(np.int32)
    causal = (seqlens[:, None] - Tq + np.arange(Tq)[None, :]).astype(np.int32)
    a = run_tree(q, k, v, seqlens, full, 0.3, chain)
    b = run(q, k, v, seqlens, causal, 0.3)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["lse"], b["lse"])
    np.testing.assert_array_equal(a["n_visible"], b["n_visible"])


def test_tree_of_the_figure_one_hot():
    """The pages' candidate tree (t+1; t+2a, t+2b, t+2c below it; t+3a below
    t+2a) with V = I: a node's output is exactly 0 on every key of another
    branch and positive on the prefix, its ancestors and itself."""
    parents = [-1, 0, 0, 0, 1]  # t+1, t+2a, t+2b, t+2c, t+3a
    Tq, L = 5, 6
    Tmax = L + Tq
    rng = np.random.default_rng(23)
    q = rng.normal(size=(1, 1, Tq, 8)); k = rng.normal(size=(1, 1, Tmax, 8))
    v = np.eye(Tmax).reshape(1, 1, Tmax, Tmax)
    res = run_tree(q, k, v, [Tmax], [[Tmax - 1] * Tq], 0.5, _ancestor_masks(parents)[None])
    sees = {0: {0}, 1: {0, 1}, 2: {0, 2}, 3: {0, 3}, 4: {0, 1, 4}}
    for i in range(Tq):
        for j in range(Tmax):
            visible = j < L or (j - L) in sees[i]
            if visible:
                assert res["out"][i, j] > 0.0
            else:
                assert res["out"][i, j] == 0.0
        assert res["n_visible"][i] == L + len(sees[i])
        assert res["out"][i].sum() == pytest.approx(1.0, abs=1e-14)


def test_tree_needs_at_most_64_nodes():
    q = np.zeros((1, 1, 65, 2)); k = np.zeros((1, 1, 70, 2)); v = np.zeros((1, 1, 70, 2))
    with pytest.raises(ValueError):
        run_tree(q, k, v, [70], [[69] * 65], 1.0, np.zeros((1, 65), dtype=np.int64))


# ---------------------------------------------------------------- sliding window
# "Chapter 33: inference compute optimisation" §33.7, the paragraph of
# eq. 33.16: a window keeps only the keys of the prescribed range (here the
# W most recent positions up to the row's own); dropping the original mass
# delta moves the output by at most 2 delta M (M bounds the value norms).

def run_window(q, k, v, seqlens, qpos, scale, window, bias=None):
    return oracle.attention(np.asarray(q, np.float64), np.asarray(k, np.float64),
                            np.asarray(v, np.float64), np.asarray(seqlens, np.int32),
                            np.asarray(qpos, np.int32), scale, bias=bias, window=window)


def test_window_bound_of_eq_33_16():
    rng = np.random.default_rng(31)
    B, Hq, Hkv, Tq, Tmax, d = 2, 4, 2, 5, 60, 8
    q = rng.normal(size=(B, Hq, Tq, d)); k = rng.normal(size=(B, Hkv, Tmax, d))
    v = rng.normal(size=(B, Hkv, Tmax, d)) * rng.uniform(0.1, 3.0, size=(B, Hkv, Tmax, 1))
    seqlens = np.array([60, 41], dtype=np.int32)
    qpos = np.stack([np.arange(55, 60), np.arange(36, 41)]).astype(np.int32)
    scale = 0.7
    full = run(q, k, v, seqlens, qpos, scale)
    G = Hq // Hkv
    for W in (1, 3, 10, 40):
        win = run_window(q, k, v, seqlens, qpos, scale, W)
        for b, h, i in itertools.product(range(B), range(Hq), range(Tq)):
            row = (b * Hq + h) * Tq + i
            pos, hk = int(qpos[b, i]), h // G
            z = scale * (k[b, hk, :pos + 1] @ q[b, h, i])
            w = np.exp(z - full["lse"][row])            # the original attention probabilities
            delta = w[:max(0, pos + 1 - W)].sum()        # the mass the window drops
            M = np.linalg.norm(v[b, hk, :pos + 1], axis=1).max()
            err = np.linalg.norm(full["out"][row] - win["out"][row])
            if delta < 1:
                assert err <= 2 * delta * M + 1e-12
            assert win["n_visible"][row] == min(W, pos + 1)


def test_window_brute_force_exact_rationals():
    rng = np.random.default_rng(32)
    B, Hq, Hkv, Tq, Tmax, dv = 2, 4, 2, 3, 9, 3
    for trial in range(6):
        with_bias = trial % 2 == 1
        q, k, vals, r, sfrac, bias, scale = _rational_problem(rng, B, Hq, Hkv, Tq, Tmax, dv, with_bias)
        seqlens = rng.integers(0, Tmax + 2, size=B).astype(np.int32)
        qpos = rng.integers(-2, Tmax + 3, size=(B, Tq)).astype(np.int32)
        W = int(rng.integers(1, 6))
        res = run_window(q, k, vals, seqlens, qpos, scale, W, bias=bias)
        G = Hq // Hkv
        for b, h, i in itertools.product(range(B), range(Hq), range(Tq)):
            row = (b * Hq + h) * Tq + i
            hk = h // G
            num = [Fraction(0)] * dv
            den = Fraction(0)
            seen = []
            for j in range(Tmax):
                if not (j < seqlens[b] and j <= qpos[b, i] and qpos[b, i] - j < W):
                    continue
                wt = r[b][hk][j]
                if with_bias:
                    s = sfrac[b][h][i][j]
                    if s is None:
                        continue
                    wt = wt * s
                seen.append(j)
                den += wt
                for t in range(dv):
                    num[t] += wt * Fraction(vals[b, hk, j, t])
            assert res["n_visible"][row] == len(seen)
            if not seen:
                assert res["lse"][row] == -math.inf and np.all(res["out"][row] == 0.0)
                continue
            np.testing.assert_allclose(res["out"][row], [float(x / den) for x in num], rtol=1e-13, atol=1e-13)


def test_window_special_cases():
    rng = np.random.default_rng(33)
    q = rng.normal(size=(1, 2, 3, 8)); k = rng.normal(size=(1, 1, 30, 8)); v = rng.normal(size=(1, 1, 30, 4))
    sl, pos = [25], [[10, 24, 29]]
    # a window at least as long as every visible range changes nothing
    a = run_window(q, k, v, sl, pos, 0.4, 30)
    b = run(q, k, v, sl, pos, 0.4)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["lse"], b["lse"])
    # a window of one key returns that key's value exactly
    c = run_window(q, k, v, sl, pos, 0.4, 1)
    for h in range(2):
        np.testing.assert_array_equal(c["out"][h * 3 + 0], v[0, 0, 10])
        np.testing.assert_array_equal(c["out"][h * 3 + 1], v[0, 0, 24])
        # position 29 is past the cache (length 25): its one-key window is empty
        assert c["lse"][h * 3 + 2] == -math.inf and np.all(c["out"][h * 3 + 2] == 0.0)
