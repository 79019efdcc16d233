"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances (written here, derived from the arithmetic): for bf16 inputs with
fp32 accumulation and an fp32 output, max |out - out_ref| <= 2e-3 * (1 +
|out_ref|) and |lse - lse_ref| <= 1e-3; for the fp32 workload 1e-5 for both.
A bf16 output may differ by its own rounding on top: half a bf16 ulp of
out_ref (at most 2^-8 |out_ref|).  Rows with no valid key must be exact:
out == +0.0 and lse == -inf.  The integer facts (which rows are fully masked)
are compared bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_blocked_attention_gb300 import blkattn, workloads
from exact_blocked_attention_gb300 import build as libbuild

pytestmark = pytest.mark.gpu

BF16_TOL_O, BF16_TOL_L = 2e-3, 1e-3
F32_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    blkattn.load()


def to_dev(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def run_gpu(inp, out_dtype=torch.float32):
    g = to_dev(inp)
    out, lse = blkattn.attention(g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], g["bias"],
                                 g["scale"], out_dtype=out_dtype, tree=g.get("tree"), window=g.get("window", 0))
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    d = out.shape[-1]
    return out.cpu(), lse.cpu(), out.double().cpu().numpy().reshape(-1, d), lse.double().cpu().numpy().reshape(-1)


def run_oracle(inp, rows=None):
    return oracle.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"], inp["qpos"], inp["scale"],
                            bias=inp["bias"], rows=rows, tree=inp.get("tree"), window=inp.get("window", 0))


def assert_parity(o, l, ref, tol_o, tol_l, out_raw=None, bf16_out=False):
    masked = ref["n_visible"] == 0
    gpu_masked = np.isneginf(l)
    np.testing.assert_array_equal(gpu_masked, masked)  # integer fact, exact
    assert np.all(o[masked] == 0.0)
    if out_raw is not None and masked.any():
        assert not torch.signbit(out_raw.float().reshape(-1, o.shape[1])[torch.from_numpy(masked)]).any()
    live = ~masked
    if not live.any():
        return
    ro = ref["out"][live]
    bound = tol_o * (1 + np.abs(ro))
    if bf16_out:
        bound = bound + np.abs(ro) * 2.0 ** -8
    err = np.abs(o[live] - ro)
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), f"out: max excess {float((err - bound).flat[worst]):.3e}, max err {err.max():.3e}"
    assert np.all(np.isfinite(l[live]))
    lerr = np.abs(l[live] - ref["lse"][live])
    assert lerr.max() <= tol_l, f"lse err {lerr.max():.3e}"
    return float((err / bound).max())  # the worst row's share of the bar


def tols(s):
    return (F32_TOL, F32_TOL) if s.dtype == "f32" else (BF16_TOL_O, BF16_TOL_L)


# ------------------------------------------------------------ reduced workloads, every row

@pytest.mark.parametrize("name", list(workloads.SMALL))
def test_small_workload_parity(name):
    s = workloads.spec(name, small=True)
    inp = workloads.generate(s)
    raw, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    assert_parity(o, l, ref, *tols(s), out_raw=raw)


@pytest.mark.parametrize("name", [n for n in workloads.SMALL if workloads.SMALL[n].dtype == "bf16"])
def test_small_workload_bf16_output(name):
    s = workloads.spec(name, small=True)
    inp = workloads.generate(s)
    raw, _, o, l = run_gpu(inp, out_dtype=torch.bfloat16)
    ref = run_oracle(inp)
    assert_parity(o, l, ref, *tols(s), out_raw=raw, bf16_out=True)


def test_tiny_fp32_workload_full():
    s = workloads.spec("tiny_fp32")
    inp = workloads.generate(s)
    _, _, o, l = run_gpu(inp)
    assert_parity(o, l, run_oracle(inp), F32_TOL, F32_TOL)


# ------------------------------------------------------------ full-size workloads

def prefill_rows(s, n_random=2000, seed=0):
    """Every row of the first and the last (sequence, head) pair, and random
    rows of the others (the oracle's cost grows with T_q^2 per head)."""
    rng = np.random.default_rng(seed)
    total = s.B * s.Hq * s.Tq
    rows = set(range(s.Tq))
    rows.update(range(total - s.Tq, total))
    rows.update(rng.choice(total, size=min(n_random, total), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def split_units(inp, ctas):
    """Units (sequence, KV head, row group) of the tcgen05 decode kernel whose
    key tiles fall in more than one CTA's range, from the kernel's published
    partition: units in (sequence, KV head, row group) order, each taking
    ceil(end / 128) key tiles (at least one; 48-row units two more), cut into
    min(#CTAs, tiles) equal contiguous ranges (no window, no tree)."""
    B, Hq, Tq, _ = inp["q"].shape
    Hkv, Tmax = inp["k"].shape[1], inp["k"].shape[2]
    rows = (Hq // Hkv) * Tq
    rg = (rows + 47) // 48
    R = (rows + rg - 1) // rg
    extra = 2 if R > 32 else 0
    lens = np.clip(inp["seqlens"].numpy().astype(np.int64), 0, Tmax)
    qpos = inp["qpos"].numpy().astype(np.int64)
    n = []
    for b in range(B):
        for _h in range(Hkv):
            for g in range(rg):
                ids = np.arange(g * R, min(g * R + R, rows)) % Tq
                mp = qpos[b, ids].max()
                end = 0 if mp < 0 else min(mp + 1, lens[b])
                n.append(max(1, -(-end // 128)) + extra)
    n = np.array(n, dtype=np.int64)
    su = np.concatenate([[0], np.cumsum(n)[:-1]])
    W = int(n.sum())
    P = min(W, ctas)
    cta_of = lambda t: ((t + 1) * P + W - 1) // W - 1
    return int(np.sum(cta_of(su) != cta_of(su + n - 1)))


@pytest.mark.parametrize("name", ["decode_gqa", "long_decode", "spec_verify", "prefill", "tree_verify",
                                  "window_decode", "window_prefill"])
def test_full_size_workload(name):
    """The full-size workloads at the sizes bench.py times: every row of the
    decode and verify workloads (the CTA boundaries of the stream-K cut fall
    at data-dependent keys), two whole heads and 2000 random rows of the
    prefill shapes."""
    s = workloads.spec(name)
    inp = workloads.generate(s)
    raw, _, o, l = run_gpu(inp)
    if s.Tq >= 64:
        rows = prefill_rows(s)
        ref = run_oracle(inp, rows=rows)
        share = assert_parity(o[rows], l[rows], ref, *tols(s))
        # P goes to the PV product as one bf16 value on key tiles every row
        # of the query tile sees in full (P_hi + P_lo elsewhere): a numpy
        # study put the worst row at 0.37 of the bar; keep a clear margin
        print(f"{name}: worst row at {share:.3f} of the output bar")
        assert share <= 0.75
    else:
        ref = run_oracle(inp)
        assert_parity(o, l, ref, *tols(s))
        if name in ("decode_gqa", "long_decode", "spec_verify"):
            plan = plan_of(inp)
            assert plan["kernel"] == 3
            # the in-kernel fold of units split across CTAs is on this path
            assert split_units(inp, plan["ctas"]) > 0
    if s.bias != "none":
        assert (ref["n_visible"] == 0).any(), "the fully masked rows must be checked"


# ------------------------------------------------------------ worked example on the GPU

def test_example_25_1_on_gpu():
    """Scores (log 2, log 1, log 6), values (1, 4, 5) -> o = 4: d = 64, fp32,
    scale 1/8, q = 8 e0, k_j = z_j e0, v_j = value_j e0."""
    d = 64
    q = torch.zeros(1, 1, 1, d); q[0, 0, 0, 0] = 8.0
    k = torch.zeros(1, 1, 3, d); k[0, 0, :, 0] = torch.tensor([math.log(2), 0.0, math.log(6)])
    v = torch.zeros(1, 1, 3, d); v[0, 0, :, 0] = torch.tensor([1.0, 4.0, 5.0])
    inp = {"q": q, "k": k, "v": v, "seqlens": torch.tensor([3], dtype=torch.int32),
           "qpos": torch.tensor([[2]], dtype=torch.int32), "bias": None, "scale": 1 / 8}
    _, _, o, l = run_gpu(inp)
    assert o[0, 0] == pytest.approx(4.0, abs=1e-5)
    assert np.all(o[0, 1:] == 0)
    assert l[0] == pytest.approx(math.log(9.0), abs=1e-5)


# ------------------------------------------------------------ merge API and split invariance

def states_from_fwd(out, lse):
    rows = out.shape[0] * out.shape[1] * out.shape[2]
    return lse.reshape(rows).contiguous(), None, out.reshape(rows, -1).contiguous()


def test_random_key_partitions_merge_to_the_whole():
    """fwd on disjoint key ranges + blkattn_merge == fwd on all keys (any
    partition, any order; eqs. 33.4-33.5 and their order independence)."""
    s = workloads.spec("tiny_fp32")
    inp = to_dev(workloads.generate(s))
    whole_o, whole_l = blkattn.attention(inp["q"], inp["k"], inp["v"], inp["seqlens"], inp["qpos"],
                                         None, inp["scale"])
    rng = np.random.default_rng(1)
    T = s.Tmax
    for trial in range(100):
        n_cuts = int(rng.integers(0, 12))
        # cuts on 4-key boundaries keep every K/V view 16-byte aligned (fp32 rows of 256 B are)
        cuts = sorted(set(rng.integers(1, T, size=n_cuts).tolist()))
        bounds = [0] + cuts + [T]
        parts = list(zip(bounds[:-1], bounds[1:]))
        rng.shuffle(parts)
        acc = None
        for lo, hi in parts:
            k = inp["k"][:, :, lo:hi]
            v = inp["v"][:, :, lo:hi]
            pos = inp["qpos"] - lo
            sl = torch.clamp(inp["seqlens"] - lo, min=0).to(torch.int32)
            o, l = blkattn.attention(inp["q"], k, v, sl, pos.to(torch.int32), None, inp["scale"])
            st = states_from_fwd(o, l)
            if acc is None:
                acc = st
            else:
                blkattn.merge(acc, st, acc)
        torch.cuda.synchronize()
        np.testing.assert_allclose(acc[2].cpu().numpy(), whole_o.reshape(1, -1).cpu().numpy(), rtol=0, atol=1e-5)
        np.testing.assert_allclose(acc[0].cpu().numpy(), whole_l.reshape(-1).cpu().numpy(), rtol=0, atol=1e-5)


def test_merge_matches_oracle_states():
    from oracle import states as ost
    rng = np.random.default_rng(4)
    rows, d = 1000, 48
    ma = rng.normal(size=rows) * 5
    mb = rng.normal(size=rows) * 5
    ma[::7] = -np.inf
    mb[::11] = -np.inf
    la = rng.uniform(0.5, 20, rows); lb = rng.uniform(0.5, 20, rows)
    ua = rng.normal(size=(rows, d)); ub = rng.normal(size=(rows, d))
    f = lambda x: torch.tensor(x, dtype=torch.float32, device="cuda")
    A = (f(ma), f(la), f(ua)); Bs = (f(mb), f(lb), f(ub))
    out = (torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda"), torch.empty(rows, d, device="cuda"))
    blkattn.merge(A, Bs, out)
    norm = (torch.empty(rows, device="cuda"), None, torch.empty(rows, d, device="cuda"))
    blkattn.merge(A, Bs, norm)
    # aliasing: out = a
    Ac = tuple(t.clone() for t in A)
    blkattn.merge(Ac, Bs, Ac)
    torch.cuda.synchronize()
    a32 = lambda x: np.asarray(x, np.float32).astype(np.float64)
    for r in range(rows):
        sa = None if ma[r] == -np.inf else (a32(ma[r]), a32(la[r]), a32(ua[r]))
        sb = None if mb[r] == -np.inf else (a32(mb[r]), a32(lb[r]), a32(ub[r]))
        st = ost.merge(sa, sb)
        if st is None:
            assert out[0][r].item() == -math.inf and norm[0][r].item() == -math.inf
            assert torch.all(norm[2][r] == 0)
            continue
        m, l, u = st
        assert out[0][r].item() == pytest.approx(m, abs=1e-6)
        assert out[1][r].item() == pytest.approx(l, rel=1e-5)
        np.testing.assert_allclose(out[2][r].cpu().numpy(), u, rtol=1e-5, atol=1e-5)
        o, lse = ost.finish(st, d)
        np.testing.assert_allclose(norm[2][r].cpu().numpy(), o, rtol=1e-5, atol=1e-5)
        assert norm[0][r].item() == pytest.approx(lse, abs=1e-5)
    for t_ref, t in zip(out, Ac):
        torch.testing.assert_close(t, t_ref, rtol=0, atol=0)


def test_merge_example_25_1_states():
    """The printed states of Example 25.1 through blkattn_merge."""
    f = lambda x: torch.tensor(x, dtype=torch.float32, device="cuda")
    A = (f([math.log(2)]), f([1.5]), f([[3.0]]))
    Bs = (f([math.log(6)]), f([1.0]), f([[5.0]]))
    out = (f([0.0]), f([0.0]), f([[0.0]]))
    blkattn.merge(A, Bs, out)
    torch.cuda.synchronize()
    assert out[1].item() == pytest.approx(1.5, abs=1e-6)
    assert out[2].item() == pytest.approx(6.0, abs=1e-5)
    assert out[2].item() / out[1].item() == pytest.approx(4.0, abs=1e-5)


# ------------------------------------------------------------ padding, masks and edge cases

@pytest.mark.parametrize("name", ["decode_gqa", "spec_verify"])
def test_poisoned_padding_is_never_read(name):
    s = workloads.spec(name, small=True)
    clean = workloads.generate(s)
    for poison in (float("nan"), float("inf")):
        dirty = workloads.generate(s, poison_padding=poison)
        _, _, o1, l1 = run_gpu(clean)
        _, _, o2, l2 = run_gpu(dirty)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def make_case(B, Hq, Hkv, Tq, Tmax, d, dtype, seqlens, qpos, bias=None, seed=0):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return {"q": torch.randn(B, Hq, Tq, d, generator=g).to(dt),
            "k": torch.randn(B, Hkv, Tmax, d, generator=g).to(dt),
            "v": torch.randn(B, Hkv, Tmax, d, generator=g).to(dt),
            "seqlens": torch.tensor(seqlens, dtype=torch.int32),
            "qpos": torch.tensor(qpos, dtype=torch.int32), "bias": bias, "scale": d ** -0.5}


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 64)])
def test_edge_positions_and_lengths(dtype, d):
    """pos < 0, len 0, len > T_max, pos beyond len, one key, ragged tails."""
    B, Hq, Hkv, Tq, Tmax = 5, 6, 3, 3, 333
    seqlens = [0, 1, 333, 500, 130]
    qpos = [[5, -1, 0], [0, 0, 7], [332, 100, -5], [1000, 64, 63], [129, 128, 127]]
    inp = make_case(B, Hq, Hkv, Tq, Tmax, d, dtype, seqlens, qpos)
    _, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    assert ref["n_visible"].min() == 0 and ref["n_visible"].max() == 333
    tol = (F32_TOL, F32_TOL) if dtype == "f32" else (BF16_TOL_O, BF16_TOL_L)
    assert_parity(o, l, ref, *tol)


def test_dense_per_head_bias_with_masked_rows():
    B, Hq, Hkv, Tq, Tmax, d = 2, 8, 2, 4, 300, 128
    g = torch.Generator().manual_seed(3)
    bias = torch.randn(B, Hq, Tq, Tmax, generator=g) * 2
    bias[torch.rand(B, Hq, Tq, Tmax, generator=g) < 0.3] = -math.inf
    bias[0, 3, 1, :] = -math.inf  # one fully masked (b, h, i) row
    bias[1, :, 2, 100:] = -math.inf
    inp = make_case(B, Hq, Hkv, Tq, Tmax, d, "bf16", [300, 257], [[299, 100, 50, 299], [0, 256, 256, 300]], bias)
    _, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    assert (ref["n_visible"] == 0).sum() >= 1
    assert_parity(o, l, ref, BF16_TOL_O, BF16_TOL_L)


def test_one_hot_values_pin_visibility():
    """V = I over T_max <= d: out[i, j] is the probability of key j, and every
    invisible key gives exactly 0.0 (visibility checked bit-exactly)."""
    B, Hq, Hkv, Tq, Tmax, d = 2, 4, 2, 5, 128, 128
    inp = make_case(B, Hq, Hkv, Tq, Tmax, d, "f32", [128, 77], [[0, 5, 64, 127, 200], [-1, 10, 76, 77, 3]])
    inp["v"] = torch.eye(Tmax, d).expand(B, Hkv, Tmax, d).contiguous()
    _, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    for r in range(o.shape[0]):
        n = ref["n_visible"][r]
        last = ref["last"][r]
        assert np.all(o[r, last + 1:] == 0.0)
        if n:
            assert np.all(o[r, :last + 1] > 0.0)
    assert_parity(o, l, ref, F32_TOL, F32_TOL)


def test_strided_views():
    """Non-contiguous q / out / lse and K/V that are views into a larger cache."""
    B, Hq, Hkv, Tq, d = 3, 8, 4, 2, 128
    g = torch.Generator().manual_seed(5)
    big_k = torch.randn(B, Hkv, 700, d, generator=g).to(torch.bfloat16).cuda()
    big_v = torch.randn(B, Hkv, 700, d, generator=g).to(torch.bfloat16).cuda()
    k = big_k[:, :, 64:600]  # row-aligned view
    v = big_v[:, :, 64:600]
    qt = torch.randn(B, Tq, Hq, d, generator=g).to(torch.bfloat16).cuda()
    q = qt.transpose(1, 2)  # [B, Hq, Tq, d] with a permuted layout
    sl = torch.tensor([536, 300, 17], dtype=torch.int32).cuda()
    qp = torch.tensor([[535, 534], [299, 400], [16, 3]], dtype=torch.int32).cuda()
    out_store = torch.empty(B, Tq, Hq, d, device="cuda")
    out = out_store.transpose(1, 2)
    lse_store = torch.empty(B, Tq, Hq, device="cuda")
    lse = lse_store.transpose(1, 2)
    blkattn.fwd(q, k, v, sl, qp, None, d ** -0.5, out, lse)
    torch.cuda.synchronize()
    ref = oracle.attention(q.cpu().contiguous(), k.cpu().contiguous(), v.cpu().contiguous(), sl.cpu(),
                           qp.cpu(), d ** -0.5)
    assert_parity(out.double().cpu().numpy().reshape(-1, d), lse.double().cpu().numpy().reshape(-1), ref,
                  BF16_TOL_O, BF16_TOL_L)


def test_empty_calls_are_no_ops():
    inp = to_dev(make_case(1, 2, 1, 1, 16, 64, "bf16", [16], [[15]]))
    out = torch.full((0, 2, 1, 64), 7.0, device="cuda")
    lse = torch.full((0, 2, 1), 7.0, device="cuda")
    z = lambda t: t[:0]
    blkattn.fwd(z(inp["q"]), z(inp["k"]), z(inp["v"]), z(inp["seqlens"]), z(inp["qpos"]), None, 0.1, out, lse)
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0


# ------------------------------------------------------------ token-tree verification
# "推理加速算法" (inference acceleration algorithms) §7.2.2 Medusa, tree
# attention verification: rows are tree nodes whose keys are the last T_q
# cache entries; each sees the prefix and its ancestors (blkattn_fwd_tree).

def _tree_masks(parents_per_seq):
    out = []
    for parents in parents_per_seq:
        row = []
        for i in range(len(parents)):
            m, node = 0, i
            while node >= 0:
                m |= 1 << node
                node = parents[node]
            row.append(m - (1 << 64) if m >= 1 << 63 else m)
        out.append(row)
    return torch.tensor(out, dtype=torch.int64)


def tree_case(name):
    rng = np.random.default_rng(["nr48", "nr32_two_groups", "nr16", "d64_mma", "fp32_split",
                                 "short_cache", "with_bias", "deep64"].index(name) + 40)
    dtype, d, bias = "bf16", 128, None
    if name == "nr48":              # 8 heads x 6 nodes = 48 rows per KV head
        B, Hq, Hkv, Tq, lens = 3, 16, 2, 6, [700, 1290, 301]
    elif name == "nr32_two_groups":  # 64 nodes, G = 1: two row groups of 32
        B, Hq, Hkv, Tq, lens = 2, 2, 2, 64, [900, 640]
    elif name == "nr16":             # 2 heads x 8 nodes = 16 rows
        B, Hq, Hkv, Tq, lens = 2, 4, 2, 8, [333, 1024]
    elif name == "d64_mma":          # head dim 64: the mma.sync split kernel
        B, Hq, Hkv, Tq, lens, d = 2, 8, 2, 10, [512, 777], 64
    elif name == "fp32_split":       # fp32: the CUDA-core split kernel
        B, Hq, Hkv, Tq, lens, dtype, d = 2, 4, 2, 7, [260, 515], "f32", 64
    elif name == "short_cache":      # cache shorter than the tree: early nodes have no key
        B, Hq, Hkv, Tq, lens = 2, 8, 2, 12, [5, 12]
    elif name == "with_bias":        # tree and an additive -inf bias together
        B, Hq, Hkv, Tq, lens = 2, 8, 2, 6, [400, 130]
    else:                            # deep64: a 64-node chain-heavy tree over 3 row groups
        B, Hq, Hkv, Tq, lens = 1, 4, 2, 64, [3000]
    Tmax = max(lens) + 3
    parents = [[-1] + [int(rng.integers(max(0, k - 3) if name == "deep64" else 0, k)) for k in range(1, Tq)]
               for _ in range(B)]
    qpos = [[ln - 1] * Tq for ln in lens]
    if name == "with_bias":
        bias = torch.zeros(B, 1, Tq, Tmax)
        bias[0, 0, :, 100:230] = -math.inf
        bias[1, 0, 2, :] = -math.inf  # one node sees nothing
    inp = make_case(B, Hq, Hkv, Tq, Tmax, d, dtype, lens, qpos, bias=bias, seed=int(rng.integers(1 << 30)))
    inp["tree"] = _tree_masks(parents)
    return inp


TREE_CASES = ["nr48", "nr32_two_groups", "nr16", "d64_mma", "fp32_split", "short_cache", "with_bias", "deep64"]


@pytest.mark.parametrize("name", TREE_CASES)
def test_tree_verify_cases(name):
    inp = tree_case(name)
    expect = {"d64_mma": 1, "fp32_split": 0}.get(name, 3)  # the kernel each case is for
    if inp["q"].shape[2] < 64:  # (the debug plan has no tree flag: with 64 rows it names prefill,
        assert plan_of(inp)["kernel"] == expect  # which tree calls never take)
    _, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    tol = (F32_TOL, F32_TOL) if inp["q"].dtype == torch.float32 else (BF16_TOL_O, BF16_TOL_L)
    assert_parity(o, l, ref, *tol)


def test_tree_chain_equals_causal_verify_bitwise():
    """A chain tree with every row at len-1 masks exactly the keys causal
    verification (row i at len - T_q + i) masks: same plan, same bits."""
    B, Hq, Hkv, Tq = 3, 16, 2, 6
    lens = [800, 1290, 1030]
    Tmax = 1290
    chain = [[-1] + list(range(Tq - 1))] * B
    full = make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", lens, [[ln - 1] * Tq for ln in lens], seed=77)
    causal = dict(full)
    causal["qpos"] = torch.tensor([[ln - Tq + i for i in range(Tq)] for ln in lens], dtype=torch.int32)
    full["tree"] = _tree_masks(chain)
    raw_t, lse_t, _, _ = run_gpu(full)
    raw_c, lse_c, _, _ = run_gpu(causal)
    assert torch.equal(raw_t, raw_c)
    assert torch.equal(lse_t, lse_c)


# "Chapter 33: inference compute optimisation" §33.7 (the paragraph of
# eq. 33.16): sliding-window attention, each row at position pos sees the keys
# pos - W < j <= pos (blkattn_fwd_window).

def window_case(name):
    rng = np.random.default_rng(WINDOW_CASES.index(name) + 60)
    dtype, d, bias = "bf16", 128, None
    if name == "tc_nr16":            # decode, 16 rows per KV head
        B, Hq, Hkv, lens, W = 3, 32, 2, [3000, 1290, 17], 500
        qpos = [[ln - 1] for ln in lens]
    elif name == "tc_verify_nr48":   # causal verification rows: a different start per row
        B, Hq, Hkv, lens, W = 3, 16, 2, [2000, 700, 300], 333
        qpos = [[ln - 6 + i for i in range(6)] for ln in lens]
    elif name == "tc_two_groups":    # 64 rows of one head (a prefill shape: the windowed prefill kernel)
        B, Hq, Hkv, lens, W = 2, 2, 2, [1900, 640], 100
        qpos = [[ln - 64 + i for i in range(64)] for ln in lens]
    elif name == "tc_window_one":    # each row sees exactly its own key
        B, Hq, Hkv, lens, W = 2, 16, 2, [900, 5], 1
        qpos = [[ln - 3 + i for i in range(3)] for ln in lens]
    elif name == "tc_tile_edges":    # windows that start on and next to key-tile edges
        B, Hq, Hkv, lens, W = 4, 16, 2, [4097, 4096, 129, 256], 128
        qpos = [[ln - 1, ln - 2] for ln in lens]
    elif name == "tc_mixed_positions":  # pos < 0, 0, beyond the length and far apart in one unit
        B, Hq, Hkv, lens, W = 3, 16, 2, [3000, 1500, 10], 50
        qpos = [[-1, 0, 2999, 1000], [5000, 1499, 1400, 60], [-3, 9, 20, 4]]
    elif name == "tc_bias":          # the window and an additive bias with -inf entries
        B, Hq, Hkv, lens, W = 2, 8, 2, [1500, 800], 400
        qpos = [[ln - 2, ln - 1] for ln in lens]
        g = torch.Generator().manual_seed(9)
        bias = torch.randn(B, Hq, 2, max(lens) + 3, generator=g)
        bias[torch.rand(B, Hq, 2, max(lens) + 3, generator=g) < 0.25] = -math.inf
        bias[0, 1, 0, 1099:] = -math.inf  # the whole window masked: an empty row
    elif name == "many_units":       # more units than the tcgen05 kernel takes with a window
        B, Hq, Hkv, W = 600, 4, 1, 100
        lens = rng.integers(1, 700, B).tolist()
        qpos = [[ln - 1] for ln in lens]
    elif name == "d64_mma":          # head dim 64: the mma.sync split kernel
        B, Hq, Hkv, lens, W, d = 2, 8, 2, [2000, 777], 300, 64
        qpos = [[ln - 4 + i for i in range(4)] for ln in lens]
    else:                            # fp32_split: the CUDA-core split kernel
        B, Hq, Hkv, lens, W, dtype, d = 2, 4, 2, [1300, 515], 77, "f32", 64
        qpos = [[ln - 3 + i for i in range(3)] for ln in lens]
    Tmax = max(lens) + 3
    Tq = len(qpos[0])
    inp = make_case(B, Hq, Hkv, Tq, Tmax, d, dtype, lens, qpos, bias=bias, seed=int(rng.integers(1 << 30)))
    inp["window"] = W
    return inp


WINDOW_CASES = ["tc_nr16", "tc_verify_nr48", "tc_two_groups", "tc_window_one", "tc_tile_edges",
                "tc_mixed_positions", "tc_bias", "many_units", "d64_mma", "fp32_split"]


@pytest.mark.parametrize("name", WINDOW_CASES)
def test_window_cases(name):
    inp = window_case(name)
    if name.startswith("tc_") and name != "tc_two_groups":  # (the debug plan has no window flag)
        assert plan_of(inp)["kernel"] == 3
    raw, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    tol = (F32_TOL, F32_TOL) if inp["q"].dtype == torch.float32 else (BF16_TOL_O, BF16_TOL_L)
    assert_parity(o, l, ref, *tol)
    if name == "tc_window_one":  # one visible key: the output is that key's value row
        B, Hq, Tq = inp["q"].shape[:3]
        G = Hq // inp["k"].shape[1]
        for b in range(B):
            for h in range(Hq):
                for i in range(Tq):
                    pos = int(inp["qpos"][b, i])
                    if 0 <= pos < int(inp["seqlens"][b]):
                        want = inp["v"][b, h // G, pos].float()
                        assert torch.allclose(raw[b, h, i], want, rtol=2.0 ** -8, atol=1e-6)


@pytest.mark.parametrize("name", ["tc_verify_nr48", "d64_mma", "fp32_split"])
def test_window_covering_the_cache_changes_no_bit(name):
    """A window at least as long as every row's key range masks nothing: the
    same kernel, the same bits as the call without a window."""
    inp = window_case(name)
    plain = dict(inp)
    plain["window"] = 0
    wide = dict(inp)
    wide["window"] = int(inp["seqlens"].max()) + 1
    raw_p, lse_p, _, _ = run_gpu(plain)
    raw_w, lse_w, _, _ = run_gpu(wide)
    assert torch.equal(raw_p, raw_w)
    assert torch.equal(lse_p, lse_w)


def window_prefill_case(name):
    """Prefill shapes (many query rows per head) with a sliding window: the
    tcgen05 prefill kernel with a first key tile per CTA and a window mask."""
    rng = np.random.default_rng(WINDOW_PREFILL_CASES.index(name) + 80)
    if name == "causal_w100":        # window shorter than a key tile, ragged T
        B, Hq, Hkv, T, lens, W = 2, 4, 4, 700, [700, 451], 100
        qpos = [list(range(T))] * B
    elif name == "causal_w128_gqa":  # window of exactly one key tile, grouped heads
        B, Hq, Hkv, T, lens, W = 1, 8, 2, 1030, [1030], 128
        qpos = [list(range(T))]
    elif name == "causal_w1":        # every row sees only its own key
        B, Hq, Hkv, T, lens, W = 1, 2, 2, 300, [300], 1
        qpos = [list(range(T))]
    elif name == "causal_w1000":     # window longer than most rows' history
        B, Hq, Hkv, T, lens, W = 1, 2, 2, 1500, [1500], 1000
        qpos = [list(range(T))]
    elif name == "last_rows":        # non-causal rows: every row sees the last W keys
        B, Hq, Hkv, T, lens, W = 2, 2, 1, 200, [900, 333], 257
        qpos = [[899] * T, [332] * T]
    elif name == "beyond_window":    # rows whose window starts at or past the length, next to live rows
        # (len 800, W 90: pos >= 889 sees nothing, pos 888 sees key 799 only)
        B, Hq, Hkv, T, lens, W = 2, 2, 1, 300, [800, 700], 90
        qpos = [[100] * 127 + [1000] + [300, 888, 889, 5000] * 43, [650] * 128 + [789, 788, 2000] * 57 + [1]]
    else:                            # random positions, including negative and beyond the length
        B, Hq, Hkv, T, lens, W = 2, 4, 2, 260, [800, 190], 90
        qpos = [rng.integers(-5, ln + 40, size=T).tolist() for ln in lens]
    Tmax = max(max(lens), T)
    inp = make_case(B, Hq, Hkv, T, Tmax, 128, "bf16", lens, qpos, seed=int(rng.integers(1 << 30)))
    inp["window"] = W
    return inp


WINDOW_PREFILL_CASES = ["causal_w100", "causal_w128_gqa", "causal_w1", "causal_w1000", "last_rows", "random_pos",
                        "beyond_window"]


@pytest.mark.parametrize("name", WINDOW_PREFILL_CASES)
def test_window_prefill_cases(name):
    inp = window_prefill_case(name)
    assert plan_of(inp)["kernel"] == 2  # the tcgen05 prefill kernel
    raw, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    assert_parity(o, l, ref, BF16_TOL_O, BF16_TOL_L, out_raw=raw)
    if name == "beyond_window":  # the empty rows share query tiles with rows that see keys
        assert (ref["n_visible"] == 0).sum() >= 2 * 43 * 2 and (ref["n_visible"] > 0).any()


def test_window_prefill_covering_the_cache_changes_no_bit():
    """A window longer than every row's history: the windowed prefill kernel
    gives the same bits as the unwindowed one."""
    inp = window_prefill_case("causal_w100")
    plain = dict(inp)
    plain["window"] = 0
    wide = dict(inp)
    wide["window"] = 100000
    raw_p, lse_p, _, _ = run_gpu(plain)
    raw_w, lse_w, _, _ = run_gpu(wide)
    assert torch.equal(raw_p, raw_w)
    assert torch.equal(lse_p, lse_w)


def test_window_error_bound_of_eq_33_16():
    """Eq. 33.16 on the kernel's own outputs: with delta the softmax mass the
    full row puts outside the window (1 - exp(lse_W - lse_full)) and M the
    largest value norm, |o_full - o_W| <= 2 delta M."""
    inp = window_case("tc_nr16")
    _, lse_w, o_w, l_w = run_gpu(inp)
    full = dict(inp)
    full["window"] = 0
    _, _, o_f, l_f = run_gpu(full)
    delta = 1.0 - np.exp(l_w.astype(np.float64) - l_f.astype(np.float64))
    M = float(inp["v"].float().norm(dim=-1).max())
    gap = np.linalg.norm(o_f.astype(np.float64) - o_w.astype(np.float64), axis=-1)
    assert np.all(gap <= 2.0 * delta * M + 1e-2)
    assert np.any(delta > 0.1)  # the window really drops mass here


# ------------------------------------------------------------ tcgen05 prefill kernel

def plan_of(inp):
    s_q = inp["q"]
    B, Hq, Tq, d = s_q.shape
    Hkv, Tmax = inp["k"].shape[1], inp["k"].shape[2]
    dt = torch.bfloat16 if s_q.dtype == torch.bfloat16 else torch.float32
    return blkattn.debug_plan(B, Hq, Hkv, Tq, Tmax, d, dt, torch.cuda.get_device_properties(0).multi_processor_count)


@pytest.mark.parametrize("case", ["causal", "gqa_cache", "noncausal", "neg_pos", "short_len", "tail"])
def test_prefill_kernel_cases(case):
    seed = ["causal", "gqa_cache", "noncausal", "neg_pos", "short_len", "tail"].index(case)
    if case == "causal":
        B, Hq, Hkv, Tq, Tmax = 2, 2, 2, 300, 300
        seqlens = [300, 300]
        qpos = [list(range(Tq))] * B
    elif case == "gqa_cache":  # new rows after a cache: positions L..L+Tq-1
        B, Hq, Hkv, Tq, Tmax = 2, 4, 2, 130, 700
        seqlens = [650, 700]
        qpos = [list(range(520, 650)), list(range(570, 700))]
    elif case == "noncausal":
        B, Hq, Hkv, Tq, Tmax = 1, 2, 1, 200, 333
        seqlens = [333]
        qpos = [[332] * Tq]
    elif case == "neg_pos":  # some rows see nothing, one tile sees nothing at all
        B, Hq, Hkv, Tq, Tmax = 1, 2, 2, 256, 256
        seqlens = [256]
        qpos = [[-1] * 128 + list(range(-60, 68))]
    elif case == "short_len":  # cache shorter than the positions
        B, Hq, Hkv, Tq, Tmax = 2, 2, 1, 192, 500
        seqlens = [100, 0]
        qpos = [list(range(192)), list(range(192))]
    else:  # T_q not a multiple of 128, T_max not a multiple of 64
        B, Hq, Hkv, Tq, Tmax = 1, 3, 1, 129, 129
        seqlens = [129]
        qpos = [list(range(129))]
    inp = make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", seqlens, qpos, seed=seed)
    assert plan_of(inp)["kernel"] == 2
    _, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    assert_parity(o, l, ref, BF16_TOL_O, BF16_TOL_L)
    raw, _, ob, lb = run_gpu(inp, out_dtype=torch.bfloat16)
    assert_parity(ob, lb, ref, BF16_TOL_O, BF16_TOL_L, out_raw=raw, bf16_out=True)


@pytest.mark.parametrize("layout", ["padded_rows", "seq_major", "odd_row_stride"])
def test_prefill_output_layouts(layout):
    """Output views into larger buffers: whole tiles go out by TMA where the
    layout allows it (fp32, 16-byte strides), row by row otherwise; memory of
    the buffer outside the view is never written (the tail tile is clipped)."""
    B, Hq, Hkv, Tq, Tmax = 2, 3, 1, 161, 161
    inp = make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", [161, 150], [list(range(Tq))] * B, seed=11)
    assert plan_of(inp)["kernel"] == 2
    g = to_dev(inp)
    sentinel = 12345.0
    if layout == "padded_rows":  # rows past T_q in the buffer
        buf = torch.full((B, Hq, Tq + 40, 128), sentinel, device="cuda")
        out = buf[:, :, :Tq]
    elif layout == "seq_major":  # [B, T, H, d] storage seen as [B, H, T, d]
        buf = torch.full((B, Tq + 8, Hq, 128), sentinel, device="cuda")
        out = buf[:, :Tq].permute(0, 2, 1, 3)
    else:  # row stride of 130 floats: not a multiple of 16 bytes
        buf = torch.full((B, Hq, Tq, 130), sentinel, device="cuda")
        out = buf[..., :128]
    lse = torch.empty(B, Hq, Tq, device="cuda")
    blkattn.fwd(g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], None, g["scale"], out, lse)
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    o = out.double().cpu().numpy().reshape(-1, 128)
    assert_parity(o, lse.double().cpu().numpy().reshape(-1), run_oracle(inp), BF16_TOL_O, BF16_TOL_L)
    outside = torch.ones_like(buf, dtype=torch.bool)
    if layout == "padded_rows":
        outside[:, :, :Tq] = False
    elif layout == "seq_major":
        outside[:, :Tq] = False
    else:
        outside[..., :128] = False
    assert torch.all(buf[outside] == sentinel)


def test_prefill_kernel_poisoned_padding():
    B, Hq, Hkv, Tq, Tmax = 1, 2, 2, 200, 512
    qpos = [list(range(100, 300))]
    clean = make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", [300], qpos)
    dirty = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in clean.items()}
    dirty["k"][:, :, 300:] = float("nan")
    dirty["v"][:, :, 300:] = float("inf")
    assert plan_of(clean)["kernel"] == 2
    _, _, o1, l1 = run_gpu(clean)
    _, _, o2, l2 = run_gpu(dirty)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    assert_parity(o1, l1, run_oracle(clean), BF16_TOL_O, BF16_TOL_L)


def test_prefill_shape_with_bias_uses_the_split_kernel():
    B, Hq, Hkv, Tq, Tmax = 1, 2, 1, 160, 160
    bias = torch.zeros(B, 1, Tq, Tmax)
    bias[0, 0, :, 5:37] = -math.inf
    inp = make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", [160], [list(range(Tq))], bias)
    _, _, o, l = run_gpu(inp)
    assert_parity(o, l, run_oracle(inp), BF16_TOL_O, BF16_TOL_L)


def test_prefill_shape_with_negative_scale():
    """A non-positive scale is valid input; it is served by the split kernel."""
    B, Hq, Hkv, Tq, Tmax = 1, 2, 1, 96, 96
    inp = make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", [96], [list(range(Tq))])
    inp["scale"] = -0.05
    _, _, o, l = run_gpu(inp)
    assert_parity(o, l, run_oracle(inp), BF16_TOL_O, BF16_TOL_L)


# ------------------------------------------------------------ tcgen05 decode kernel
# One persistent CTA per SM shares the key tiles of all (sequence, KV head,
# row group) units equally; units spanning several CTAs are merged.  The
# cases below cover the shapes of that schedule: fewer tiles than CTAs, many
# units per CTA, units over many CTAs, two row groups, each row count class
# (16 / 32 / 48 columns), rescaling in the middle of a CTA's range, and rows
# whose first visible key comes late.

def tc_case(name):
    rng = np.random.default_rng(11)
    if name == "fewer_tiles_than_ctas":
        return make_case(2, 4, 1, 1, 300, 128, "bf16", [100, 0], [[99], [0]])
    if name == "many_units":
        B = 300
        lens = rng.integers(0, 257, B)
        lens[:3] = [0, 1, 256]
        pos = (lens - 1)[:, None]
        return make_case(B, 8, 2, 1, 256, 128, "bf16", lens.tolist(), pos.tolist(), seed=1)
    if name == "units_over_many_ctas":
        return make_case(1, 8, 2, 2, 20000, 128, "bf16", [19999], [[19997, 19998]], seed=2)
    if name == "two_row_groups":
        B, Hq, Hkv, Tq, Tmax = 3, 32, 2, 4, 1500
        g = torch.Generator().manual_seed(4)
        bias = torch.randn(B, Hq, Tq, Tmax, generator=g)
        bias[torch.rand(B, Hq, Tq, Tmax, generator=g) < 0.2] = -math.inf
        return make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", [1500, 700, 1],
                         [[1496, 1497, 1498, 1499], [10, 699, 300, -1], [0, 0, 5, 0]], bias, seed=3)
    if name == "rows32":
        return make_case(4, 16, 2, 4, 3000, 128, "bf16", [3000, 2999, 1200, 64],
                         [[2996, 2997, 2998, 2999], [2995, 2996, 2997, 2998], [1196, 1197, 1198, 1199],
                          [60, 61, 62, 63]], seed=5)
    if name == "rising_scores":
        inp = make_case(8, 8, 8, 1, 8192, 128, "bf16", [8192] * 8, [[8191]] * 8, seed=6)
        # scores grow along the cache: the reference maximum must be raised
        # (and U^T rescaled) in the middle of a CTA's key range
        ramp = torch.linspace(0.2, 3.0, 8192)[None, None, :, None]
        inp["k"] = (inp["k"].float() * ramp).to(torch.bfloat16)
        return inp
    if name == "many_tiles_long":
        # more than 32 key tiles per CTA over a few long units
        return make_case(2, 8, 8, 1, 40000, 128, "bf16", [40000, 39001], [[39999], [39000]], seed=8)
    if name == "many_tiles_many_units":
        B = 600
        lens = rng.integers(1000, 1200, B)
        pos = (lens - 1)[:, None]
        return make_case(B, 4, 1, 1, 1200, 128, "bf16", lens.tolist(), pos.tolist(), seed=9)
    if name == "late_first_key":
        B, Hq, Hkv, Tq, Tmax = 2, 8, 2, 3, 2000
        bias = torch.zeros(B, 1, Tq, Tmax)
        bias[0, 0, 0, :1500] = -math.inf  # first visible key in a late tile
        bias[1, 0, 1, :1999] = -math.inf  # exactly one visible key
        bias[1, 0, 2, :] = -math.inf      # none
        return make_case(B, Hq, Hkv, Tq, Tmax, 128, "bf16", [2000, 2000],
                         [[1997, 1998, 1999], [1997, 1998, 1999]], bias, seed=7)
    raise KeyError(name)


TC_CASES = ["fewer_tiles_than_ctas", "many_units", "units_over_many_ctas", "two_row_groups", "rows32",
            "rising_scores", "late_first_key", "many_tiles_long", "many_tiles_many_units"]


@pytest.mark.parametrize("case", TC_CASES)
def test_tc_decode_kernel_cases(case):
    inp = tc_case(case)
    assert plan_of(inp)["kernel"] == 3
    raw, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    assert_parity(o, l, ref, BF16_TOL_O, BF16_TOL_L, out_raw=raw)


@pytest.mark.parametrize("name", ["decode_gqa", "long_decode", "spec_verify"])
def test_tc_decode_kernel_serves_the_decode_workloads(name):
    s = workloads.spec(name)
    p = blkattn.debug_plan(s.B, s.Hq, s.Hkv, s.Tq, s.Tmax, s.d, torch.bfloat16,
                           torch.cuda.get_device_properties(0).multi_processor_count)
    assert p["kernel"] == 3


@pytest.fixture
def force_split_mma(monkeypatch):
    monkeypatch.setenv("BLKATTN_KERNEL", "mma")
    yield


@pytest.mark.parametrize("name", ["decode_gqa", "long_decode", "spec_verify"])
def test_split_mma_kernel_small_workloads(force_split_mma, name):
    """The mma.sync split-KV kernel stays correct (it serves d = 64 and
    non-contiguous query rows)."""
    s = workloads.spec(name, small=True)
    inp = workloads.generate(s)
    assert plan_of(inp)["kernel"] == 1
    raw, _, o, l = run_gpu(inp)
    assert_parity(o, l, run_oracle(inp), *tols(s), out_raw=raw)


@pytest.mark.parametrize("case", ["many_units", "two_row_groups", "late_first_key"])
def test_split_mma_kernel_cases(force_split_mma, case):
    inp = tc_case(case)
    assert plan_of(inp)["kernel"] == 1
    raw, _, o, l = run_gpu(inp)
    assert_parity(o, l, run_oracle(inp), BF16_TOL_O, BF16_TOL_L, out_raw=raw)


def test_tc_decode_counters_are_left_clean_between_shapes():
    """Units spanning several CTAs are folded by the last CTA to arrive (a
    per-unit counter that every launch must leave at zero): interleaved shapes
    with different unit counts give the same results as when run alone."""
    cases = [tc_case("units_over_many_ctas"), tc_case("rows32"), tc_case("many_tiles_many_units"),
             tc_case("many_units"), tc_case("many_tiles_long")]
    first = [run_gpu(c)[2:] for c in cases]
    for _ in range(2):
        for c, (o0, l0) in zip(reversed(cases), reversed(first)):
            _, _, o, l = run_gpu(c)
            np.testing.assert_array_equal(o, o0)
            np.testing.assert_array_equal(l, l0)


# ------------------------------------------------------------ device checks of the boundary

def test_tensors_must_be_on_the_current_device():
    """A call whose tensors are not all on the current device is refused with
    BLKATTN_ERR_INVALID_ARG before anything is enqueued; the next call on the
    same buffers still gives the oracle's result."""
    import ctypes
    s = workloads.spec("decode_gqa", small=True)
    inp = workloads.generate(s)
    g = to_dev(inp)
    out = torch.full((s.B, s.Hq, s.Tq, s.d), 7.0, device="cuda")
    lse = torch.full((s.B, s.Hq, s.Tq), 7.0, device="cuda")
    lib = blkattn.load()
    args = (g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], None)

    def call(descs):
        ref = lambda d: None if d is None else ctypes.byref(d)
        return lib.blkattn_fwd(*[ref(d) for d in descs[:6]], ctypes.c_float(g["scale"]), ref(descs[6]),
                               ref(descs[7]), None)

    descs = [blkattn.describe(t) for t in args + (out, lse)]
    for i in (1, 6):  # one tensor naming another device
        descs[i].device = torch.cuda.current_device() + 1
        assert call(descs) == blkattn.ERR_INVALID_ARG
        descs[i].device = torch.cuda.current_device()
    for d in descs:  # every tensor naming a device that is not current
        if d is not None:
            d.device = torch.cuda.current_device() + 1
    assert call(descs) == blkattn.ERR_INVALID_ARG
    with pytest.raises(ValueError):  # a host tensor (device -1 in its descriptor)
        blkattn.fwd(g["q"], inp["k"], g["v"], g["seqlens"], g["qpos"], None, g["scale"], out, lse)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())  # nothing was enqueued
    blkattn.fwd(*args, g["scale"], out, lse)
    torch.cuda.synchronize()
    o = out.double().cpu().numpy().reshape(-1, s.d)
    l = lse.double().cpu().numpy().reshape(-1)
    assert_parity(o, l, run_oracle(inp), BF16_TOL_O, BF16_TOL_L)


# ------------------------------------------------------------ bounded waits

def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_correct():
    """One CTA of the tcgen05 decode kernel is stopped at a wait nothing
    completes (the test hook).  Its bounded waits run out: the call returns,
    the device error word reads BLKATTN_ERR_DEVICE_TIMEOUT, and the next call
    on the same device and buffers matches the oracle on every row, although
    the stopped CTA left split units half counted."""
    import time
    s = workloads.spec("decode_gqa", small=True)
    inp = workloads.generate(s)
    g = to_dev(inp)
    plan = plan_of(inp)
    assert plan["kernel"] == 3 and plan["ctas"] > 1
    out = torch.empty(s.B, s.Hq, s.Tq, s.d, device="cuda")
    lse = torch.empty(s.B, s.Hq, s.Tq, device="cuda")
    args = (g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], None, g["scale"], out, lse)
    blkattn.fwd(*args)
    assert blkattn.check_device_error() == 0
    blkattn.stall_next_decode(1)  # (CTA 1 holds key tiles of split units)
    t0 = time.perf_counter()
    blkattn.fwd(*args)
    assert blkattn.check_device_error() == blkattn.ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 30.0  # bounded: about 2 s of waits
    assert blkattn.check_device_error() == 0  # read and cleared
    for _ in range(2):
        out.fill_(7.0)
        blkattn.fwd(*args)
        assert blkattn.check_device_error() == 0
        o = out.double().cpu().numpy().reshape(-1, s.d)
        l = lse.double().cpu().numpy().reshape(-1)
        assert_parity(o, l, run_oracle(inp), BF16_TOL_O, BF16_TOL_L)


# ------------------------------------------------------------ guard bands

@pytest.mark.parametrize("name", list(workloads.SMALL))
def test_outputs_stay_inside_their_views(name):
    """out and lse as views inside larger buffers filled with a sentinel
    (padding on every dimension): every kernel path writes its view and
    nothing around it."""
    s = workloads.spec(name, small=True)
    inp = workloads.generate(s)
    g = to_dev(inp)
    sentinel = -7777.0
    obuf = torch.full((s.B + 1, s.Hq + 2, s.Tq + 3, s.d + 8), sentinel, device="cuda")
    lbuf = torch.full((s.B + 1, s.Hq + 2, s.Tq + 5), sentinel, device="cuda")
    out = obuf[1:, 1:-1, 2:-1, 4:-4]
    lse = lbuf[:-1, 2:, 3:-2]
    blkattn.fwd(g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], g["bias"], g["scale"], out, lse,
                tree=g.get("tree"), window=g.get("window", 0))
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    omask = torch.ones_like(obuf, dtype=torch.bool)
    omask[1:, 1:-1, 2:-1, 4:-4] = False
    lmask = torch.ones_like(lbuf, dtype=torch.bool)
    lmask[:-1, 2:, 3:-2] = False
    assert bool((obuf[omask] == sentinel).all()) and bool((lbuf[lmask] == sentinel).all())
    o = out.double().cpu().numpy().reshape(-1, s.d)
    l = lse.double().cpu().numpy().reshape(-1)
    assert_parity(o, l, run_oracle(inp), *tols(s))


# ------------------------------------------------------------ tensor-map cache

def test_tensor_maps_stay_valid_when_the_cache_turns_over_inside_a_call():
    """The library caches TMA descriptors per (tensor, box) in a small ring.
    One K cache is reused across calls (a cache hit every time) while each
    call brings a fresh V (a miss, written at the ring's next position); after
    at most one turn of the ring that miss lands on the very entry K was found
    in, during the same call.  Every call must still read its own K and V."""
    g = torch.Generator().manual_seed(77)
    B, Hq, Hkv, T, d = 2, 8, 2, 300, 128
    q = torch.randn(B, Hq, 1, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
    sl = torch.tensor([T, 211], dtype=torch.int32)
    qp = (sl - 1).view(B, 1).to(torch.int32)
    qd, kd, sld, qpd = q.cuda(), k.cuda(), sl.cuda(), qp.cuda()
    keep = []  # every V stays alive: each call's V is at a new address
    for it in range(40):
        v = torch.randn(B, Hkv, T, d, generator=g).to(torch.bfloat16)
        vd = v.cuda()
        keep.append(vd)
        out, lse = blkattn.attention(qd, kd, vd, sld, qpd, None, d ** -0.5)
        torch.cuda.synchronize()
        ref = oracle.attention(q, k, v, sl, qp, d ** -0.5)
        assert_parity(out.double().cpu().numpy().reshape(-1, d), lse.double().cpu().numpy().reshape(-1), ref,
                      BF16_TOL_O, BF16_TOL_L)


# ------------------------------------------------------------ CUDA graphs

@pytest.mark.parametrize("name", ["decode_gqa", "spec_verify", "window_decode", "prefill"])
def test_a_captured_call_replays_on_new_data(name):
    """A serving loop captures the call once in a CUDA graph and replays it on
    new inputs written into the same buffers: after one uncaptured call (which
    grows the scratch, builds the tensor maps), the captured call allocates
    nothing, and every replay gives the oracle's result for the data in the
    buffers at replay time (the split-unit counters are left at zero by every
    launch, so replays do not see each other's state)."""
    s = workloads.spec(name, small=True)
    inp = workloads.generate(s)
    g = to_dev(inp)
    out = torch.empty(s.B, s.Hq, s.Tq, s.d, device="cuda")
    lse = torch.empty(s.B, s.Hq, s.Tq, device="cuda")
    call = lambda: blkattn.fwd(g["q"], g["k"], g["v"], g["seqlens"], g["qpos"], g["bias"], g["scale"], out, lse,
                               tree=g.get("tree"), window=g.get("window", 0))
    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call()
    torch.cuda.current_stream().wait_stream(side)
    gen = torch.Generator().manual_seed(5)
    for rep in range(3):
        new = dict(inp)
        for key in ("q", "k", "v"):
            new[key] = torch.randn(inp[key].shape, generator=gen).to(inp[key].dtype)
            g[key].copy_(new[key])
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert blkattn.check_device_error() == 0
        o = out.double().cpu().numpy().reshape(-1, s.d)
        l = lse.double().cpu().numpy().reshape(-1)
        assert_parity(o, l, run_oracle(new), *tols(s))


# ------------------------------------------------------------ large offsets

@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
def test_caches_larger_than_2_gib_per_tensor(dtype, d):
    """K and V of one call larger than 2^31 bytes each (4 KV heads of 2.2 to
    4.4 M keys; the last head's last rows lie past 2 GiB): every kernel path (tcgen05
    decode for bf16 d = 128, the mma.sync kernel for bf16 d = 64, CUDA cores
    for fp32) addresses them with 64-bit offsets.  Checked on one row of the
    first and one of the last KV head against the oracle."""
    B, Hkv, G = 1, 4, 2
    Hq = Hkv * G
    elt = 2 if dtype == torch.bfloat16 else 4
    T = int(2 ** 31 * 1.05) // (Hkv * d * elt)  # 5 % past 2 GiB per tensor
    assert Hkv * T * d * elt > 2 ** 31
    gen = torch.Generator(device="cuda").manual_seed(11)
    k = torch.randn(B, Hkv, T, d, device="cuda", generator=gen, dtype=dtype)
    v = torch.randn(B, Hkv, T, d, device="cuda", generator=gen, dtype=dtype)
    q = torch.randn(B, Hq, 1, d, device="cuda", generator=gen, dtype=dtype)
    sl = torch.tensor([T], dtype=torch.int32)
    qp = torch.tensor([[T - 1]], dtype=torch.int32)
    out, lse = blkattn.attention(q, k, v, sl.cuda(), qp.cuda(), None, d ** -0.5)
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    rows = np.array([0, Hq - 1])  # head 0 (KV head 0) and head Hq - 1 (KV head 3)
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), sl, qp, d ** -0.5, rows=rows)
    o = out.double().cpu().numpy().reshape(-1, d)[rows]
    l = lse.double().cpu().numpy().reshape(-1)[rows]
    tol = (BF16_TOL_O, BF16_TOL_L) if dtype == torch.bfloat16 else (F32_TOL, F32_TOL)
    assert_parity(o, l, ref, *tol)


# ------------------------------------------------------------ token-major caches

@pytest.mark.parametrize("kind", ["decode_d128", "decode_d64", "verify_48_rows", "prefill"])
def test_token_major_layouts(kind):
    """Q, K and V stored token-major ([B, T, H, d], as many serving caches
    keep them) and passed as [B, H, T, d] views with permuted strides: the
    tensor maps and the row addressing follow the strides."""
    g = torch.Generator().manual_seed(21)
    d = 64 if kind == "decode_d64" else 128
    if kind == "prefill":
        B, Hq, Hkv, Tq, T = 2, 4, 2, 300, 300
        sl = torch.tensor([300, 251], dtype=torch.int32)
        qp = torch.stack([torch.arange(Tq), torch.arange(Tq) - 49]).to(torch.int32)
    else:
        B, Hq, Hkv, T = 3, 16 if kind == "verify_48_rows" else 8, 2, 900
        Tq = 5 if kind == "verify_48_rows" else 1
        sl = torch.tensor([900, 413, 37], dtype=torch.int32)
        qp = (sl.view(B, 1) - Tq + torch.arange(Tq).view(1, Tq)).to(torch.int32)
    kt = torch.randn(B, T, Hkv, d, generator=g).to(torch.bfloat16)
    vt = torch.randn(B, T, Hkv, d, generator=g).to(torch.bfloat16)
    qt = torch.randn(B, Tq, Hq, d, generator=g).to(torch.bfloat16)
    k, v, q = kt.cuda().permute(0, 2, 1, 3), vt.cuda().permute(0, 2, 1, 3), qt.cuda().permute(0, 2, 1, 3)
    out, lse = blkattn.attention(q, k, v, sl.cuda(), qp.cuda(), None, d ** -0.5)
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    ref = oracle.attention(qt.permute(0, 2, 1, 3).contiguous(), kt.permute(0, 2, 1, 3).contiguous(),
                           vt.permute(0, 2, 1, 3).contiguous(), sl, qp, d ** -0.5)
    assert_parity(out.double().cpu().numpy().reshape(-1, d), lse.double().cpu().numpy().reshape(-1), ref,
                  BF16_TOL_O, BF16_TOL_L)


# ------------------------------------------------------------ unit-table limits

@pytest.mark.parametrize("B,window", [(1024, 0), (1025, 0), (512, 40), (513, 40)])
def test_unit_table_boundaries(B, window):
    """The tcgen05 decode kernel keeps its (sequence, row group) table in
    shared memory: at most 1024 entries, 512 with a sliding window (the other
    half holds the units' first tiles).  Batches at the limit run on it, one
    past it on the split-KV fallback; both give the oracle's results."""
    rng = np.random.default_rng(B + window)
    T = 96
    lens = rng.integers(1, T + 1, B)
    lens[:2] = [T, 1]
    inp = make_case(B, 4, 1, 1, T, 128, "bf16", lens.tolist(), (lens - 1)[:, None].tolist(), seed=B)
    if window:
        inp["window"] = window
    if not window:
        assert (plan_of(inp)["kernel"] == 3) == (B <= 1024)
    _, _, o, l = run_gpu(inp)
    ref = run_oracle(inp)
    assert_parity(o, l, ref, BF16_TOL_O, BF16_TOL_L)


def test_prefill_at_the_longest_query_block():
    """One head of a 131072-token causal prefill (512 CTAs of two query tiles,
    the longest rows over 1024 key tiles) against the oracle on sampled rows,
    the first and last rows included."""
    T, d = 131072, 128
    gen = torch.Generator(device="cuda").manual_seed(31)
    q = torch.randn(1, 1, T, d, device="cuda", generator=gen, dtype=torch.bfloat16)
    k = torch.randn(1, 1, T, d, device="cuda", generator=gen, dtype=torch.bfloat16)
    v = torch.randn(1, 1, T, d, device="cuda", generator=gen, dtype=torch.bfloat16)
    sl = torch.tensor([T], dtype=torch.int32)
    qp = torch.arange(T, dtype=torch.int32).view(1, T)
    assert plan_of({"q": q, "k": k})["kernel"] == 2
    out, lse = blkattn.attention(q, k, v, sl.cuda(), qp.cuda(), None, d ** -0.5)
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, T - 257, T - 1],
                                     np.random.default_rng(3).integers(0, T, 40)]))
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), sl, qp, d ** -0.5, rows=rows)
    o = out.double().cpu().numpy().reshape(-1, d)[rows]
    l = lse.double().cpu().numpy().reshape(-1)[rows]
    assert_parity(o, l, ref, BF16_TOL_O, BF16_TOL_L)
