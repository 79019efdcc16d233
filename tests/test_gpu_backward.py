"""GPU parity of the backward pass (blkattn_bwd) against the fp64 oracle of
eqs. 33.6-33.8 ("Chapter 33: inference compute optimisation" §33.3).

Tolerance, from the arithmetic: the products take P and dS as bf16 operands
(relative rounding <= 2^-9 per term) and accumulate in fp32, so each
gradient element may move by a small multiple of 2^-9 times the sum of the
absolute values of its terms; the oracle returns those sums (error scales
dq_abs, dk_abs, dv_abs) and the bound is 2^-7 of them, plus 1e-6 of the
tensor's largest scale for fp32 noise.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import backward as obwd
from exact_blocked_attention_gb300 import blkattn, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    blkattn.load()


def make(B, Hq, Hkv, Tq, Tmax, seqlens, qpos, bias=None, seed=0, d=128):
    g = torch.Generator().manual_seed(seed)
    return {"q": torch.randn(B, Hq, Tq, d, generator=g).to(torch.bfloat16),
            "k": torch.randn(B, Hkv, Tmax, d, generator=g).to(torch.bfloat16),
            "v": torch.randn(B, Hkv, Tmax, d, generator=g).to(torch.bfloat16),
            "go": torch.randn(B, Hq, Tq, d, generator=g).to(torch.bfloat16),
            "seqlens": torch.tensor(seqlens, dtype=torch.int32),
            "qpos": torch.tensor(qpos, dtype=torch.int32), "bias": bias, "scale": d ** -0.5}


def reference(c, units=None):
    return obwd.attention_backward(c["q"], c["k"], c["v"], c["seqlens"], c["qpos"], c["scale"], c["go"],
                                   bias=c["bias"], units=units, window=c.get("window", 0))


def run(c, o, lse):
    """blkattn_bwd with the given forward output and lse (CPU tensors)."""
    dev = lambda t: None if t is None else t.cuda()
    dq, dk, dv = blkattn.attention_backward(dev(c["q"]), dev(c["k"]), dev(c["v"]), dev(c["seqlens"]),
                                            dev(c["qpos"]), dev(o), dev(lse), dev(c["go"]),
                                            mask_bias=dev(c["bias"]), scale=c["scale"], window=c.get("window", 0))
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


def oracle_forward_state(ref):
    """The forward output and lse from the oracle, as fp32 (the kernel's inputs)."""
    return torch.from_numpy(ref["o"]).float(), torch.from_numpy(ref["lse"]).float()


def assert_grads(got, ref, units=None, extra=None):
    for name, g in zip(("dq", "dk", "dv"), got):
        want, scale = ref[name], ref[name + "_abs"]
        if extra is not None and name in extra:
            scale = scale + 2.0 ** 7 * extra[name]  # (bound = 2^-7 scale)
        g = g.double().numpy()
        if units is not None:  # compare only what the oracle computed
            G = ref["dq"].shape[1] // ref["dk"].shape[1]
            sel = [(b, slice(hk * G, hk * G + G) if name == "dq" else hk) for b, hk in units]
            g = np.concatenate([g[b, s].reshape(-1, g.shape[-1]) for b, s in sel])
            want = np.concatenate([want[b, s].reshape(-1, want.shape[-1]) for b, s in sel])
            scale = np.concatenate([scale[b, s].reshape(-1, scale.shape[-1]) for b, s in sel])
        assert np.all(np.isfinite(g)), name
        bound = 2.0 ** -7 * scale + 1e-6 * max(float(scale.max()), 1e-30)
        err = np.abs(g - want)
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        assert np.all(err <= bound), (f"{name}: worst excess {float((err - bound)[worst]):.3e} at {worst}, "
                                      f"err {float(err[worst]):.3e}, scale {float(scale[worst]):.3e}")
        # exact zeros where nothing is seen
        np.testing.assert_array_equal(g[scale == 0], 0.0)


def case(name):
    if name == "causal_mha":        # prefill-shaped, ragged tail (300 = 2 x 128 + 44)
        T = 300
        return make(2, 4, 4, T, T, [T, T], [list(range(T))] * 2, seed=1)
    if name == "causal_gqa_short":  # G = 4, a sequence shorter than the cache
        T = 257
        return make(2, 8, 2, T, T + 40, [T + 40, 200], [list(range(T)), list(range(T))], seed=2)
    if name == "decode_rows":       # few rows, long cache, empty and beyond-length rows
        return make(3, 8, 2, 5, 700, [700, 300, 1], [[699, 698, -1, 0, 350], [900, 299, 10, 128, 127],
                                                     [0, -5, 0, 3, 0]], seed=3)
    if name == "bias":               # -inf blocks, a fully masked (b, i) row, a fully masked head row
        B, H, T = 2, 4, 200
        g = torch.Generator().manual_seed(4)
        bias = torch.randn(B, H, T, T, generator=g)
        bias[torch.rand(B, H, T, T, generator=g) < 0.2] = -math.inf
        bias[:, :, 17, :] = -math.inf
        bias[1, 2, 100, :] = -math.inf
        return make(B, H, H, T, T, [T, 150], [list(range(T))] * 2, bias=bias, seed=5)
    if name == "noncausal":          # every row sees the whole cache
        return make(1, 2, 1, 130, 260, [260], [[259] * 130], seed=6)
    raise KeyError(name)


CASES = ["causal_mha", "causal_gqa_short", "decode_rows", "bias", "noncausal"]


@pytest.mark.parametrize("name", CASES)
def test_backward_matches_the_oracle(name):
    c = case(name)
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    assert_grads(run(c, o, lse), ref)


def test_backward_after_the_library_forward():
    """End to end: blkattn_fwd's own output and lse feed blkattn_bwd."""
    c = case("causal_gqa_short")
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in c.items()}
    out, lse = blkattn.attention(dev["q"], dev["k"], dev["v"], dev["seqlens"], dev["qpos"], None, c["scale"])
    torch.cuda.synchronize()
    assert_grads(run(c, out.cpu(), lse.cpu()), reference(c))


def test_backward_with_bf16_forward_output():
    """o rounded to bf16 moves D_i = g_o,i . o_i by dD_i (known exactly here);
    G_S moves by P dD, so dq moves by at most scale dD_i max_j |k_j| (the P of
    a row sum to 1) and dk_j by at most scale sum_i dD_i |q_i| (P <= 1)."""
    c = case("causal_mha")
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    o16 = o.to(torch.bfloat16)
    go = c["go"].double().numpy()
    dD = np.abs((go * (o16.double().numpy() - ref["o"])).sum(-1))  # [B, H, T]
    G = c["q"].shape[1] // c["k"].shape[1]
    kmax = np.abs(c["k"].double().numpy()).max(axis=2)            # [B, H_kv, d]
    kmax = np.repeat(kmax, G, axis=1)[:, :, None, :]
    qa = np.abs(c["q"].double().numpy())
    dk_extra = (dD[..., None] * qa).sum(axis=2)                     # [B, H_q, d]
    dk_extra = dk_extra.reshape(dk_extra.shape[0], -1, G, dk_extra.shape[-1]).sum(axis=2)[:, :, None, :]
    extra = {"dq": c["scale"] * dD[..., None] * kmax,
             "dk": c["scale"] * np.broadcast_to(dk_extra, ref["dk"].shape)}
    assert_grads(run(c, o16, lse), ref, extra=extra)


def test_backward_is_deterministic_and_ignores_cache_padding():
    """Two runs give the same bits; NaN in the cache rows past each length
    changes no bit, and those rows get zero gradient."""
    c = case("causal_gqa_short")
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    a = run(c, o, lse)
    b = run(c, o, lse)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    dirty = dict(c)
    for key in ("k", "v"):
        t = c[key].clone()
        t[1, :, 200:] = float("nan")
        dirty[key] = t
    d = run(dirty, o, lse)
    for x, y in zip(a, d):
        assert torch.equal(x, y)
    assert not a[1][1, :, 200:].any() and not a[2][1, :, 200:].any()


def test_key_gradients_sum_to_zero_per_head():
    """Shift invariance (Exercise 33.4): for each KV head, sum_j dk_j = 0."""
    c = case("decode_rows")
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    _, dk, _ = run(c, o, lse)
    s = dk.double().sum(dim=2).numpy()
    bound = 2.0 ** -7 * ref["dk_abs"].sum(axis=2) + 1e-5
    assert np.all(np.abs(s) <= bound)


def test_no_query_rows_gives_zero_key_gradients():
    c = make(2, 4, 2, 0, 300, [300, 100], np.zeros((2, 0), dtype=np.int32), seed=7)
    dk = torch.full((2, 2, 300, 128), 7.0, device="cuda")
    dv = torch.full((2, 2, 300, 128), 7.0, device="cuda")
    dq = torch.empty(2, 4, 0, 128, device="cuda")
    o = torch.empty(2, 4, 0, 128, device="cuda")
    lse = torch.empty(2, 4, 0, device="cuda")
    cu = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in c.items()}
    blkattn.bwd(cu["q"], cu["k"], cu["v"], cu["seqlens"], cu["qpos"], None, c["scale"], o, lse, cu["go"],
                dq, dk, dv)
    torch.cuda.synchronize()
    assert not dk.any() and not dv.any()


def test_full_size_backward_sampled_heads():
    """The backward workload at full size (B=2, 32 heads, T=8192, causal);
    every element of one (sequence, head) unit against the oracle."""
    s = workloads.backward_spec()
    inp = workloads.generate_backward(s)
    cu = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    out, lse = blkattn.attention(cu["q"], cu["k"], cu["v"], cu["seqlens"], cu["qpos"], None, inp["scale"])
    dq, dk, dv = blkattn.attention_backward(cu["q"], cu["k"], cu["v"], cu["seqlens"], cu["qpos"], out, lse,
                                            cu["go"], scale=inp["scale"])
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    units = [(1, s.Hkv - 1)]
    ref = obwd.attention_backward(inp["q"], inp["k"], inp["v"], inp["seqlens"], inp["qpos"], inp["scale"],
                                  inp["go"], units=units)
    assert_grads((dq.cpu(), dk.cpu(), dv.cpu()), ref, units=units)


def test_backward_into_strided_gradient_views():
    """dq, dk, dv written into views of larger buffers (padded rows): the
    same bits as contiguous outputs, and nothing outside the views changes."""
    c = case("decode_rows")
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    a = run(c, o, lse)
    cu = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in c.items()}
    views = []
    for t in (c["q"], c["k"], c["v"]):
        shape = tuple(t.shape)
        big = torch.full(shape[:-1] + (shape[-1] + 8,), 7.0, device="cuda")
        views.append((big, big[..., 4:4 + shape[-1]]))
    blkattn.bwd(cu["q"], cu["k"], cu["v"], cu["seqlens"], cu["qpos"], None, c["scale"], o.cuda(), lse.cuda(),
                cu["go"], views[0][1], views[1][1], views[2][1])
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    for (big, view), want in zip(views, a):
        assert torch.equal(view.cpu(), want)
        assert bool((big[..., :4] == 7.0).all()) and bool((big[..., -4:] == 7.0).all())


def test_backward_bias_broadcast_over_heads_with_groups():
    """A [B, 1, T_q, T_max] bias (stride 0 over heads) with grouped heads."""
    B, Hq, Hkv, T = 2, 8, 2, 190
    g = torch.Generator().manual_seed(12)
    bias = torch.randn(B, 1, T, T + 30, generator=g)
    bias[torch.rand(B, 1, T, T + 30, generator=g) < 0.15] = -math.inf
    bias[0, 0, 50, :] = -math.inf
    c = make(B, Hq, Hkv, T, T + 30, [T + 30, 120], [list(range(T))] * 2, bias=bias, seed=13)
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    assert_grads(run(c, o, lse), ref)


# sliding window ("Chapter 33" §33.7, the paragraph of eq. 33.16): keys
# pos - W < j <= pos; the dQ blocks start at their rows' earliest visible key
# tile and the dK/dV blocks visit only the query tiles whose windows reach them

def window_case(name):
    if name == "causal_w100":
        T = 300
        c = make(2, 4, 4, T, T, [T, 251], [list(range(T))] * 2, seed=21)
        c["window"] = 100
    elif name == "causal_w128_gqa":
        T = 520
        c = make(1, 8, 2, T, T, [T], [list(range(T))], seed=22)
        c["window"] = 128
    elif name == "w1":
        T = 200
        c = make(1, 2, 2, T, T, [T], [list(range(T))], seed=23)
        c["window"] = 1
    elif name == "decode_rows":
        c = case("decode_rows")
        c["window"] = 77
    elif name == "bias_broadcast":
        B, T = 2, 260
        g = torch.Generator().manual_seed(24)
        bias = torch.randn(B, 1, T, T, generator=g)
        bias[torch.rand(B, 1, T, T, generator=g) < 0.2] = -math.inf
        c = make(B, 4, 2, T, T, [T, 190], [list(range(T))] * 2, bias=bias, seed=25)
        c["window"] = 60
    elif name == "beyond_window":  # rows whose window starts at or past the length, next to live rows
        T = 300
        c = make(2, 2, 1, T, 800, [800, 700], [[100] * 127 + [1000] + [300, 888, 889, 5000] * 43,
                                               [650] * 128 + [789, 788, 2000] * 57 + [1]], seed=28)
        c["window"] = 90
    else:  # random positions, some beyond the length or negative
        rng = np.random.default_rng(26)
        B, T = 2, 270
        c = make(B, 4, 2, T, 700, [700, 300], [rng.integers(-4, 740, T).tolist(), rng.integers(-4, 330, T).tolist()],
                 seed=27)
        c["window"] = 150
    return c


WINDOW_CASES = ["causal_w100", "causal_w128_gqa", "w1", "decode_rows", "bias_broadcast", "random_pos", "beyond_window"]


@pytest.mark.parametrize("name", WINDOW_CASES)
def test_window_backward_matches_the_oracle(name):
    c = window_case(name)
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    assert_grads(run(c, o, lse), ref)


def test_window_backward_after_the_library_windowed_forward():
    c = window_case("causal_w128_gqa")
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in c.items()}
    out, lse = blkattn.attention(dev["q"], dev["k"], dev["v"], dev["seqlens"], dev["qpos"], None, c["scale"],
                                 window=c["window"])
    torch.cuda.synchronize()
    assert_grads(run(c, out.cpu(), lse.cpu()), reference(c))


@pytest.mark.parametrize("window", [0, 300])
def test_many_key_tiles_with_a_bias(window):
    """Nine key tiles per head, with a bias that masks a fifth of the
    entries: the dQ kernel's K ring (three slots) and V ring (two) wrap
    several times, and its bias instantiations read S chunk by chunk."""
    B, H, T = 1, 2, 1100
    g = torch.Generator().manual_seed(31 + window)
    bias = torch.randn(B, H, T, T, generator=g)
    bias[torch.rand(B, H, T, T, generator=g) < 0.2] = -math.inf
    c = make(B, H, 1, T, T, [T], [list(range(T))], bias=bias, seed=32 + window)
    c["window"] = window
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    assert_grads(run(c, o, lse), ref)


def test_window_covering_everything_changes_no_bit():
    """A window longer than every row's history: the windowed kernels give the
    same bits as the unwindowed ones."""
    c = window_case("causal_w100")
    ref = reference(dict(c, window=0))
    o, lse = oracle_forward_state(ref)
    a = run(dict(c, window=0), o, lse)
    b = run(dict(c, window=100000), o, lse)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_a_captured_backward_replays_on_new_data():
    """blkattn_bwd captured once in a CUDA graph (after one uncaptured call)
    and replayed on new Q, K, V and g_o written into the same buffers: each
    replay's gradients are the oracle's for the data present at replay time."""
    c = case("causal_gqa_short")
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in c.items()}
    od, lsed = o.cuda(), lse.cuda()
    dq = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(dev["k"].shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(dev["v"].shape, dtype=torch.float32, device="cuda")
    call = lambda: blkattn.bwd(dev["q"], dev["k"], dev["v"], dev["seqlens"], dev["qpos"], None, c["scale"],
                               od, lsed, dev["go"], dq, dk, dv)
    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call()
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(2):
        new = make(2, 8, 2, 257, 297, [297, 200], [list(range(257)), list(range(257))], seed=40 + rep)
        ref = reference(new)
        o, lse = oracle_forward_state(ref)
        for key in ("q", "k", "v", "go"):
            dev[key].copy_(new[key])
        od.copy_(o)
        lsed.copy_(lse)
        dq.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert blkattn.check_device_error() == 0
        assert_grads((dq.cpu(), dk.cpu(), dv.cpu()), ref)


def test_token_major_layouts():
    """Q, K, V and g_o stored token-major ([B, T, H, d]) and passed as
    [B, H, T, d] views: the backward's tensor maps follow the strides."""
    c = case("causal_gqa_short")
    ref = reference(c)
    o, lse = oracle_forward_state(ref)
    tm = lambda t: t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)  # token-major storage
    dq, dk, dv = blkattn.attention_backward(tm(c["q"]), tm(c["k"]), tm(c["v"]), c["seqlens"].cuda(),
                                            c["qpos"].cuda(), o.cuda(), lse.cuda(), tm(c["go"]),
                                            mask_bias=None, scale=c["scale"])
    torch.cuda.synchronize()
    assert blkattn.check_device_error() == 0
    assert_grads((dq.cpu(), dk.cpu(), dv.cpu()), ref)
