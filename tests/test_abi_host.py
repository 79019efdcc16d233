"""Host-side checks of the C ABI: the library builds and loads, exports every
function include/blkattn.h declares, rejects invalid requests before any CUDA
call, and plans splits that partition the cache exactly once.  No GPU needed.
"""
import ctypes
import math
import os
import re

import pytest
import torch

from exact_blocked_attention_gb300 import blkattn, workloads
from exact_blocked_attention_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return blkattn.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "blkattn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\*)\s+(blkattn_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert set(blkattn.EXPORTED) <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert blkattn.status_string(st)
    assert blkattn.status_string(-99) == "unknown status"


class FakeTensor:
    """Descriptor with a fake (never dereferenced) device address."""

    def __init__(self, shape, dtype, strides=None, addr=0x10000, device=0):
        self.device = device
        self.shape = tuple(shape)
        self.dtype = dtype
        if strides is None:
            strides, acc = [], 1
            for s in reversed(self.shape):
                strides.insert(0, acc)
                acc *= s
        self.strides = tuple(strides)
        self.addr = addr

    def desc(self):
        d = blkattn.Tensor()
        d.data = self.addr
        d.dtype = {torch.bfloat16: 1, torch.float32: 2, torch.int32: 3, torch.int64: 4}[self.dtype]
        d.ndim = len(self.shape)
        d.device = self.device
        for i, (s, st) in enumerate(zip(self.shape, self.strides)):
            d.sizes[i] = s
            d.strides[i] = st
        return d


def call_fwd(lib, q, k, v, sl, qp, bias, out, lse):
    ds = [None if t is None else t.desc() for t in (q, k, v, sl, qp, bias, out, lse)]
    ref = lambda d: None if d is None else ctypes.byref(d)
    return lib.blkattn_fwd(ref(ds[0]), ref(ds[1]), ref(ds[2]), ref(ds[3]), ref(ds[4]), ref(ds[5]),
                           ctypes.c_float(0.1), ref(ds[6]), ref(ds[7]), None)


def good_args(B=2, Hq=8, Hkv=2, Tq=3, Tmax=100, d=128, dt=torch.bfloat16):
    return dict(
        q=FakeTensor((B, Hq, Tq, d), dt), k=FakeTensor((B, Hkv, Tmax, d), dt),
        v=FakeTensor((B, Hkv, Tmax, d), dt), sl=FakeTensor((B,), torch.int32),
        qp=FakeTensor((B, Tq), torch.int32), bias=None,
        out=FakeTensor((B, Hq, Tq, d), torch.float32), lse=FakeTensor((B, Hq, Tq), torch.float32))


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: a.update(q=FakeTensor((2, 8, 3, 128), torch.int32)), -1),
    (lambda a: a.update(k=FakeTensor((2, 2, 100, 128), torch.float32)), -1),  # mixed q/k dtypes
    (lambda a: a.update(k=FakeTensor((2, 3, 100, 128), torch.bfloat16),
                        v=FakeTensor((2, 3, 100, 128), torch.bfloat16)), -1),  # 8 % 3 != 0
    (lambda a: a.update(v=FakeTensor((2, 2, 99, 128), torch.bfloat16)), -1),
    (lambda a: a.update(qp=FakeTensor((2, 4), torch.int32)), -1),
    (lambda a: a.update(sl=FakeTensor((3,), torch.int32)), -1),
    (lambda a: a.update(sl=FakeTensor((2,), torch.float32)), -1),
    (lambda a: a.update(lse=FakeTensor((2, 8, 3), torch.bfloat16)), -1),
    (lambda a: a.update(out=FakeTensor((2, 8, 3, 64), torch.float32)), -1),
    (lambda a: a.update(k=FakeTensor((2, 2, 100, 128), torch.bfloat16, strides=(25600, 12800, 128, 2))), -1),
    (lambda a: a.update(k=FakeTensor((2, 2, 100, 128), torch.bfloat16, strides=(25600, 12803, 128, 1))), -1),
    (lambda a: a.update(k=FakeTensor((2, 2, 100, 128), torch.bfloat16, addr=0x10008)), -1),  # not 16-B aligned
    (lambda a: a.update(bias=FakeTensor((2, 8, 3, 99), torch.float32)), -1),
    (lambda a: a.update(bias=FakeTensor((2, 2, 3, 100), torch.float32)), -1),
    (lambda a: a.update(bias=FakeTensor((2, 8, 3, 100), torch.bfloat16)), -1),
    (lambda a: a.update(q=FakeTensor((2, 8, 3, 128), torch.bfloat16, addr=0)), -1),  # NULL data
    (lambda a: a.update(**good_args(d=96)), -2),  # head dim without a kernel
    (lambda a: a.update(q=None), -1),
    (lambda a: a.update(k=FakeTensor((2, 2, 100, 128), torch.bfloat16, device=1)), -1),  # device mismatch
    (lambda a: a.update(lse=FakeTensor((2, 8, 3), torch.float32, device=3)), -1),
    (lambda a: a.update(bias=FakeTensor((2, 8, 3, 100), torch.float32, device=1)), -1),
    (lambda a: a.update(**{n: FakeTensor(t.shape, t.dtype, t.strides, device=-1)
                           for n, t in good_args().items() if t is not None}), -1),  # host memory
], ids=["q-int", "mixed-dtype", "hq-not-multiple", "v-len", "qpos-shape", "seqlens-shape",
        "seqlens-dtype", "lse-dtype", "out-dim", "k-inner-stride", "k-row-misaligned",
        "k-base-misaligned", "bias-shape", "bias-heads", "bias-dtype", "null-data", "d96", "missing-q",
        "k-other-device", "lse-other-device", "bias-other-device", "host-memory"])
def test_invalid_requests_are_rejected_before_cuda(lib, mutate, expect):
    a = good_args()
    mutate(a)
    assert call_fwd(lib, a["q"], a["k"], a["v"], a["sl"], a["qp"], a["bias"], a["out"], a["lse"]) == expect


def call_fwd_tree(lib, q, k, v, sl, qp, tree, bias, out, lse):
    ds = [None if t is None else t.desc() for t in (q, k, v, sl, qp, tree, bias, out, lse)]
    ref = lambda d: None if d is None else ctypes.byref(d)
    return lib.blkattn_fwd_tree(*[ref(x) for x in ds[:7]], ctypes.c_float(0.1), ref(ds[7]), ref(ds[8]), None)


@pytest.mark.parametrize("tree,expect", [
    (None, -1),                                                  # the tree is required
    (FakeTensor((2, 3), torch.int32), -1),                       # masks are int64
    (FakeTensor((2, 4), torch.int64), -1),                       # [B, T_q]
    (FakeTensor((3, 3), torch.int64), -1),
    (FakeTensor((2, 3, 1), torch.int64), -1),
    (FakeTensor((2, 3), torch.int64, addr=0), -1),               # NULL data
], ids=["missing", "int32", "tq", "batch", "ndim", "null-data"])
def test_tree_requests_are_validated_before_cuda(lib, tree, expect):
    a = good_args()
    assert call_fwd_tree(lib, a["q"], a["k"], a["v"], a["sl"], a["qp"], tree, None, a["out"], a["lse"]) == expect


def test_tree_needs_at_most_64_rows(lib):
    a = good_args(Tq=65)
    tree = FakeTensor((2, 65), torch.int64)
    assert call_fwd_tree(lib, a["q"], a["k"], a["v"], a["sl"], a["qp"], tree, None, a["out"], a["lse"]) == -1
    e = good_args(B=0)
    for t in e.values():
        if t is not None:
            t.addr = 0
    empty_tree = FakeTensor((0, 3), torch.int64, addr=0)
    assert call_fwd_tree(lib, e["q"], e["k"], e["v"], e["sl"], e["qp"], empty_tree, None, e["out"], e["lse"]) == 0


def call_fwd_window(lib, a, window):
    ds = [None if a[n] is None else a[n].desc() for n in ("q", "k", "v", "sl", "qp", "bias", "out", "lse")]
    ref = lambda d: None if d is None else ctypes.byref(d)
    return lib.blkattn_fwd_window(*[ref(x) for x in ds[:5]], ctypes.c_int64(window), ref(ds[5]),
                                  ctypes.c_float(0.1), ref(ds[6]), ref(ds[7]), None)


@pytest.mark.parametrize("window", [0, -1, -(1 << 40), 1 << 31, 1 << 40],
                         ids=["zero", "negative", "very-negative", "above-int32", "huge"])
def test_window_must_be_a_positive_int32(lib, window):
    a = good_args()
    assert call_fwd_window(lib, a, window) == -1


def test_window_requests_share_the_tensor_checks(lib):
    a = good_args()
    a["qp"] = FakeTensor((2, 4), torch.int32)
    assert call_fwd_window(lib, a, 100) == -1
    a = good_args(d=96)
    assert call_fwd_window(lib, a, 100) == -2
    e = good_args(B=0)
    for t in e.values():
        if t is not None:
            t.addr = 0
    assert call_fwd_window(lib, e, 1) == 0            # empty problem: nothing to do
    assert call_fwd_window(lib, e, (1 << 31) - 1) == 0


def test_window_and_tree_are_exclusive_in_the_binding():
    with pytest.raises(ValueError):
        blkattn.fwd(*([None] * 6), 0.1, None, None, tree=object(), window=4)


def bwd_args(B=2, Hq=8, Hkv=2, Tq=3, Tmax=100, d=128, dt=torch.bfloat16):
    a = good_args(B, Hq, Hkv, Tq, Tmax, d, dt)
    a.update(dout=FakeTensor((B, Hq, Tq, d), dt), dq=FakeTensor((B, Hq, Tq, d), torch.float32),
             dk=FakeTensor((B, Hkv, Tmax, d), torch.float32), dv=FakeTensor((B, Hkv, Tmax, d), torch.float32))
    return a


def call_bwd(lib, a, scale=0.1):
    names = ("q", "k", "v", "sl", "qp", "bias", "out", "lse", "dout", "dq", "dk", "dv")
    ds = [None if a[n] is None else a[n].desc() for n in names]
    ref = lambda d: None if d is None else ctypes.byref(d)
    return lib.blkattn_bwd(*[ref(x) for x in ds[:6]], ctypes.c_float(scale), *[ref(x) for x in ds[6:]], None)


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: a.update(dout=FakeTensor((2, 8, 3, 128), torch.float32)), -1),      # g_o dtype = q dtype
    (lambda a: a.update(dout=FakeTensor((2, 8, 4, 128), torch.bfloat16)), -1),     # g_o shape
    (lambda a: a.update(dq=FakeTensor((2, 8, 3, 128), torch.bfloat16)), -1),       # gradients are f32
    (lambda a: a.update(dk=FakeTensor((2, 2, 99, 128), torch.float32)), -1),       # dk shape
    (lambda a: a.update(dv=FakeTensor((2, 8, 100, 128), torch.float32)), -1),      # dv heads
    (lambda a: a.update(dq=FakeTensor((2, 8, 3, 128), torch.float32, addr=0x10008)), -1),  # not 16-B aligned
    (lambda a: a.update(dk=FakeTensor((2, 2, 100, 128), torch.float32, strides=(25600, 12800, 129, 1))), -1),
    (lambda a: a.update(q=FakeTensor((2, 8, 3, 128), torch.bfloat16, strides=(3072, 384, 130, 1))), -1),
    (lambda a: a.update(dout=None), -1),
    (lambda a: a.update(**bwd_args(d=64)), -2),                                     # d = 64: no backward kernel
    (lambda a: a.update(**bwd_args(dt=torch.float32)), -2),                         # f32: no backward kernel
    (lambda a: a.update(**bwd_args(B=1, Tq=131073)), -2),                           # > 1024 query tiles
    (lambda a: a.update(dk=FakeTensor((2, 2, 100, 128), torch.float32, device=1)), -1),   # device mismatch
    (lambda a: a.update(dout=FakeTensor((2, 8, 3, 128), torch.bfloat16, device=2)), -1),
], ids=["dout-dtype", "dout-shape", "dq-dtype", "dk-shape", "dv-heads", "dq-misaligned", "dk-row-stride",
        "q-row-stride", "missing-dout", "d64", "f32", "too-many-rows", "dk-other-device", "dout-other-device"])
def test_backward_requests_are_validated_before_cuda(lib, mutate, expect):
    a = bwd_args()
    mutate(a)
    assert call_bwd(lib, a) == expect


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), -float("inf")])
def test_backward_needs_a_finite_scale(lib, scale):
    assert call_bwd(lib, bwd_args(), scale) == -1


@pytest.mark.parametrize("window", [0, -3, 1 << 31])
def test_backward_window_must_be_a_positive_int32(lib, window):
    a = bwd_args()
    names = ("q", "k", "v", "sl", "qp", "bias", "out", "lse", "dout", "dq", "dk", "dv")
    ds = [None if a[n] is None else a[n].desc() for n in names]
    ref = lambda d: None if d is None else ctypes.byref(d)
    st = lib.blkattn_bwd_window(*[ref(x) for x in ds[:5]], ctypes.c_int64(window), ref(ds[5]), ctypes.c_float(0.1),
                                *[ref(x) for x in ds[6:]], None)
    assert st == -1


def test_backward_empty_batch_is_a_no_op(lib):
    a = bwd_args(B=0)
    for t in a.values():
        if t is not None:
            t.addr = 0
    assert call_bwd(lib, a) == 0


def call_spec(lib, p, q, draft, ua, us, n, tok):
    ds = [None if t is None else t.desc() for t in (p, q, draft, ua, us, n, tok)]
    ref = lambda d: None if d is None else ctypes.byref(d)
    return lib.blkattn_spec_sample(*[ref(x) for x in ds], None)


def good_spec(B=4, k=3, V=1000):
    return dict(p=FakeTensor((B, k + 1, V), torch.float32), q=FakeTensor((B, k, V), torch.float32),
                draft=FakeTensor((B, k), torch.int32), ua=FakeTensor((B, k), torch.float32),
                us=FakeTensor((B,), torch.int32), n=FakeTensor((B,), torch.int32),
                tok=FakeTensor((B,), torch.int32))


@pytest.mark.parametrize("mutate", [
    lambda a: a.update(p=FakeTensor((4, 4, 1000), torch.bfloat16)),
    lambda a: a.update(q=FakeTensor((4, 4, 1000), torch.float32)),          # k must match
    lambda a: a.update(q=FakeTensor((4, 3, 999), torch.float32)),
    lambda a: a.update(draft=FakeTensor((4, 3), torch.int64)),
    lambda a: a.update(ua=FakeTensor((4, 2), torch.float32)),
    lambda a: a.update(us=FakeTensor((5,), torch.int32)),
    lambda a: a.update(tok=FakeTensor((4,), torch.float32)),
    lambda a: a.update(p=FakeTensor((4, 4, 1000), torch.float32, strides=(8000, 2000, 2))),  # vocab stride
    lambda a: a.update(p=FakeTensor((4, 4, 1000), torch.float32, addr=0)),
    lambda a: a.update(p=None),
    lambda a: a.update(tok=FakeTensor((4,), torch.int32, device=1)),                   # device mismatch
    lambda a: a.update(**{n: FakeTensor(t.shape, t.dtype, t.strides, device=-1) for n, t in good_spec().items()}),
], ids=["p-dtype", "k-mismatch", "vocab", "draft-dtype", "uacc-shape", "usmp-shape", "tok-dtype",
        "vocab-stride", "null-p", "missing-p", "tok-other-device", "host-memory"])
def test_spec_sample_rejects_bad_requests(lib, mutate):
    a = good_spec()
    mutate(a)
    assert call_spec(lib, a["p"], a["q"], a["draft"], a["ua"], a["us"], a["n"], a["tok"]) == -1


def test_spec_sample_empty_batch(lib):
    a = good_spec(B=0)
    for t in a.values():
        t.addr = 0
    assert call_spec(lib, a["p"], a["q"], a["draft"], a["ua"], a["us"], a["n"], a["tok"]) == 0


def test_empty_problem_is_a_no_op(lib):
    a = good_args(B=0)
    for t in a.values():
        if t is not None:
            t.addr = 0
    assert call_fwd(lib, a["q"], a["k"], a["v"], a["sl"], a["qp"], None, a["out"], a["lse"]) == 0
    a = good_args(Tq=0)
    assert call_fwd(lib, a["q"], a["k"], a["v"], a["sl"], a["qp"], None, a["out"], a["lse"]) == 0


def test_merge_rejects_mismatched_states(lib):
    def st(rows, d, stride=None):
        s = blkattn.States()
        s.m, s.l, s.u = 0x1000, None, 0x2000
        s.rows, s.d_v, s.u_row_stride = rows, d, stride or d
        return s
    a, b = st(4, 8), st(5, 8)
    assert lib.blkattn_merge(ctypes.byref(a), ctypes.byref(b), ctypes.byref(a), None) == -1
    a, b = st(4, 8), st(4, 8, stride=4)
    assert lib.blkattn_merge(ctypes.byref(a), ctypes.byref(b), ctypes.byref(a), None) == -1
    z = st(0, 8)
    assert lib.blkattn_merge(ctypes.byref(z), ctypes.byref(z), ctypes.byref(z), None) == 0


def _check_partition(p, Tmax):
    chunk, n = p["chunk_keys"], p["n_splits"]
    assert chunk % p["tile_keys"] == 0 and chunk > 0
    # consecutive chunks [s*chunk, min((s+1)*chunk, Tmax)) cover [0, Tmax) exactly once
    covered = []
    for s in range(n):
        lo, hi = s * chunk, min((s + 1) * chunk, Tmax)
        assert lo < hi
        covered.extend(range(lo, hi))
    assert covered == list(range(Tmax))


def _check_tc_decode_plan(p, B, Hq, Hkv, Tq, d, sms):
    rows = (Hq // Hkv) * Tq
    rg = math.ceil(rows / 48)
    R = math.ceil(rows / rg)
    assert p["kernel"] == 3 and p["tile_keys"] == 128 and p["chunk_keys"] == 0
    assert p["row_groups"] == rg and p["rows_per_cta"] == R <= 48
    assert p["ctas"] == sms  # one persistent CTA per SM
    units = B * Hkv * rg
    assert p["n_splits"] == sms + units  # workspace slots: CTA index + unit index
    slots = p["n_splits"]
    assert p["workspace_bytes"] >= slots * R * (d + 2) * 4


@pytest.mark.parametrize("name", list(workloads.SPECS))
def test_plan_partitions_every_workload(lib, name):
    for small in (False, True):
        s = workloads.spec(name, small)
        p = blkattn.debug_plan(s.B, s.Hq, s.Hkv, s.Tq, s.Tmax, s.d,
                               torch.bfloat16 if s.dtype == "bf16" else torch.float32, 152)
        rows = s.G * s.Tq
        if s.dtype == "bf16" and s.Tq >= 64 and s.d == 128:
            assert p["kernel"] == 2 and p["rows_per_cta"] == 256 and p["n_splits"] == 1
            assert p["row_groups"] == math.ceil(s.Tq / 256)
            assert p["ctas"] == p["row_groups"] * s.Hq * s.B
            continue
        if s.dtype == "bf16" and s.d == 128:
            _check_tc_decode_plan(p, s.B, s.Hq, s.Hkv, s.Tq, s.d, 152)
            continue
        _check_partition(p, s.Tmax)
        if s.dtype == "bf16":
            assert p["kernel"] == 1 and p["rows_per_cta"] in (16, 32, 48)
        else:
            assert p["kernel"] == 0 and p["rows_per_cta"] in (1, 2, 4, 8)
        assert p["row_groups"] == math.ceil(rows / p["rows_per_cta"])
        assert p["ctas"] == p["n_splits"] * s.Hkv * s.B * p["row_groups"]
        if p["n_splits"] > 1:
            assert p["workspace_bytes"] >= s.B * s.Hq * s.Tq * p["n_splits"] * (s.d + 2) * 4
        else:
            assert p["workspace_bytes"] == 0


def test_plan_random_shapes(lib):
    g = torch.Generator().manual_seed(0)
    for _ in range(300):
        B = int(torch.randint(1, 40, (1,), generator=g))
        Hkv = int(torch.randint(1, 9, (1,), generator=g))
        G = int(torch.randint(1, 9, (1,), generator=g))
        Tq = int(torch.randint(1, 20, (1,), generator=g))
        Tmax = int(torch.randint(1, 300000, (1,), generator=g))
        sms = int(torch.randint(1, 200, (1,), generator=g))
        d = 64 if int(torch.randint(0, 2, (1,), generator=g)) else 128
        p = blkattn.debug_plan(B, Hkv * G, Hkv, Tq, Tmax, d, torch.bfloat16, sms)
        if d == 128:
            _check_tc_decode_plan(p, B, Hkv * G, Hkv, Tq, d, sms)
        else:
            assert p["kernel"] == 1
            _check_partition(p, Tmax)


def test_plan_large_batches_leave_the_tc_decode_kernel(lib):
    # the (sequence, row group) table of the tcgen05 decode kernel holds 1024 entries
    assert blkattn.debug_plan(1024, 8, 8, 1, 4096, 128, torch.bfloat16, 152)["kernel"] == 3
    assert blkattn.debug_plan(1025, 8, 8, 1, 4096, 128, torch.bfloat16, 152)["kernel"] == 1
    assert blkattn.debug_plan(512, 64, 1, 1, 4096, 128, torch.bfloat16, 152)["kernel"] == 3  # 2 row groups
    assert blkattn.debug_plan(513, 64, 1, 1, 4096, 128, torch.bfloat16, 152)["kernel"] == 1
    assert blkattn.debug_plan(1, 8, 8, 1, 65535 * 128 + 1, 128, torch.bfloat16, 152)["kernel"] == 1


def test_plan_rejects_bad_shapes(lib):
    with pytest.raises(ValueError):
        blkattn.debug_plan(1, 6, 4, 1, 100, 128)
    with pytest.raises(ValueError):
        blkattn.debug_plan(1, 4, 4, 1, 0, 128)


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "exact_blocked_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "attention_oracle" not in text, f
