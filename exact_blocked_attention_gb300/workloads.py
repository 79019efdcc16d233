"""Seeded synthetic inputs for the attention workloads.

This module only draws numbers: shapes, value distributions, cache lengths,
logical positions and mask patterns.  It holds none of the attention
arithmetic, and it is the one module that both the CUDA path's callers and the
oracle's callers share.  Everything is generated on the CPU from fixed seeds
(numpy PCG64, split into a fixed number of independent streams so that the
result does not depend on the thread count), then cast to the workload dtype.

Workloads (the problem statement of "Chapter 33: inference compute
optimisation" §33.2: single-head Q [T_q, d_h], K [T_k, d_h], V [T_k, d_v], an
additive bias M_j, grouped heads, and the cached-decoding positions of
"Generation and Caching with the Same Model"):

  tiny_fp32     1 seq, 1 head, d=64, T_q=1 at position T_k-1, T_k=1000, fp32
  decode_gqa    batch 32, 32 query / 8 KV heads, d=128, T_q=1, cache lengths
                uniform in [512, 8192], query at len-1, bf16
  long_decode   batch 1, 32/8 heads, d=128, T_q=1, T_k=131072, 1% of key
                positions scaled x3 (sharp maxima), bf16
  spec_verify   batch 8, 64/8 heads, d=128, T_q=5 rows at L..L+4 (L uniform in
                [1024, 32768], cache length L+5), a {0,-inf} bias that masks
                random 128-key blocks of 10% of the sequences and every key of
                1% of the (sequence, row) pairs, bf16
  prefill       batch 2, 32 heads (MHA), d=128, T_q=T_k=8192, row i at i, bf16
  window_decode batch 16, 32/8 heads, d=128, T_q=1 at len-1, cache lengths
                uniform in [8192, 16384], a sliding window of 4096 keys
                ("Chapter 33" §33.7, the paragraph of eq. 33.16), bf16
  window_prefill prefill's shapes (B=2, 32 heads, T=8192, causal) with a sliding
                window of 1024 keys, bf16
  tree_verify   spec_verify's batch, heads, cache lengths and values with a
                token tree of T_q=6 draft nodes per sequence ("推理加速算法"
                §7.2.2 Medusa, tree attention verification): seeded random
                parents, every row at len-1 and the tree region shaped by
                ancestor masks, no bias

Each has a reduced twin (``small=True``) that the fp64 oracle finishes in
seconds while still spanning several key tiles and a ragged tail.

The backward workload (§33.3, eqs. 33.6-33.8) is prefill's inputs plus an
upstream gradient g_o drawn like q (N(0, 1), cast to bf16).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np
import torch

_STREAMS = 64  # independent generator streams per array (fixed, thread-count free)


@dataclass(frozen=True)
class Spec:
    name: str
    B: int
    Hq: int
    Hkv: int
    Tq: int
    Tmax: int
    d: int
    dtype: str                   # "bf16" or "f32"
    lens: tuple                  # ("fixed", n) | ("uniform", lo, hi) | ("verify", lo, hi)
    pos: str                     # "last" | "verify" | "causal"
    seed: int
    sharp_frac: float = 0.0      # fraction of key positions whose K is scaled
    sharp_gain: float = 1.0
    bias: str = "none"           # "none" | "verify_blocks"
    bias_seq_frac: float = 0.0
    bias_block: int = 128
    bias_block_frac: float = 0.0
    masked_row_frac: float = 0.0
    tree: str = "none"           # "none" | "random" (token tree of T_q nodes per sequence)
    window: int = 0              # sliding window of keys (0: none)
    notes: str = field(default="", compare=False)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


SPECS = {
    "tiny_fp32": Spec("tiny_fp32", 1, 1, 1, 1, 1000, 64, "f32", ("fixed", 1000), "last", 0),
    "decode_gqa": Spec("decode_gqa", 32, 32, 8, 1, 8192, 128, "bf16", ("uniform", 512, 8192), "last", 1),
    "long_decode": Spec("long_decode", 1, 32, 8, 1, 131072, 128, "bf16", ("fixed", 131072), "last", 2,
                        sharp_frac=0.01, sharp_gain=3.0),
    "spec_verify": Spec("spec_verify", 8, 64, 8, 5, 32776, 128, "bf16", ("verify", 1024, 32768), "verify", 3,
                        bias="verify_blocks", bias_seq_frac=0.10, bias_block=128, bias_block_frac=0.10,
                        masked_row_frac=0.01),
    "prefill": Spec("prefill", 2, 32, 32, 8192, 8192, 128, "bf16", ("fixed", 8192), "causal", 5),
    # spec_verify's seed: the same cache lengths and values, a 6-node tree in
    # place of the 5-row chain and the bias
    "tree_verify": Spec("tree_verify", 8, 64, 8, 6, 32774, 128, "bf16", ("verify", 1024, 32768), "tree", 3,
                        tree="random"),
    "window_decode": Spec("window_decode", 16, 32, 8, 1, 16384, 128, "bf16", ("uniform", 8192, 16384), "last", 8,
                          window=4096),
    "window_prefill": Spec("window_prefill", 2, 32, 32, 8192, 8192, 128, "bf16", ("fixed", 8192), "causal", 9,
                           window=1024),
}

# Reduced twins: same structure, sizes the fp64 oracle covers in seconds, still
# several 64/128-key tiles per split and a ragged tail.
SMALL = {
    "tiny_fp32": SPECS["tiny_fp32"],
    "decode_gqa": replace(SPECS["decode_gqa"], B=3, Hq=8, Hkv=2, Tmax=1000, lens=("uniform", 1, 1000)),
    "long_decode": replace(SPECS["long_decode"], B=1, Hq=8, Hkv=2, Tmax=5003, lens=("fixed", 5003)),
    "spec_verify": replace(SPECS["spec_verify"], B=3, Hq=16, Hkv=2, Tmax=1290,
                           lens=("verify", 300, 1285), bias_seq_frac=0.34, masked_row_frac=0.07),
    "prefill": replace(SPECS["prefill"], B=1, Hq=2, Hkv=2, Tq=333, Tmax=333, lens=("fixed", 333)),
    "tree_verify": replace(SPECS["tree_verify"], B=3, Hq=16, Hkv=2, Tmax=1290, lens=("verify", 300, 1284)),
    "window_decode": replace(SPECS["window_decode"], B=3, Hq=8, Hkv=2, Tmax=1500, lens=("uniform", 200, 1500),
                             window=333),
    "window_prefill": replace(SPECS["window_prefill"], B=1, Hq=2, Hkv=2, Tq=333, Tmax=333, lens=("fixed", 333),
                              window=100),
}


def spec(name: str, small: bool = False) -> Spec:
    return (SMALL if small else SPECS)[name]


def _normal(shape, seed: int, tag: int) -> np.ndarray:
    """Standard normal float32 array, deterministic for (seed, tag)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    kids = np.random.SeedSequence([seed, tag]).spawn(_STREAMS)
    bounds = np.linspace(0, n, _STREAMS + 1).astype(np.int64)

    def fill(i):
        g = np.random.Generator(np.random.PCG64(kids[i]))
        g.standard_normal(out=out[bounds[i]:bounds[i + 1]], dtype=np.float32)

    with ThreadPoolExecutor(8) as ex:
        list(ex.map(fill, range(_STREAMS)))
    return out.reshape(shape)


def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(a)
    return t.to(torch.bfloat16) if dtype == "bf16" else t.clone()


def generate(s: Spec, poison_padding: float | None = None) -> dict:
    """Draw one batch of inputs for workload ``s`` on the CPU.

    Returns q, k, v (torch, bf16 or f32), seqlens int32 [B], qpos int32 [B,T_q],
    bias (float32 [B,1,T_q,T_max] or None), tree (int64 [B,T_q] node masks or
    None), scale, and the spec.  Cache rows
    at or beyond a sequence's length are drawn like the rest unless
    ``poison_padding`` is given (e.g. float('nan')), in which case they hold it.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([s.seed, 99])))
    kind = s.lens[0]
    if kind == "fixed":
        lens = np.full(s.B, s.lens[1], dtype=np.int64)
    elif kind == "uniform":
        lens = rng.integers(s.lens[1], s.lens[2] + 1, size=s.B)
    elif kind == "verify":
        # history L uniform in [lo, hi]; the cache also holds the T_q new rows
        L = rng.integers(s.lens[1], s.lens[2] + 1, size=s.B)
        lens = L + s.Tq
    else:
        raise ValueError(kind)
    lens = np.minimum(lens, s.Tmax)

    if s.pos == "last":
        qpos = (lens - 1)[:, None] + np.zeros((1, s.Tq), dtype=np.int64)
    elif s.pos == "verify":
        qpos = (lens - s.Tq)[:, None] + np.arange(s.Tq)[None, :]
    elif s.pos == "causal":
        qpos = np.broadcast_to(np.arange(s.Tq)[None, :], (s.B, s.Tq)).copy()
    elif s.pos == "tree":  # the whole cache; the tree masks shape the tree region
        qpos = (lens - 1)[:, None] + np.zeros((1, s.Tq), dtype=np.int64)
    else:
        raise ValueError(s.pos)

    q = _normal((s.B, s.Hq, s.Tq, s.d), s.seed, 1)
    k = _normal((s.B, s.Hkv, s.Tmax, s.d), s.seed, 2)
    v = _normal((s.B, s.Hkv, s.Tmax, s.d), s.seed, 3)
    if s.sharp_frac > 0:
        n_sharp = int(round(s.sharp_frac * s.Tmax))
        sharp = rng.choice(s.Tmax, size=n_sharp, replace=False)
        k[:, :, sharp, :] *= s.sharp_gain
    if poison_padding is not None:
        for b in range(s.B):
            k[b, :, lens[b]:, :] = poison_padding
            v[b, :, lens[b]:, :] = poison_padding

    bias = None
    if s.bias == "verify_blocks":
        bias = np.zeros((s.B, 1, s.Tq, s.Tmax), dtype=np.float32)
        n_seq = max(1, math.ceil(s.bias_seq_frac * s.B))
        for b in rng.choice(s.B, size=n_seq, replace=False):
            n_blocks = math.ceil(lens[b] / s.bias_block)
            n_mask = max(1, math.ceil(s.bias_block_frac * n_blocks))
            for blk in rng.choice(n_blocks, size=n_mask, replace=False):
                bias[b, 0, :, blk * s.bias_block:(blk + 1) * s.bias_block] = -np.inf
        n_rows = max(1, math.ceil(s.masked_row_frac * s.B * s.Tq))
        for flat in rng.choice(s.B * s.Tq, size=n_rows, replace=False):
            bias[flat // s.Tq, 0, flat % s.Tq, :] = -np.inf

    tree = None
    if s.tree == "random":
        # per sequence a tree of T_q nodes: node 0 the root, node k's parent
        # uniform over the earlier nodes; bit k of a row's mask = node k is
        # the row's node or one of its ancestors
        tree = np.zeros((s.B, s.Tq), dtype=np.int64)
        for b in range(s.B):
            parent = [-1] + [int(rng.integers(0, k)) for k in range(1, s.Tq)]
            for i in range(s.Tq):
                m, node = 0, i
                while node >= 0:
                    m |= 1 << node
                    node = parent[node]
                tree[b, i] = m - (1 << 64) if m >= 1 << 63 else m
    elif s.tree != "none":
        raise ValueError(s.tree)

    return {
        "q": _cast(q, s.dtype),
        "k": _cast(k, s.dtype),
        "v": _cast(v, s.dtype),
        "seqlens": torch.from_numpy(lens.astype(np.int32)),
        "qpos": torch.from_numpy(qpos.astype(np.int32)),
        "bias": None if bias is None else torch.from_numpy(bias),
        "tree": None if tree is None else torch.from_numpy(tree),
        "window": s.window,
        "scale": s.scale,
        "spec": s,
    }


def kv_bytes(s: Spec, seqlens) -> int:
    """Algorithmic K+V bytes one call reads: the visible cache rows of every
    (sequence, KV head), each read once."""
    elt = 2 if s.dtype == "bf16" else 4
    lens = np.minimum(np.asarray(seqlens, dtype=np.int64), s.Tmax)
    if s.window and s.pos == "last":  # rows at len - 1 see only the last `window` keys
        lens = np.minimum(lens, s.window)
    return int(lens.sum()) * s.Hkv * s.d * elt * 2


# ---------------------------------------------------------------- speculative sampling
def backward_spec(small: bool = False) -> Spec:
    """Shapes of the backward workload: the causal prefill's."""
    return spec("prefill", small)


def generate_backward(s: Spec) -> dict:
    """generate(s) plus the upstream gradient "go" [B, H_q, T_q, d]."""
    inp = generate(s)
    inp["go"] = _cast(_normal((s.B, s.Hq, s.Tq, s.d), s.seed, 21), s.dtype)
    return inp


# One verification step ("Chapter 33: inference compute optimisation" §33.5,
# eqs. 33.10-33.13): target and draft distributions over a vocabulary, the
# draft's candidates, and the random numbers of the step.  The draft's logits
# are the target's plus Gaussian noise, so that acceptance is neither certain
# nor rare.

@dataclass(frozen=True)
class SampleSpec:
    name: str
    B: int          # sequences
    k: int          # candidates per sequence
    V: int          # vocabulary
    seed: int
    noise: float    # std of the draft's logit perturbation
    temp: float = 1.0


SAMPLE_SPECS = {
    "spec_sample": SampleSpec("spec_sample", 64, 4, 128256, 7, 1.0),
}
SAMPLE_SMALL = {
    "spec_sample": SampleSpec("spec_sample", 16, 3, 1000, 7, 1.0),
}


def sample_spec(name: str, small: bool = False) -> SampleSpec:
    return (SAMPLE_SMALL if small else SAMPLE_SPECS)[name]


def generate_sampling(s: SampleSpec) -> dict:
    """p f32 [B,k+1,V], q f32 [B,k,V] (softmax rows), draft int32 [B,k] drawn
    from q, u_accept f32 [B,k] in [0,1), u_sample int32 [B] (32 random bits)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([s.seed, 98])))
    z = _normal((s.B, s.k + 1, s.V), s.seed, 11) * 3.0
    zq = z[:, :s.k] + _normal((s.B, s.k, s.V), s.seed, 12) * s.noise

    def softmax(a):
        a = a / s.temp
        a = a - a.max(axis=-1, keepdims=True)
        e = np.exp(a.astype(np.float64))
        return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)

    p = softmax(z)
    q = softmax(zq)
    draft = np.zeros((s.B, s.k), dtype=np.int32)
    for b in range(s.B):
        for i in range(s.k):
            c = np.cumsum(q[b, i].astype(np.float64))
            draft[b, i] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), s.V - 1)
    u_accept = rng.random((s.B, s.k), dtype=np.float32)
    u_sample = rng.integers(0, 2**32, size=s.B, dtype=np.uint64).astype(np.uint32).view(np.int32)
    return {"p": torch.from_numpy(p), "q": torch.from_numpy(q), "draft": torch.from_numpy(draft),
            "u_accept": torch.from_numpy(u_accept), "u_sample": torch.from_numpy(u_sample.copy()), "spec": s}
