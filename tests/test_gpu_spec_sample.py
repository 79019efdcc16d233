"""The speculative-sampling step (blkattn_spec_sample) against the oracle
(oracle/spec_sampling.py, pinned to Chapter 33 §33.5): the kept-candidate
counts and the emitted tokens are integers decided the same way on both
sides, so they must match exactly."""
import numpy as np
import pytest
import torch

from exact_blocked_attention_gb300 import blkattn, workloads
from exact_blocked_attention_gb300 import build as libbuild
from oracle import spec_sampling as ss

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    blkattn.load()


def run_both(p, q, draft, u_acc, u_smp):
    dev = [t.cuda() for t in (p, q, draft, u_acc, u_smp)]
    n, tok = blkattn.spec_sample(*dev)
    torch.cuda.synchronize()
    on, ot = ss.verify_step(p.numpy(), q.numpy(), draft.numpy(), u_acc.numpy(),
                            u_smp.numpy().view(np.uint32))
    return n.cpu().numpy(), tok.cpu().numpy(), on, ot


@pytest.mark.parametrize("small", [True, False])
def test_workload_matches_oracle(small):
    g = workloads.generate_sampling(workloads.sample_spec("spec_sample", small))
    n, tok, on, ot = run_both(g["p"], g["q"], g["draft"], g["u_accept"], g["u_sample"])
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(tok, ot)
    assert len(set(n.tolist())) > 1  # the workload exercises several outcomes


def random_case(B, k, V, seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, k + 1)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, k)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
    u = rng.random((B, k), dtype=np.float32)
    s = rng.integers(0, 2**32, size=B, dtype=np.uint64).astype(np.uint32).view(np.int32)
    return [torch.from_numpy(np.ascontiguousarray(a)) for a in (p, q, draft, u, s)]


@pytest.mark.parametrize("B,k,V", [(9, 0, 37), (33, 1, 5), (17, 2, 33), (5, 6, 65537), (64, 3, 1)])
def test_random_shapes(B, k, V):
    n, tok, on, ot = run_both(*random_case(B, k, V, seed=B * 1000 + k * 10 + V))
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(tok, ot)


def test_degenerate_cases():
    V = 40
    B, k = 5, 2
    p = np.full((B, k + 1, V), 1.0 / V, dtype=np.float32)
    q = np.full((B, k, V), 1.0 / V, dtype=np.float32)
    draft = np.full((B, k), 3, dtype=np.int32)
    u = np.full((B, k), 0.75, dtype=np.float32)
    # row 0: a rejection that meets a zero residual (mass below 2^-40 only):
    # the candidate is kept, so both are kept
    q[0, 0, 3] = 2.0**-30; p[0, 0, 3] = 2.0**-31
    q[0, 0, 7] = 2.0**-45; p[0, 0, 7] = 2.0**-45 + 2.0**-50
    # row 1: a candidate outside the vocabulary is rejected
    draft[1, 0] = V
    # row 2: a candidate the draft gives no probability is rejected
    q[2, 0, 3] = 0.0
    # row 3: every candidate kept and the next target has no mass: token 0
    p[3, k] = 0.0
    # row 4: a negative candidate is rejected
    draft[4, 1] = -1
    t = [torch.from_numpy(a) for a in (p, q, draft, u)]
    s = torch.from_numpy(np.array([1, 2**31 - 1, -5, 7, 123456], dtype=np.int32))
    n, tok, on, ot = run_both(*t, s)
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(tok, ot)
    assert n[0] == 2 and n[1] == 0 and n[2] == 0 and n[3] == 2 and tok[3] == 0 and n[4] == 1


def test_strided_views():
    p, q, draft, u, s = random_case(7, 3, 300, seed=5)
    big_p = torch.zeros(7, 6, 300); big_p[:, 1:5] = p      # non-contiguous along k
    big_q = torch.zeros(9, 3, 300); big_q[1:8] = q
    n, tok = blkattn.spec_sample(big_p[:, 1:5].cuda(), big_q[1:8].cuda(), draft.cuda(), u.cuda(), s.cuda())
    pv = big_p.cuda()[:, 1:5]
    qv = big_q.cuda()[1:8]
    n2, tok2 = blkattn.spec_sample(pv, qv, draft.cuda(), u.cuda(), s.cuda())
    torch.cuda.synchronize()
    on, ot = ss.verify_step(p.numpy(), q.numpy(), draft.numpy(), u.numpy(), s.numpy().view(np.uint32))
    for a, b_ in ((n, tok), (n2, tok2)):
        np.testing.assert_array_equal(a.cpu().numpy(), on)
        np.testing.assert_array_equal(b_.cpu().numpy(), ot)


def rounded_residual_token(p_row, q_row, s):
    """The token a residual rounded to fp32 before F would give (a planted
    mistake, used only to show that the rows below discriminate)."""
    m = (np.asarray(p_row, np.float32) - np.asarray(q_row, np.float32)).astype(np.float64)
    return ss.inverse_cdf(ss.fixed(m), s)


def adversarial_rows(B, k, V, seed):
    """Rows whose first candidate is rejected (its p is 0) and whose 32-bit
    draw sits where the exact residual of eq. 33.12 and the fp32-rounded one
    emit different tokens."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, k + 1)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, k)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
    u = rng.random((B, k), dtype=np.float32)
    s = np.zeros(B, dtype=np.uint64)
    for b in range(B):
        x = int(draft[b, 0])
        p[b, 0, x] = 0.0
        q[b, 0, x] = max(q[b, 0, x], np.float32(1e-3))
        w = ss.weights(p[b, 0], q[b, 0])
        wr = ss.fixed((p[b, 0] - q[b, 0]).astype(np.float64))
        Z, Zr = int(w.sum()), int(wr.sum())
        C, Cr = np.cumsum(w), np.cumsum(wr)
        # first draw past each token boundary, exact and rounded
        first = [-(-(int(c) << 32) // Z) for c in C[:-1]]
        first_r = [-(-(int(c) << 32) // Zr) for c in Cr[:-1]]
        cand = [min(a, c) for a, c in zip(first, first_r) if a != c and min(a, c) < 2**32]
        assert cand, "no discriminating draw in this row"
        s[b] = cand[int(rng.integers(len(cand)))]
        assert ss.inverse_cdf(w, int(s[b])) != rounded_residual_token(p[b, 0], q[b, 0], int(s[b]))
    return [torch.from_numpy(np.ascontiguousarray(a)) for a in (p, q, draft, u, s.astype(np.uint32).view(np.int32))]


@pytest.mark.parametrize("B,k,V", [(32, 2, 5000), (8, 4, 128256)])
def test_residual_is_drawn_from_the_exact_difference(B, k, V):
    """Eq. 33.12's [p - q]_+ is the exact difference: on rows where rounding
    it changes the token, the kernel emits the exact residual's token."""
    n, tok, on, ot = run_both(*adversarial_rows(B, k, V, seed=V + k))
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(tok, ot)
    assert np.all(n == 0)


def test_unaligned_rows_take_plain_loads():
    """Rows that do not start on a 16-byte boundary are read with plain loads
    (no bulk copies); the results are the same integers."""
    p, q, draft, u, s = random_case(6, 2, 5003, seed=9)
    bp = torch.zeros(6 * 3 * 5003 + 1)
    bp[1:] = p.reshape(-1)
    bq = torch.zeros(6 * 2 * 5003 + 3)
    bq[3:] = q.reshape(-1)
    pv = bp.cuda()[1:].view(6, 3, 5003)  # 4-byte offsets: not 16-byte aligned
    qv = bq.cuda()[3:].view(6, 2, 5003)
    n, tok = blkattn.spec_sample(pv, qv, draft.cuda(), u.cuda(), s.cuda())
    torch.cuda.synchronize()
    on, ot = ss.verify_step(p.numpy(), q.numpy(), draft.numpy(), u.numpy(), s.numpy().view(np.uint32))
    np.testing.assert_array_equal(n.cpu().numpy(), on)
    np.testing.assert_array_equal(tok.cpu().numpy(), ot)


def test_vocabulary_beyond_the_recorded_chunks():
    """A vocabulary of 1.3 M entries: each CTA's half spans more ring slots
    than it records sums for, so chunks hold several slots and the last
    scan covers a whole chunk."""
    n, tok, on, ot = run_both(*random_case(3, 1, 1300003, seed=77))
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(tok, ot)


def test_more_candidates_than_a_warp_tests_at_once():
    """k = 40 candidates: the first 35 positions have p = q (always kept for
    u < 1), so the in-order test runs past the first 32 candidates."""
    B, k, V = 4, 40, 777
    p, q, draft, u, s = [t.numpy().copy() for t in random_case(B, k, V, seed=41)]
    for b in range(B):
        for i in range(35):
            q[b, i] = p[b, i]
            draft[b, i] = int(np.argmax(q[b, i]))  # a proposable candidate (q > 0)
    n, tok, on, ot = run_both(*[torch.from_numpy(np.ascontiguousarray(a)) for a in (p, q, draft, u, s)])
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(tok, ot)
    assert np.all(n >= 35)


def test_masses_outside_the_unit_interval():
    """Rows of a full-size vocabulary with a few masses outside [0, 1] (-0,
    negatives, above 1 and 2, NaN, inf) among ordinary ones: the slots holding
    them take the clamped form of the weights, the others the short form, and
    the draw is the oracle's."""
    B, k, V = 8, 2, 128256
    rng = np.random.default_rng(11)
    p = rng.dirichlet(np.ones(V) * 0.5, size=(B, k + 1)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=(B, k)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, k)).astype(np.int32)
    u = rng.random((B, k), dtype=np.float32)
    odd = np.array([-0.0, -1e-3, 1.5, 3.0, np.nan, np.inf, -np.inf, 2.0, 1.0000001], dtype=np.float32)
    for b in range(B):
        if b >= 5:  # every candidate kept: the next target row is drawn from
            u[b] = 0.0
            for i in range(k):
                p[b, i, draft[b, i]] = max(p[b, i, draft[b, i]], np.float32(1e-6))
                q[b, i, draft[b, i]] = max(q[b, i, draft[b, i]], np.float32(1e-6))
        else:  # the first candidate is rejected: its residual is drawn from
            p[b, 0, draft[b, 0]] = 0.0
            q[b, 0, draft[b, 0]] = max(q[b, 0, draft[b, 0]], np.float32(1e-3))
        if b % 2 == 0:
            continue  # even rows stay in range
        for j, x in enumerate(rng.choice(V, size=6, replace=False)):
            if x != draft[b, 0]:
                (p if j % 2 == 0 else q)[b, 0, x] = odd[(b + j) % len(odd)]
        p[b, k, rng.integers(V)] = odd[b % len(odd)]
    s = rng.integers(0, 2**32, size=B, dtype=np.uint64).astype(np.uint32).view(np.int32)
    t = [torch.from_numpy(np.ascontiguousarray(a)) for a in (p, q, draft, u, s)]
    n, tok, on, ot = run_both(*t)
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(tok, ot)
    assert np.all(n[:5] == 0) and np.all(n[5:] == k)


def test_a_captured_step_replays_on_new_data():
    """The verification step captured once in a CUDA graph and replayed on new
    distributions, candidates and random numbers written into the same
    buffers: every replay decides as the oracle does on that data."""
    B, k, V = 16, 3, 20000
    t = [x.cuda() for x in random_case(B, k, V, seed=1)]
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    call = lambda: blkattn.spec_sample(*t, n, tok)
    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call()
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(3):
        new = random_case(B, k, V, seed=100 + rep)
        for dst, src in zip(t, new):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        on, ot = ss.verify_step(new[0].numpy(), new[1].numpy(), new[2].numpy(), new[3].numpy(),
                                new[4].numpy().view(np.uint32))
        np.testing.assert_array_equal(n.cpu().numpy(), on)
        np.testing.assert_array_equal(tok.cpu().numpy(), ot)
