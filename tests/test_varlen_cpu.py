"""Variable-length batches on the CPU: the oracle's varlen wrapper pinned to a
brute-force packed formulation, and the host copy of the planning kernel's
task list (coverage, order, bounds).  No CUDA call."""
import itertools

import numpy as np
import pytest

import oracle
import synthetic


# ---------------------------------------------------------------------------
# oracle
# ---------------------------------------------------------------------------

def packed_bruteforce(q, k, v, cu_q, cu_k, causal, scale):
    """Attention over the packed rows with an explicit mask: query row t sees
    key u iff both lie in the same sequence b and, under the causal mask,
    u - k0 <= (t - q0) + sk - sq (bottom-right inside the sequence).  A row
    that sees no key gets O = 0, LSE = -inf.  Plain float64 numpy, the whole
    score matrix at once."""
    total_q, Hq, _ = q.shape
    total_k, Hkv, dv = v.shape
    seq_q = np.full(total_q, -1)
    seq_k = np.full(total_k, -1)
    for b in range(len(cu_q) - 1):
        seq_q[cu_q[b]:cu_q[b + 1]] = b
        seq_k[cu_k[b]:cu_k[b + 1]] = b
    t = np.arange(total_q)[:, None]
    u = np.arange(total_k)[None, :]
    same = (seq_q[:, None] == seq_k[None, :]) & (seq_q[:, None] >= 0)
    mask = same.copy()
    if causal:
        bq = np.maximum(seq_q, 0)
        q0 = np.asarray(cu_q)[bq][:, None]
        sq = (np.asarray(cu_q)[bq + 1] - np.asarray(cu_q)[bq])[:, None]
        k0 = np.asarray(cu_k)[bq][:, None]
        sk = (np.asarray(cu_k)[bq + 1] - np.asarray(cu_k)[bq])[:, None]
        mask &= (u - k0) <= (t - q0) + sk - sq
    o = np.zeros((total_q, Hq, dv))
    lse = np.full((Hq, total_q), -np.inf)
    ratio = Hq // Hkv
    for h in range(Hq):
        s = scale * (q[:, h, :] @ k[:, h // ratio, :].T)
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        has = np.isfinite(m[:, 0])
        e = np.where(mask, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)
        l = e.sum(axis=1)
        o[has, h, :] = (e[has] @ v[:, h // ratio, :]) / l[has, None]
        lse[h, has] = m[has, 0] + np.log(l[has])
    return o, lse


CASES = [
    # seqlens_q, seqlens_k, Hq, Hkv, causal
    ((5, 0, 12, 1), (7, 3, 0, 4), 4, 2, True),
    ((5, 0, 12, 1), (7, 3, 0, 4), 4, 2, False),
    ((9, 9, 9), (4, 13, 9), 2, 1, True),
    ((1,), (1,), 1, 1, True),
    ((6, 3), (2, 8), 3, 3, False),
]


@pytest.mark.parametrize("case", CASES)
def test_oracle_varlen_equals_packed_bruteforce(case):
    lq, lk, Hq, Hkv, causal = case
    rng = np.random.default_rng(sum(lq) * 7 + sum(lk))
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(int)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(int)
    d, dv = 8, 6
    q = rng.standard_normal((cu_q[-1], Hq, d))
    k = rng.standard_normal((cu_k[-1], Hkv, d))
    v = rng.standard_normal((cu_k[-1], Hkv, dv))
    scale = 0.4
    o, lse = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, causal=causal, scale=scale, threads=2)
    ob, lb = packed_bruteforce(q, k, v, cu_q, cu_k, causal, scale)
    assert np.array_equal(np.isinf(lse), np.isinf(lb))
    fin = np.isfinite(lb)
    assert np.allclose(lse[fin], lb[fin], atol=1e-12, rtol=0)
    assert np.allclose(o, ob, atol=1e-12, rtol=0)
    # sampled rows agree with the full call
    rows = np.array([[t, h] for t in range(cu_q[-1]) for h in range(Hq)][::3])
    ro, rl = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, causal=causal, scale=scale, rows=rows, threads=2)
    assert np.allclose(ro, o[rows[:, 0], rows[:, 1]], atol=0, rtol=0)
    assert np.array_equal(rl, lse[rows[:, 1], rows[:, 0]])


def test_oracle_varlen_equal_lengths_is_the_batched_problem():
    B, S, Hq, Hkv, d = 3, 11, 4, 2, 8
    rng = np.random.default_rng(3)
    q = rng.standard_normal((B, S, Hq, d))
    k = rng.standard_normal((B, S + 2, Hkv, d))
    v = rng.standard_normal((B, S + 2, Hkv, d))
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal=causal, threads=2)
        cu_q = np.arange(B + 1) * S
        cu_k = np.arange(B + 1) * (S + 2)
        ov, lv = oracle.attn_fwd_varlen(q.reshape(B * S, Hq, d), k.reshape(-1, Hkv, d), v.reshape(-1, Hkv, d),
                                        cu_q, cu_k, causal=causal, threads=2)
        assert np.array_equal(ov.reshape(B, S, Hq, d), o)
        assert np.array_equal(lv.reshape(Hq, B, S).transpose(1, 0, 2), lse)


def test_oracle_varlen_rows_outside_sequences():
    q = np.zeros((6, 1, 4))
    k = np.zeros((2, 1, 4))
    v = np.ones((2, 1, 4))
    o, lse = oracle.attn_fwd_varlen(q, k, v, [2, 4], [0, 2])
    assert np.isnan(o[:2]).all() and np.isnan(o[4:]).all()
    assert np.allclose(o[2:4], 1.0) and np.allclose(lse[0, 2:4], np.log(2.0))


def packed_bruteforce_bwd(q, k, v, dout, cu_q, cu_k, causal, scale):
    """The backward of packed_bruteforce through the same explicit mask, from
    the softmax's own derivative written over the packed rows (P from the
    forward's LSE; D = rowsum(dO o O); dS = P (dP - D); dQ = scale dS K,
    dK = scale dS^T Q, dV = P^T dO, with the K/V gradients of a GQA group
    summed over its query heads).  Plain float64 numpy."""
    total_q, Hq, _ = q.shape
    total_k, Hkv, _ = k.shape
    o, lse = packed_bruteforce(q, k, v, cu_q, cu_k, causal, scale)
    seq_q = np.full(total_q, -1)
    seq_k = np.full(total_k, -1)
    for b in range(len(cu_q) - 1):
        seq_q[cu_q[b]:cu_q[b + 1]] = b
        seq_k[cu_k[b]:cu_k[b + 1]] = b
    t = np.arange(total_q)[:, None]
    u = np.arange(total_k)[None, :]
    mask = (seq_q[:, None] == seq_k[None, :]) & (seq_q[:, None] >= 0)
    if causal:
        bq = np.maximum(seq_q, 0)
        q0 = np.asarray(cu_q)[bq][:, None]
        sq = (np.asarray(cu_q)[bq + 1] - np.asarray(cu_q)[bq])[:, None]
        k0 = np.asarray(cu_k)[bq][:, None]
        sk = (np.asarray(cu_k)[bq + 1] - np.asarray(cu_k)[bq])[:, None]
        mask &= (u - k0) <= (t - q0) + sk - sq
    ratio = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        kh = k[:, h // ratio, :]
        vh = v[:, h // ratio, :]
        s = scale * (q[:, h, :] @ kh.T)
        lrow = lse[h][:, None]
        p = np.where(mask & np.isfinite(lrow), np.exp(s - np.where(np.isfinite(lrow), lrow, 0.0)), 0.0)
        g = dout[:, h, :]
        dp = g @ vh.T
        dd = (g * o[:, h, :]).sum(axis=1, keepdims=True)
        ds = p * (dp - dd)
        dq[:, h, :] = scale * (ds @ kh)
        dk[:, h // ratio, :] += scale * (ds.T @ q[:, h, :])
        dv[:, h // ratio, :] += p.T @ g
    return dq, dk, dv


@pytest.mark.parametrize("case", CASES)
def test_oracle_varlen_backward_equals_packed_bruteforce(case):
    seq_q, seq_k, Hq, Hkv, causal = case
    cu_q = np.concatenate([[0], np.cumsum(seq_q)]).astype(int)
    cu_k = np.concatenate([[0], np.cumsum(seq_k)]).astype(int)
    rng = np.random.default_rng(sum(seq_q) * 31 + Hq)
    d, dvh = 8, 6
    q = rng.standard_normal((cu_q[-1], Hq, d))
    k = rng.standard_normal((cu_k[-1], Hkv, d))
    v = rng.standard_normal((cu_k[-1], Hkv, dvh))
    g = rng.standard_normal((cu_q[-1], Hq, dvh))
    scale = 0.4
    got = oracle.attn_bwd_varlen(q, k, v, g, cu_q, cu_k, causal=causal, scale=scale, threads=2)
    want = packed_bruteforce_bwd(q, k, v, g, cu_q, cu_k, causal, scale)
    for a, b in zip(got, want):
        assert np.allclose(a, b, rtol=1e-10, atol=1e-12)


def test_oracle_varlen_backward_equal_lengths_is_the_batched_problem():
    B, S, Hq, Hkv, d = 3, 11, 4, 2, 8
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, S, Hq, d))
    k = rng.standard_normal((B, S + 2, Hkv, d))
    v = rng.standard_normal((B, S + 2, Hkv, d))
    g = rng.standard_normal((B, S, Hq, d))
    for causal in (False, True):
        ref = oracle.attn_bwd(q, k, v, g, causal=causal, threads=2)
        cu_q = np.arange(B + 1) * S
        cu_k = np.arange(B + 1) * (S + 2)
        got = oracle.attn_bwd_varlen(q.reshape(B * S, Hq, d), k.reshape(-1, Hkv, d), v.reshape(-1, Hkv, d),
                                     g.reshape(B * S, Hq, d), cu_q, cu_k, causal=causal, threads=2)
        for a, b in zip(got, ref):
            assert np.array_equal(a.reshape(b.shape), b)


def test_varlen_workloads_recipe():
    for w in synthetic.varlen_workloads().values():
        assert w.total_q == 32768 and w.total_k == 32768
        assert all(128 <= n <= 8192 for n in w.seqlens_q[:-1]) and 1 <= w.seqlens_q[-1] <= 8192
        assert w.cu_seqlens_q[-1] == 32768 and w.cu_seqlens_q.dtype == np.int32
    a = synthetic.loguniform_lengths(5000, 100, 1000, seed=9)
    assert a == synthetic.loguniform_lengths(5000, 100, 1000, seed=9) and sum(a) == 5000


# ---------------------------------------------------------------------------
# host copy of the planning kernel
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_08_gb300 as m
    from exact_attention_forward_08_gb300 import _build
    _build.build()
    m.load_library()
    return m


def check_plan(fa, lq, lk, Hq, Hkv, dq, dv, causal, pack=0, l2=1 << 22):
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(int)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(int)
    recs = fa.fa_varlen_plan_host(cu_q, cu_k, Hq, Hkv, dq, dv, causal, l2_bytes=l2, pack=pack)
    assert len(recs) <= fa.fa_varlen_workspace_size(len(lq), Hq, int(cu_q[-1])) // 32
    base = fa.fa_make_plan(1, Hq, Hkv, 1, 1, dq, dv, causal, l2, pack)
    P, groups = base.pos_per_tile, base.groups
    # 1. records carry the sequence's offsets and lengths
    for r in recs:
        assert (r.q_row0, r.seqlen_q, r.k_row0, r.seqlen_k) == (cu_q[r.b], lq[r.b], cu_k[r.b], lk[r.b])
    # 2. every (sequence, head group, tile) with queries is covered exactly once
    seen = set()
    for r in recs:
        for s in range(2):
            pos0 = (2 * r.mblock + s) * P
            if pos0 < r.seqlen_q:
                key = (r.b, r.g, pos0)
                assert key not in seen
                seen.add(key)
    want = {(b, g, t * P) for b in range(len(lq)) for g in range(groups) for t in range(-(-lq[b] // P))}
    assert seen == want
    # 3. sequences appear in one block each, longest heaviest tile first, ties by index
    order = [r.b for r in recs]
    blocks = [b for b, _ in itertools.groupby(order)]
    assert len(blocks) == len(set(blocks))
    keys = [(-(-(lk[b]) // 128), -b) for b in blocks]
    assert keys == sorted(keys, reverse=True)
    # 4. inside a sequence: the fixed-length task order of a batch of one
    for b in blocks:
        mine = [(r.g, r.mblock) for r in recs if r.b == b]
        plan = fa.fa_make_plan(1, Hq, Hkv, lq[b], lk[b], dq, dv, causal, l2, pack)
        ref = [(t.g, t.mblock) for t in (fa.fa_plan_task(plan, i) for i in range(plan.num_tasks))]
        assert mine == ref
    return recs


@pytest.mark.parametrize("causal", [False, True])
def test_plan_small(fa, causal):
    check_plan(fa, [100, 300, 1, 0, 513, 128], [100, 400, 400, 7, 0, 129], 16, 4, 128, 128, causal)


def test_plan_pack_and_dims(fa):
    check_plan(fa, [77, 0, 300], [77, 5, 260], 6, 2, 192, 128, True)
    check_plan(fa, [257, 40], [513, 40], 4, 2, 64, 64, False, pack=1)
    check_plan(fa, [1000, 20, 3000], [1000, 20, 3000], 32, 1, 128, 128, True, l2=1 << 20)


def test_plan_random(fa):
    rng = np.random.default_rng(11)
    for _ in range(20):
        B = int(rng.integers(1, 12))
        lq = [int(x) for x in rng.integers(0, 700, B)]
        lk = [int(x) for x in rng.integers(0, 900, B)]
        check_plan(fa, lq, lk, 8, 2, 128, 64, bool(rng.integers(0, 2)))


def test_plan_empty_and_errors(fa):
    assert fa.fa_varlen_plan_host([0], [0], 4, 4, 128, 128, 0) == []
    assert fa.fa_varlen_plan_host([0, 0, 0], [0, 5, 9], 4, 4, 128, 128, 1) == []
    with pytest.raises(fa.FaError):
        fa.fa_varlen_plan_host([0, 5, 3], [0, 1, 2], 4, 4, 128, 128, 0)  # decreasing offsets


def test_workspace_bound(fa):
    rng = np.random.default_rng(5)
    for _ in range(50):
        B = int(rng.integers(1, 40))
        lq = [int(x) for x in rng.integers(0, 600, B)]
        Hq = int(rng.choice([1, 2, 8, 32]))
        recs = fa.fa_varlen_plan_host(np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lq)]),
                                      Hq, 1, 64, 64, int(rng.integers(0, 2)), pack=int(rng.choice([0, 1])))
        assert 256 + 32 * len(recs) <= fa.fa_varlen_workspace_size(B, Hq, sum(lq))


def test_first_masked_block_matches_block_rule(fa):
    for sq, sk, causal in [(300, 300, 1), (200, 456, 1), (456, 200, 1), (77, 77, 0), (130, 1, 1), (5, 130, 1),
                           (1000, 1000, 0), (128, 256, 0), (1, 1, 1)]:
        plan = fa.fa_make_plan(1, 2, 2, sq, sk, 128, 128, causal)
        for pos0 in range(0, sq, plan.pos_per_tile):
            jm = fa.fa_plan_first_masked_block(plan, pos0)
            for j in range(plan.kv_blocks + 1):
                assert fa.fa_plan_block_masked(plan, pos0, j) == (j >= jm), (sq, sk, causal, pos0, j)
