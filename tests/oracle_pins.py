"""Checks that tie the CPU oracle to facts that do not come from the oracle itself.

Each ``check_*`` takes an oracle-like module ``o`` (the real one, or a copy with a
planted mistake) and raises AssertionError when ``o`` disagrees with:
  * the worked examples printed on the pages (``tests/golden/``),
  * closed forms and invariants of the mathematics,
  * brute force on tiny inputs (O(n^2) ranking, exhaustive 4-bit pairs),
  * 40-digit ``decimal`` arithmetic, or
  * an independent library routine (torch's scaled_dot_product_attention and
    logsumexp in float64 on the CPU).
"""

from __future__ import annotations

import decimal
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = {}
    keys = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.setdefault(parts[0], []).append(parts[1:])
            keys.append(parts)
    return rows, keys


def _bits(s):
    return int(s, 2)


def _py_popcount(x):
    return bin(x & 0xFFFFFFFF).count("1")


# --------------------------------------------------------------------------- SCORE

def check_four_bit_example(o):
    """HashAttention, Eq. (2) worked example: 1011 vs 1011/1001/0110 -> 0/1/3."""
    rows, _ = _golden("hamming_4bit.txt")
    q = _bits(rows["query"][0][0])
    keys = np.array([_bits(k[0]) for k in rows["key"]], dtype=np.int64)
    want = np.array([int(k[1]) for k in rows["key"]])
    got = o.hamming_distances(q, keys)
    assert np.array_equal(got, want), (got, want)
    # the highest SCORE is the smallest distance: a budget of one keeps key 1011,
    # a budget of two keeps 1011 and 1001
    assert list(o.selected_set(q, keys, 3, 1, 0, 0)) == [0]
    assert list(o.selected_set(q, keys, 3, 2, 0, 0)) == [0, 1]


def check_popcount_invariants(o):
    """popcount(0)=0, popcount(~0)=32, one bit per power of two, x and ~x sum to 32."""
    assert int(o.popcount32(np.array([0]))[0]) == 0
    assert int(o.popcount32(np.array([0xFFFFFFFF]))[0]) == 32
    powers = np.array([1 << j for j in range(32)], dtype=np.int64)
    assert np.all(o.popcount32(powers) == 1)
    rng = np.random.default_rng(7)
    x = rng.integers(0, 2**32, size=4096, dtype=np.int64)
    pc = o.popcount32(x)
    assert np.all(pc + o.popcount32(x ^ 0xFFFFFFFF) == 32)
    assert np.array_equal(pc, [_py_popcount(int(v)) for v in x])
    # signed 32-bit storage of the same word gives the same count
    signed = x.astype(np.uint32).view(np.int32)
    assert np.array_equal(o.popcount32(signed), pc)
    # distances are symmetric and zero on the diagonal
    y = rng.integers(0, 2**32, size=64, dtype=np.int64)
    for a in y[:8]:
        assert np.array_equal(o.hamming_distances(int(a), y),
                              [_py_popcount(int(a) ^ int(b)) for b in y])
        assert int(o.hamming_distances(int(a), np.array([a]))[0]) == 0


def check_exhaustive_4bit(o):
    """All 16 x 16 four-bit pairs against bit counting of the XOR."""
    keys = np.arange(16, dtype=np.int64)
    for q in range(16):
        got = o.hamming_distances(q, keys)
        want = [bin(q ^ k).count("1") for k in range(16)]
        assert list(got) == want


def check_histogram(o):
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 2**32, size=3000, dtype=np.int64)
    dist = o.hamming_distances(12345, codes)
    h = o.distance_histogram(dist)
    assert h.shape == (33,) and int(h.sum()) == 3000
    want = [0] * 33
    for v in dist:
        want[int(v)] += 1
    assert list(h) == want


# --------------------------------------------------------------------------- TOPK

def _rank_bruteforce(dist):
    n = len(dist)
    return [sum(1 for j in range(n) if (dist[j], j) < (dist[i], i)) for i in range(n)]


def check_topm_bruteforce(o):
    """Tie rule (distance, then index) against an O(n^2) rank count, tiny n."""
    rng = np.random.default_rng(3)
    for trial in range(60):
        n = int(rng.integers(0, 48))
        # few distinct codes -> many ties
        pool = rng.integers(0, 2**32, size=int(rng.integers(1, 6)), dtype=np.int64)
        codes = pool[rng.integers(0, len(pool), size=n)] if n else np.zeros(0, np.int64)
        q = int(rng.integers(0, 2**32))
        m = int(rng.integers(0, n + 3))
        dist = o.hamming_distances(q, codes) if n else np.zeros(0, np.int64)
        rank = _rank_bruteforce(list(dist))
        want = [i for i in range(n) if rank[i] < m]
        got = list(o.top_m_by_score(dist, m))
        assert got == want, (trial, got, want)


def check_topm_ties(o):
    n, m = 50, 7
    codes = np.full(n, 0xDEADBEEF, dtype=np.int64)
    dist = o.hamming_distances(0x12345678, codes)
    assert list(o.top_m_by_score(dist, m)) == list(range(m))      # all tied -> first m
    dist = np.arange(n)[::-1].copy()                                 # all distinct
    assert list(o.top_m_by_score(dist, m)) == list(range(n - m, n))
    assert list(o.top_m_by_score(dist, 0)) == []
    assert list(o.top_m_by_score(dist, n + 5)) == list(range(n))


def check_windows(o):
    """First n_sink and most recent n_local positions, clamped to [0, n)."""
    assert list(o.window_positions(10, 3, 2)) == [0, 1, 2, 8, 9]
    assert list(o.window_positions(3, 4, 16)) == [0, 1, 2]
    assert list(o.window_positions(10, 0, 0)) == []
    assert list(o.window_positions(10, 0, 1)) == [9]
    assert list(o.window_positions(10, 1, 0)) == [0]
    assert list(o.window_positions(0, 4, 4)) == []
    assert list(o.window_positions(6, 4, 4)) == [0, 1, 2, 3, 4, 5]


def check_budget(o):
    """Sec. 4.4 budget accounting: 16,384 tokens, m=1,024, 128+128 -> <= 1,280 = 7.81 %."""
    rows, _ = _golden("budget_16384.txt")
    n, m = int(rows["n"][0][0]), int(rows["m"][0][0])
    S, L = int(rows["n_sink"][0][0]), int(rows["n_local"][0][0])
    cap = int(rows["max_reads"][0][0])
    pct = float(rows["percent_rounded"][0][0])
    assert o.max_reads(n, m, S, L) == cap
    assert round(100.0 * cap / n, 2) == pct
    rng = np.random.default_rng(5)
    q = 0
    # top-m tokens all in the middle (distance 0), others far (distance 32):
    codes = np.full(n, 0xFFFFFFFF, dtype=np.int64)
    mid = rng.choice(np.arange(S, n - L), size=m, replace=False)
    codes[mid] = q
    sel = o.selected_set(q, codes, n, m, S, L)
    assert len(sel) == cap                       # no overlap: the bound is reached
    assert set(mid) <= set(sel) and set(range(S)) <= set(sel)
    # force the top-m onto the sink window: the union shrinks by the overlap
    codes = np.full(n, 0xFFFFFFFF, dtype=np.int64)
    codes[:64] = q
    codes[mid[: m - 64]] = q
    sel = o.selected_set(q, codes, n, m, S, L)
    assert len(sel) == cap - 64


# --------------------------------------------------------------------------- GATHER-ATT

def _rand_qkv(rng, n, d):
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    return q, K, V


def check_dense_vs_sdpa(o):
    """m >= n: the estimator is full softmax attention (torch SDPA, float64 CPU)."""
    import torch
    rng = np.random.default_rng(13)
    for n, d in [(1, 64), (17, 64), (300, 128)]:
        q, K, V = _rand_qkv(rng, n, d)
        codes = rng.integers(0, 2**32, size=n, dtype=np.int64)
        idx, _, out, lse = o.decode_head(q, 77, codes, K, V, n, n + 4, 0, 0)
        assert list(idx) == list(range(n))
        tq = torch.tensor(q).view(1, 1, 1, d)
        tK = torch.tensor(K).view(1, 1, n, d)
        tV = torch.tensor(V).view(1, 1, n, d)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tK, tV).view(d).numpy()
        ref_lse = float(torch.logsumexp(torch.tensor(K @ q) / math.sqrt(d), 0))
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
        assert abs(lse - ref_lse) < 1e-12 * max(1.0, abs(ref_lse))


def check_decimal(o):
    """n <= 8 against 40-digit decimal arithmetic."""
    decimal.getcontext().prec = 40
    rng = np.random.default_rng(17)
    for n in range(1, 9):
        d = 4
        q, K, V = _rand_qkv(rng, n, d)
        q, K, V = q * 3, K * 2, V
        idx = np.arange(n)
        out, lse = o.attend(q, K, V, idx)
        D = decimal.Decimal
        z = [sum(D(float(K[i, t])) * D(float(q[t])) for t in range(d)) / D(d).sqrt()
             for i in range(n)]
        e = [zi.exp() for zi in z]
        s = sum(e)
        want_lse = s.ln()
        want = [sum(e[i] * D(float(V[i, t])) for i in range(n)) / s for t in range(d)]
        assert abs(D(lse) - want_lse) < D("1e-13")
        for t in range(d):
            assert abs(D(float(out[t])) - want[t]) < D("1e-13")


def check_weighted_sum(o):
    """Appendix B.1 numbers: a=(0.45,0.35,0.20), v=(1,-1,1) -> o=0.30, residuals 0.15/0.10."""
    rows, _ = _golden("weighted_sum.txt")
    a = np.array([float(x) for x in rows["a"][0]])
    v = np.array([float(x) for x in rows["v"][0]])
    o_want = float(rows["o"][0][0])
    e_first = float(rows["err_keep_first"][0][0])
    e_last = float(rows["err_keep_last"][0][0])
    # d = 1, q = 1, k_i = log a_i: z_i = log a_i, so the softmax weights are a
    q = np.array([1.0])
    K = np.log(a).reshape(3, 1)
    V = v.reshape(3, 1)
    out, lse = o.attend(q, K, V, np.arange(3))
    assert abs(out[0] - o_want) < 1e-12 and abs(lse) < 1e-12
    for keep, err in [(0, e_first), (2, e_last)]:
        part, lse_part = o.attend(q, K, V, np.array([keep]))
        contribution = math.exp(lse_part - lse) * part[0]   # a_keep * v_keep
        assert abs(abs(o_want - contribution) - err) < 1e-12


def check_lse_bounds(o):
    """max z <= lse <= max z + log |I|."""
    rng = np.random.default_rng(19)
    for n in [1, 2, 9, 400]:
        q, K, V = _rand_qkv(rng, n, 64)
        idx = np.sort(rng.choice(n, size=max(1, n // 2), replace=False))
        _, lse = o.attend(q, K, V, idx)
        z = K[idx] @ q / 8.0
        assert z.max() - 1e-12 <= lse <= z.max() + math.log(len(idx)) + 1e-12


def check_lse_gradient(o):
    """Nectar App. B, Eq. (B.1): grad_q lse = K^T softmax(K q / sqrt d) / sqrt d."""
    rng = np.random.default_rng(23)
    n, d = 40, 16
    q, K, V = _rand_qkv(rng, n, d)
    idx = np.arange(n)
    z = K @ q / math.sqrt(d)
    p = np.exp(z - z.max())
    p /= p.sum()
    want = K.T @ p / math.sqrt(d)
    eps = 1e-6
    for t in range(d):
        e = np.zeros(d)
        e[t] = eps
        _, lp = o.attend(q + e, K, V, idx)
        _, lm = o.attend(q - e, K, V, idx)
        assert abs((lp - lm) / (2 * eps) - want[t]) < 1e-7


def check_low_temperature(o):
    """Nectar App. B, Eq. (B.2): (1/beta) log sum exp(beta q.k) -> max q.k."""
    rng = np.random.default_rng(29)
    n, d = 30, 16
    q, K, V = _rand_qkv(rng, n, d)
    beta = 1e4
    _, lse = o.attend(beta * q, K, V, np.arange(n))
    assert abs(lse * math.sqrt(d) / beta - (K @ q).max()) < 1e-3


def check_empty(o):
    out, lse = o.attend(np.ones(8), np.ones((4, 8)), np.ones((4, 8)), np.array([], dtype=np.int64))
    assert lse == -math.inf and np.all(out == 0)
    idx, _, out, lse = o.decode_head(np.ones(8), 0, np.zeros(4, np.int64), np.ones((4, 8)),
                                     np.ones((4, 8)), 4, 0, 0, 0)
    assert len(idx) == 0 and lse == -math.inf and np.all(out == 0)


# --------------------------------------------------------------------------- merge

def check_merge_partition(o):
    """Nectar Eq. (3.4): merging the two halves of any partition gives the whole."""
    rng = np.random.default_rng(31)
    for trial in range(20):
        n, d = int(rng.integers(2, 200)), 32
        q, K, V = _rand_qkv(rng, n, d)
        q *= 2.0
        perm = rng.permutation(n)
        cut = int(rng.integers(1, n))
        p1, p2 = np.sort(perm[:cut]), np.sort(perm[cut:])
        o1, l1 = o.attend(q, K, V, p1)
        o2, l2 = o.attend(q, K, V, p2)
        o_all, l_all = o.attend(q, K, V, np.arange(n))
        om, lm = o.merge(o1, l1, o2, l2)
        assert np.allclose(om, o_all, rtol=1e-12, atol=1e-12)
        assert abs(lm - l_all) < 1e-12 * max(1.0, abs(l_all))
        assert abs(lm - np.logaddexp(l1, l2)) < 1e-12 * max(1.0, abs(lm))
        # Eq. (3.5) gate form with a = lse_1 and Z_loc = e^{lse_2}
        og = o.merge_gate(o1, l1, o2, l2)
        assert np.allclose(og, o_all, rtol=1e-12, atol=1e-12)
    # an empty part (lse = -inf) is neutral
    o1, l1 = o.attend(q, K, V, np.arange(n))
    om, lm = o.merge(o1, l1, np.zeros(d), -math.inf)
    assert np.allclose(om, o1) and lm == l1
    om, lm = o.merge(np.zeros(d), -math.inf, np.zeros(d), -math.inf)
    assert lm == -math.inf and np.all(om == 0)


def check_merge_segments(o):
    """Nectar Sec. 3 / Eq. (3.4) over k segments: merging the parts of any partition
    of I (some parts empty) gives attention over I; segment order does not matter."""
    rng = np.random.default_rng(41)
    for trial in range(25):
        n, d = int(rng.integers(1, 160)), 16
        q, K, V = _rand_qkv(rng, n, d)
        q *= 1.5
        k = int(rng.integers(1, 7))
        label = rng.integers(0, k, n)  # a part may get no token
        parts = [np.flatnonzero(label == s) for s in range(k)]
        res = [o.attend(q, K, V, p) for p in parts]
        outs = np.stack([r[0] for r in res])
        lses = np.array([r[1] for r in res])
        o_all, l_all = o.attend(q, K, V, np.arange(n))
        om, lm = o.merge_segments(outs, lses)
        assert np.allclose(om, o_all, rtol=1e-12, atol=1e-12)
        assert abs(lm - l_all) < 1e-12 * max(1.0, abs(l_all))
        perm = rng.permutation(k)
        om2, lm2 = o.merge_segments(outs[perm], lses[perm])
        assert np.allclose(om2, om, rtol=1e-12, atol=1e-12) and abs(lm2 - lm) < 1e-12 * max(1.0, abs(lm))
    # one segment is returned as it is; all-empty segments give (0, -inf)
    om, lm = o.merge_segments(outs[:1], lses[:1])
    assert np.allclose(om, outs[0]) and lm == lses[0]
    om, lm = o.merge_segments(np.ones((3, d)), np.full(3, -math.inf))
    assert lm == -math.inf and np.all(om == 0)


def check_encode(o):
    """Sign-projection codes: a worked 2-d example, identity projections (bit j is
    the sign of x_j), x = 0 gives 0 (sign(0) maps to bit 0), sign symmetry, positive
    scaling, and row permutations of W permuting the bits."""
    W2 = np.zeros((32, 2))
    W2[0] = (1.0, 1.0)
    W2[1] = (1.0, -1.0)
    assert o.encode(np.array([1.0, 0.5]), W2) == 0b11       # projections (1.5, 0.5)
    assert o.encode(np.array([0.5, 1.0]), W2) == 0b01       # projections (1.5, -0.5)
    rng = np.random.default_rng(43)
    d = 32
    x = rng.standard_normal(d)
    want = sum(1 << j for j in range(32) if x[j] > 0)
    assert o.encode(x, np.eye(32)) == want
    W = rng.standard_normal((32, 48))
    assert o.encode(np.zeros(48), W) == 0
    for _ in range(20):
        v = rng.standard_normal(48)
        c = o.encode(v, W)
        assert o.encode(-v, W) == (~c) & 0xFFFFFFFF          # no projection is exactly 0 here
        assert o.encode(3.7 * v, W) == c
        perm = rng.permutation(32)
        cp = o.encode(v, W[perm])
        assert all(((cp >> j) & 1) == ((c >> perm[j]) & 1) for j in range(32))
    # the ambiguity mask flags exactly the bits whose projection is (near) zero
    Wz = np.eye(32)
    xz = np.ones(32)
    xz[5] = 0.0
    assert o.encode_ambiguous(xz, Wz) == 1 << 5


def check_encode_mlp(o):
    """MLP map codes: a worked 2 -> 3 -> 3 -> 32 example in which both ReLUs clip
    a value and one output is exactly 0 (bit 0, the only ambiguous bit); identity
    hidden layers on non-negative inputs reduce to the sign projection; zero
    weights leave the bits of the last bias."""
    W1 = np.array([[1.0, -1.0], [2.0, 0.0], [-1.0, 0.0]])
    b1 = np.array([0.0, -1.0, 1.0])          # W1 x + b1 = (2, 5, -2) -> h1 = (2, 5, 0)
    W2 = np.array([[1.0, 0.0, 1.0], [-1.0, 1.0, 0.0], [0.0, 0.0, 1.0]])
    b2 = np.array([-3.0, 0.0, 1.0])          # W2 h1 + b2 = (-1, 3, 1) -> h2 = (0, 3, 1)
    W3 = np.array([[1.0, (-1.0) ** j, 1.0] for j in range(32)])
    b3 = np.array([j - 16.0 for j in range(32)])  # F_j = 3 (-1)^j + j - 15
    x = np.array([3.0, 1.0])
    # F_j > 0: even j >= 14 and odd j >= 19; F_12 = 0
    assert o.encode_mlp(x, W1, b1, W2, b2, W3, b3) == 0xFFFD4000
    assert o.encode_mlp_ambiguous(x, W1, b1, W2, b2, W3, b3) == 1 << 12
    rng = np.random.default_rng(53)
    d = 24
    I = np.eye(d)
    for _ in range(10):
        Wp = rng.standard_normal((32, d))
        v = np.abs(rng.standard_normal(d))
        z = np.zeros(d)
        assert o.encode_mlp(v, I, z, I, z, Wp, np.zeros(32)) == o.encode(v, Wp)
    bz = rng.standard_normal(32)
    H = 16
    assert o.encode_mlp(rng.standard_normal(d), np.zeros((H, d)), np.zeros(H), np.zeros((H, H)), np.zeros(H),
                        np.zeros((32, H)), bz) == sum(1 << j for j in range(32) if bz[j] > 0)


def check_exact_topm_and_recall(o):
    """Exact top-m by dot score against an O(n^2) rank, ties by index, m >= n; the
    rounding band brackets the boundary; recall on worked examples."""
    rng = np.random.default_rng(47)
    for trial in range(30):
        n, d = int(rng.integers(1, 70)), 8
        K = rng.standard_normal((n, d))
        if trial % 3 == 0:                    # repeated rows: exact ties
            K[rng.integers(0, n, n // 2)] = K[0]
        q = rng.standard_normal(d)
        m = int(rng.integers(0, n + 3))
        z = [float(np.dot(K[i], q)) for i in range(n)]
        rank = [sum(1 for j in range(n) if z[j] > z[i] or (z[j] == z[i] and j < i)) for i in range(n)]
        want = sorted(i for i in range(n) if rank[i] < m)
        got = o.top_m_by_dot(q, K, n, m)
        assert list(got) == want, (n, m)
        sure, band = o.top_m_band(q, K, n, m)
        assert set(sure) <= set(want) and set(want) <= set(sure) | set(band)
    K = np.tile(rng.standard_normal((1, 4)), (10, 1))  # all scores equal: the first m
    assert list(o.top_m_by_dot(rng.standard_normal(4), K, 10, 3)) == [0, 1, 2]
    assert o.recall([1, 2, 3], [2, 3, 4, 5]) == 0.5
    assert o.recall([7, 9], [7, 9]) == 1.0 and o.recall([1], [2]) == 0.0 and o.recall([], []) == 1.0
    assert abs(o.recall(np.arange(10), np.arange(5, 20)) - 5 / 15) < 1e-15


def check_exclusive_windows(o):
    """Exclusive reading: |I| = min(n, m + |W|), W inside I, and I minus W is the
    brute-force top-m of the tokens outside the windows; with no windows both
    readings agree. Per-head budgets reach every head."""
    rng = np.random.default_rng(53)
    for trial in range(40):
        n = int(rng.integers(1, 60))
        codes = rng.integers(0, 16, n) * 0x1111  # few distinct codes: many ties
        q = int(rng.integers(0, 2 ** 32))
        m, S, L = int(rng.integers(0, n + 4)), int(rng.integers(0, 6)), int(rng.integers(0, 6))
        I = o.selected_set(q, codes, n, m, S, L, exclusive=True)
        W = set(range(min(S, n))) | set(range(max(0, n - L), n))
        assert len(I) == min(n, m + len(W)) and W <= set(I)
        outside = [i for i in range(n) if i not in W]
        d = [_py_popcount(q ^ int(codes[i])) for i in outside]
        rank = _rank_bruteforce(d)
        assert set(I) - W == {outside[j] for j in range(len(outside)) if rank[j] < m}
        assert np.array_equal(o.selected_set(q, codes, n, m, 0, 0, exclusive=True),
                              o.selected_set(q, codes, n, m, 0, 0))
    B, Hq, Hkv, n_cap, dd = 2, 4, 2, 40, 4
    qv = rng.standard_normal((B, Hq, dd))
    Kv = rng.standard_normal((B, Hkv, n_cap, dd))
    q_sig = rng.integers(0, 2 ** 32, (B, Hq))
    k_sig = rng.integers(0, 2 ** 32, (B, Hkv, n_cap))
    mph = rng.integers(0, 20, (B, Hq))
    res = o.decode_batch(qv, q_sig, k_sig, Kv, Kv, np.array([40, 33]), 20, 2, 3, m_per_head=mph, exclusive=True)
    for (b, h), (idx, _, _, _) in res.items():
        want = o.selected_set(int(q_sig[b, h]), k_sig[b, h // 2], [40, 33][b], int(mph[b, h]), 2, 3, exclusive=True)
        assert np.array_equal(idx, want)


def check_wide_codes(o):
    """Codes of W 32-bit words: the distance is the bit count of the XOR of the
    concatenated integers (Python big ints), the histogram has 32 W + 1 bins, and
    the selection is the brute-force rank over those distances."""
    rng = np.random.default_rng(59)
    for W in (2, 4, 16):
        n = 60
        k = rng.integers(0, 2 ** 32, (n, W))
        if W == 2:
            k[rng.integers(0, n, 20)] = k[0]   # repeated codes: ties
        q = rng.integers(0, 2 ** 32, W)
        big = lambda words: sum(int(x) << (32 * j) for j, x in enumerate(words))
        want = [bin(big(k[i]) ^ big(q)).count("1") for i in range(n)]
        d = o.hamming_distances(q, k)
        assert list(d) == want
        h = o.distance_histogram(d, 32 * W + 1)
        assert len(h) == 32 * W + 1 and h.sum() == n and all(h[v] == want.count(v) for v in set(want))
        m, S, L = 17, 3, 5
        rank = _rank_bruteforce(want)
        top = {i for i in range(n) if rank[i] < m}
        win = set(range(S)) | set(range(n - L, n))
        assert set(o.selected_set(q, k, n, m, S, L)) == top | win
    # one word in the wide layout equals the 32-bit path
    k1 = rng.integers(0, 2 ** 32, (30, 1))
    q1 = rng.integers(0, 2 ** 32, 1)
    assert np.array_equal(o.hamming_distances(q1, k1), o.hamming_distances(int(q1[0]), k1[:, 0]))


def check_decode_composition(o):
    """decode_head = attend over selected_set, and decode_batch maps h to KV head h // G."""
    rng = np.random.default_rng(37)
    B, Hq, Hkv, n_cap, d = 2, 4, 2, 90, 8
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, n_cap, d))
    V = rng.standard_normal((B, Hkv, n_cap, d))
    k_sig = rng.integers(0, 2**32, size=(B, Hkv, n_cap), dtype=np.int64)
    q_sig = rng.integers(0, 2**32, size=(B, Hq), dtype=np.int64)
    lens = np.array([90, 37])
    res = o.decode_batch(q, q_sig, k_sig, K, V, lens, 11, 3, 5)
    for (b, h), (idx, dist, out, lse) in res.items():
        g = h // (Hq // Hkv)
        n = int(lens[b])
        want_idx = o.selected_set(int(q_sig[b, h]), k_sig[b, g], n, 11, 3, 5)
        assert list(idx) == list(want_idx)
        assert len(dist) == n
        # brute-force the selection independently from the distances
        rank = _rank_bruteforce([_py_popcount(int(q_sig[b, h]) ^ int(c)) for c in k_sig[b, g, :n]])
        top = {i for i in range(n) if rank[i] < 11}
        win = set(range(min(3, n))) | set(range(max(0, n - 5), n))
        assert set(idx) == top | win
        z = K[b, g, idx] @ q[b, h] / math.sqrt(d)
        w = np.exp(z - z.max())
        assert np.allclose(out, (w / w.sum()) @ V[b, g, idx], rtol=1e-12, atol=1e-12)


ALL_CHECKS = [
    check_four_bit_example, check_popcount_invariants, check_exhaustive_4bit, check_histogram,
    check_topm_bruteforce, check_topm_ties, check_windows, check_budget,
    check_dense_vs_sdpa, check_decimal, check_weighted_sum, check_lse_bounds,
    check_lse_gradient, check_low_temperature, check_empty,
    check_merge_partition, check_merge_segments, check_encode, check_encode_mlp, check_exact_topm_and_recall,
    check_exclusive_windows, check_wide_codes, check_decode_composition,
]


def failing_checks(o):
    """Names of the checks that ``o`` fails (exceptions of any kind count as failures)."""
    bad = []
    for chk in ALL_CHECKS:
        try:
            chk(o)
        except Exception:  # noqa: BLE001 - a crash in a mutated oracle is a detection too
            bad.append(chk.__name__)
    return bad

