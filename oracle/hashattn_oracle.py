"""Plain, slow CPU oracle of the HashAttention sparse-decode path.

TEST INFRASTRUCTURE ONLY. This module is imported by the tests, by
``__graft_entry__.smoke()`` and by ``bench.py``'s CPU-baseline / reference arm,
and by nothing else. The product path (the CUDA library and its Python binding)
never imports, links or calls it, and it shares no code, table or helper with
that path.

Everything is NumPy in float64 (signature work in Python/NumPy integers), one
(batch, query head) at a time, written straight from the definitions:

* HashAttention: Semantic Sparsity for Faster Inference (Desai et al., ICML 2025,
  arXiv:2412.14468v2)
    - "Only selection is approximate; selected KV stay in full form" (Sec. 4):
      z_i = <q, k_i>/sqrt(d); o_hat = sum_{i in I} e^{z_i} v_i / sum_{j in I} e^{z_j};
      three stages SCORE / TOPK / GATHER-ATT.
    - "A 32-bit signature makes scoring cheap" (Eqs. (1)-(2), Sec. 4.1):
      SCORE(k_i, q) = -popcount(h_i XOR h_q).
    - Sec. 5: the selection is compared with the exact top-k by attention score
      (``top_m_by_dot``) through its recall (``recall``).
    - Sec. 4.1: the signature is ReLU(sign(.)) of a projection of q or k
      (``encode``; bit j set iff projection j is positive).
    - Sec. 5 (latency setup): the map as an MLP d -> 128 -> 128 -> 32
      (``encode_mlp``: ReLU hidden layers with biases, a reading).
    - "Token-level sparsity still needs a careful kernel" (Sec. 4.4, budget
      accounting): the retrieval budget m is joined by the first and the most
      recent tokens of the context.
* Nectar: Neural Estimation of Cached-Token Attention via Regression
  (arXiv:2605.09778v2)
    - Sec. 3, Eq. (3.1): alpha(q) = log sum_j e^{s_j} (log attention mass),
      A(q) = sum_j e^{s_j} v_j / sum_j e^{s_j}.
    - Eqs. (3.4)-(3.5): ATT_full = (e^alpha A + N_loc) / (e^alpha + Z_loc); the
      split of the softmax sum is exact; gate form g = sigmoid(a - log Z_loc).
    - Sec. 3 (virtual logit/value pair): any number of segments merge the same
      way (``merge_segments``).

Readings where the pages are silent (each is listed in the design notes):
  * keep the m SMALLEST Hamming distances (SCORE is the negated distance);
  * ties are broken by token index ascending, so the selected set is unique;
  * T (top-min(m, n) over all n tokens) is UNIONED with the windows
    [0, min(S, n)) and [max(0, n - Lw), n); duplicates are counted once (the
    other reading, T over the tokens outside the windows with |I| fixed at
    min(n, m + |W|), is available as ``exclusive``);
  * a budget may be given per sequence or per query head (each <= m);
  * the softmax scale is 1/sqrt(d); lse is the natural log of the sum over I;
  * an empty selected set gives out = 0 and lse = -inf;
  * the query head h reads KV head h // G (contiguous GQA groups).

Pins: ``tests/test_oracle_pins.py`` ties every function here to something
other than itself (the worked examples printed on the pages, closed forms,
brute force on tiny inputs, extended-precision arithmetic, and an independent
library routine); ``tests/test_oracle_mutations.py`` plants plausible mistakes
in copies of these functions and shows that a pin fails for each.
"""

from __future__ import annotations

import math

import numpy as np

N_BINS = 33  # a 32-bit Hamming distance takes the values 0..32


# ---------------------------------------------------------------------------
# SCORE -- HashAttention, Eq. (2): SCORE(k_i, q) = -popcount(h_i XOR h_q)
# ---------------------------------------------------------------------------

def popcount32(x) -> np.ndarray:
    """Number of set bits of each 32-bit word, as the plain sum of its 32 bits."""
    w = np.asarray(x).astype(np.int64) & 0xFFFFFFFF
    total = np.zeros(w.shape, dtype=np.int64)
    for j in range(32):
        total += (w >> j) & 1
    return total


def hamming_distances(q_code, k_codes) -> np.ndarray:
    """popcount(h_q XOR h_i) for every key code h_i (the negated SCORE).

    32-bit codes: ``q_code`` an integer, ``k_codes`` [n]. Wider codes (HashAttention
    Sec. 5 varies the signature length): ``q_code`` [W] and ``k_codes`` [n, W]
    32-bit words; the distance sums over the words.
    """
    k = np.asarray(k_codes).astype(np.int64) & 0xFFFFFFFF
    if k.ndim == 1:
        q = np.int64(int(q_code) & 0xFFFFFFFF)
        return popcount32(k ^ q)
    q = (np.asarray(q_code).astype(np.int64) & 0xFFFFFFFF).reshape(1, -1)
    return popcount32(k ^ q).sum(axis=1)


def encode(x, W) -> int:
    """32-bit code of vector x under the projection W [32, d].

    HashAttention, Sec. 4.1: the signature is ReLU(sign(F(x))), so bit j is 1 iff
    the j-th projection is positive (0 maps to bit 0). F is the learned map on the
    pages; a given linear W (sign random projection) stands in for it here.
    Decided in float64.
    """
    proj = np.asarray(W, dtype=np.float64) @ np.asarray(x, dtype=np.float64)
    code = 0
    for j in range(32):
        if proj[j] > 0.0:
            code |= 1 << j
    return code


def encode_ambiguous(x, W, eps: float = 2.0 ** -22) -> int:
    """Bits of ``encode`` that float32 arithmetic may decide either way: those whose
    projection lies within d * eps * sum_k |W_jk x_k| of zero (a bound on the
    rounding error of any float32 summation order)."""
    W = np.asarray(W, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    proj = W @ x
    bound = W.shape[1] * eps * (np.abs(W) @ np.abs(x))
    mask = 0
    for j in range(32):
        if abs(proj[j]) <= bound[j]:
            mask |= 1 << j
    return mask


def mlp_forward(x, W1, b1, W2, b2, W3, b3):
    """F(x) = W3 relu(W2 relu(W1 x + b1) + b2) + b3 in float64, with the hidden
    values (h1, h2) it passes through.

    HashAttention, Sec. 5 (latency setup) runs the signature map F as an MLP
    d -> 128 -> 128 -> 32. The pages give the widths only; the plainest reading
    is two hidden layers with biases and a ReLU after each (the signature itself
    is ReLU(sign(.)) of the last layer, Sec. 4.1).
    """
    x = np.asarray(x, dtype=np.float64)
    h1 = np.maximum(np.asarray(W1, np.float64) @ x + np.asarray(b1, np.float64), 0.0)
    h2 = np.maximum(np.asarray(W2, np.float64) @ h1 + np.asarray(b2, np.float64), 0.0)
    f = np.asarray(W3, np.float64) @ h2 + np.asarray(b3, np.float64)
    return f, h1, h2


def encode_mlp(x, W1, b1, W2, b2, W3, b3) -> int:
    """32-bit code of x under the MLP map: bit j is 1 iff F_j(x) > 0 (0 maps to
    bit 0), decided in float64."""
    f, _, _ = mlp_forward(x, W1, b1, W2, b2, W3, b3)
    code = 0
    for j in range(32):
        if f[j] > 0.0:
            code |= 1 << j
    return code


def encode_mlp_ambiguous(x, W1, b1, W2, b2, W3, b3, eps: float = 2.0 ** -23) -> int:
    """Bits of ``encode_mlp`` that float32 evaluation may decide either way.

    One float32 layer y = W h + b over K inputs, in any summation order, is off
    by at most (K + 1) eps (|W| |h| + |b|), with eps twice the unit roundoff; an
    error e in its input adds |W| e, and ReLU does not enlarge an error. The
    bound is carried through the three layers (using |h| + e for the float32
    hidden values); bit j is ambiguous when |F_j| is within it."""
    W1, W2, W3 = (np.asarray(w, np.float64) for w in (W1, W2, W3))
    b1, b2, b3 = (np.asarray(b, np.float64) for b in (b1, b2, b3))
    x = np.asarray(x, dtype=np.float64)
    f, h1, h2 = mlp_forward(x, W1, b1, W2, b2, W3, b3)
    e1 = (W1.shape[1] + 1) * eps * (np.abs(W1) @ np.abs(x) + np.abs(b1))
    e2 = (W2.shape[1] + 1) * eps * (np.abs(W2) @ (h1 + e1) + np.abs(b2)) + np.abs(W2) @ e1
    e3 = (W3.shape[1] + 1) * eps * (np.abs(W3) @ (h2 + e2) + np.abs(b3)) + np.abs(W3) @ e2
    mask = 0
    for j in range(32):
        if abs(f[j]) <= e3[j]:
            mask |= 1 << j
    return mask


def distance_histogram(dist, nbins: int = N_BINS) -> np.ndarray:
    """Count of tokens at each distance 0..nbins-1 (33 bins for 32-bit codes, b + 1 for b bits)."""
    return np.bincount(np.asarray(dist, dtype=np.int64), minlength=nbins)[:nbins]


# ---------------------------------------------------------------------------
# TOPK -- HashAttention, Sec. 4 (three stages) and Sec. 4.4 (fixed windows)
# ---------------------------------------------------------------------------

def top_m_by_score(dist, m: int) -> np.ndarray:
    """Indices of the min(m, n) tokens with the highest SCORE, ascending.

    Highest SCORE = smallest distance; ties go to the smaller token index.
    """
    dist = np.asarray(dist, dtype=np.int64)
    n = dist.shape[0]
    k = max(0, min(int(m), n))
    order = np.lexsort((np.arange(n), dist))  # last key is primary: distance, then index
    return np.sort(order[:k]).astype(np.int64)


def window_positions(n: int, n_sink: int, n_local: int) -> np.ndarray:
    """The first n_sink and the most recent n_local positions of an n-token context."""
    sink = np.arange(0, max(0, min(int(n_sink), n)), dtype=np.int64)
    local = np.arange(max(0, n - int(n_local)), n, dtype=np.int64)
    return np.union1d(sink, local).astype(np.int64)


def selected_set(q_code, k_codes, n: int, m: int, n_sink: int, n_local: int,
                 exclusive: bool = False) -> np.ndarray:
    """I = top-m by SCORE joined with the sink/local windows.

    Default reading: the top-m is taken over all n tokens (windows may repeat some
    of them, so |I| <= m + |windows|). ``exclusive``: the other reading of the
    budget arithmetic (HashAttention Sec. 4.4, m plus the fixed positions): the
    top-m is taken over the tokens outside the windows, so |I| = min(n, m + |W|).
    """
    dist = hamming_distances(q_code, np.asarray(k_codes)[:n])
    win = window_positions(n, n_sink, n_local)
    if exclusive:
        outside = np.setdiff1d(np.arange(n, dtype=np.int64), win)
        top = outside[top_m_by_score(dist[outside], m)]
    else:
        top = top_m_by_score(dist, m)
    return np.union1d(top, win).astype(np.int64)


def max_reads(n: int, m: int, n_sink: int, n_local: int) -> int:
    """Upper bound on |I|: the budget plus every fixed window position, capped at n."""
    return min(n, m + n_sink + n_local)


# ---------------------------------------------------------------------------
# The exact comparator of the selection -- HashAttention, Sec. 5 (oracle top-k
# by attention score) and the recall of the hashed selection against it
# ---------------------------------------------------------------------------

def dot_scores(q, K, n: int) -> np.ndarray:
    """<q, k_i> for the first n rows of K, in float64 (the ranking is that of z_i)."""
    return np.asarray(K, dtype=np.float64)[:n] @ np.asarray(q, dtype=np.float64)


def top_m_by_dot(q, K, n: int, m: int) -> np.ndarray:
    """Indices of the min(m, n) largest <q, k_i>, ascending; ties go to the smaller index."""
    z = dot_scores(q, K, n)
    k = max(0, min(int(m), n))
    order = np.lexsort((np.arange(n), -z))  # score descending, then index ascending
    return np.sort(order[:k]).astype(np.int64)


def top_m_band(q, K, n: int, m: int, eps: float = 2.0 ** -22):
    """(sure, band): the tokens certainly in the top min(m, n) and those whose score
    lies within the float32 rounding bound d * eps * sum_k |q_k k_ik| of the
    min(m, n)-th largest score (either decision is valid for them)."""
    q = np.asarray(q, dtype=np.float64)
    Kf = np.asarray(K, dtype=np.float64)[:n]
    z = Kf @ q
    k = max(0, min(int(m), n))
    if k == 0 or k == n:
        return np.arange(k, dtype=np.int64), np.zeros(0, dtype=np.int64)
    bound = Kf.shape[1] * eps * (np.abs(Kf) @ np.abs(q))
    zk = np.sort(z)[::-1][k - 1]
    band = np.flatnonzero(np.abs(z - zk) <= bound + bound.max())
    sure = np.flatnonzero(z - bound - bound.max() > zk)
    return sure.astype(np.int64), band.astype(np.int64)


def recall(selected, reference) -> float:
    """|selected & reference| / |reference| (1.0 when the reference is empty)."""
    ref = np.unique(np.asarray(reference, dtype=np.int64))
    if ref.size == 0:
        return 1.0
    hit = np.intersect1d(np.unique(np.asarray(selected, dtype=np.int64)), ref).size
    return hit / ref.size


# ---------------------------------------------------------------------------
# GATHER-ATT -- HashAttention, Sec. 4; log-normaliser from Nectar, Eq. (3.1)
# ---------------------------------------------------------------------------

def attend(q, K, V, idx):
    """Softmax attention of one query over the rows ``idx`` of K/V, in float64.

    Returns (out, lse): out = sum_i e^{z_i} v_i / sum_j e^{z_j} and
    lse = log sum_j e^{z_j}, z_i = <q, k_i>/sqrt(d), i, j over idx.
    Empty idx gives (zeros, -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size == 0:
        return np.zeros(np.asarray(V).shape[-1], dtype=np.float64), -math.inf
    k_rows = np.asarray(K)[idx].astype(np.float64)
    v_rows = np.asarray(V)[idx].astype(np.float64)
    z = k_rows @ q / math.sqrt(d)
    z_max = z.max()
    w = np.exp(z - z_max)
    total = w.sum()
    lse = z_max + math.log(total)
    out = (w / total) @ v_rows
    return out, lse


def merge(out_a, lse_a, out_b, lse_b):
    """Exact merge of two partial attentions over disjoint token sets.

    Nectar, Eq. (3.4): with e^{lse_a} the mass of part a and N_b = e^{lse_b} out_b,
    ATT = (e^{lse_a} out_a + e^{lse_b} out_b) / (e^{lse_a} + e^{lse_b});
    the merged log-normaliser is log(e^{lse_a} + e^{lse_b}).
    """
    out_a = np.asarray(out_a, dtype=np.float64)
    out_b = np.asarray(out_b, dtype=np.float64)
    if lse_a == -math.inf and lse_b == -math.inf:
        return np.zeros_like(out_a), -math.inf
    top = max(lse_a, lse_b)
    wa = math.exp(lse_a - top)
    wb = math.exp(lse_b - top)
    out = (wa * out_a + wb * out_b) / (wa + wb)
    return out, top + math.log(wa + wb)


def merge_gate(out_a, lse_a, out_loc, lse_loc):
    """Nectar, Eq. (3.5) gate form: g = sigmoid(lse_a - lse_loc); g*A + (1-g)*A_loc."""
    g = 1.0 / (1.0 + math.exp(-(lse_a - lse_loc)))
    return g * np.asarray(out_a, dtype=np.float64) + (1.0 - g) * np.asarray(out_loc, dtype=np.float64)


def merge_segments(outs, lses):
    """Exact merge of any number of partial attentions over disjoint token sets.

    Nectar, Sec. 3: a segment whose scores are not materialised enters the
    softmax as one virtual logit lse_s with value out_s; with Eq. (3.4) applied to
    every segment, L = log sum_s e^{lse_s} and out = sum_s e^{lse_s - L} out_s.
    ``outs`` [k, d] (k >= 1), ``lses`` [k]; segments with lse = -inf contribute
    nothing, and if all are empty the result is (zeros, -inf).
    """
    outs = np.asarray(outs, dtype=np.float64)
    lse_list = [float(x) for x in np.asarray(lses, dtype=np.float64).reshape(-1)]
    live = [s for s, l in enumerate(lse_list) if l != -math.inf]
    if not live:
        return np.zeros(outs.shape[-1], dtype=np.float64), -math.inf
    peak = max(lse_list[s] for s in live)
    mass = [math.exp(lse_list[s] - peak) for s in live]
    norm = sum(mass)
    merged = sum(m_s * outs[s] for m_s, s in zip(mass, live)) / norm
    return merged, peak + math.log(norm)


# ---------------------------------------------------------------------------
# The whole path, one (batch, query head) at a time
# ---------------------------------------------------------------------------

def decode_head(q, q_code, k_codes, K, V, n: int, m: int, n_sink: int, n_local: int,
                dense: bool = False, exclusive: bool = False):
    """One query head's sparse decode: SCORE -> TOPK -> GATHER-ATT.

    K, V: [n_cap, d] rows of the query's KV head (any float dtype; widened to
    float64 on the selected rows). ``dense`` attends over every token (the
    m >= n reading of Sec. 4: the estimator equals full attention when I is all
    tokens). Returns (idx, dist, out, lse).
    """
    if dense:
        idx = np.arange(n, dtype=np.int64)
        dist = None
    else:
        dist = hamming_distances(q_code, np.asarray(k_codes)[:n])
        idx = selected_set(q_code, k_codes, n, m, n_sink, n_local, exclusive=exclusive)
    out, lse = attend(q, K, V, idx)
    return idx, dist, out, lse


def decode_batch(q, q_sig, k_sig, K, V, seq_lens, m, n_sink, n_local,
                 m_per_seq=None, dense=False, heads=None, m_per_head=None, exclusive=False):
    """Run ``decode_head`` over (b, h) pairs.

    Layouts (NumPy arrays): q [B, Hq, d]; q_sig [B, Hq] (32-bit words);
    k_sig [B, Hkv, n_cap]; K, V [B, Hkv, n_cap, d] (a batch extent of 1 is shared
    by every batch entry); seq_lens [B]; m_per_head [B, Hq] overrides the
    budgets. ``heads`` restricts the work to a list of (b, h) pairs. Returns
    {(b, h): (idx, dist, out, lse)}.
    """
    B, Hq = q.shape[0], q.shape[1]
    Hkv = K.shape[1]
    G = Hq // Hkv
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    res = {}
    for b, h in pairs:
        g = h // G
        kb = 0 if K.shape[0] == 1 else b
        sb = 0 if (k_sig is None or k_sig.shape[0] == 1) else b
        n = int(seq_lens[b])
        mb = int(m_per_seq[b]) if m_per_seq is not None else int(m)
        if m_per_head is not None:
            mb = int(m_per_head[b, h])
        codes = None if dense else k_sig[sb, g]
        qc = None if dense else int(q_sig[b, h])
        res[(b, h)] = decode_head(q[b, h], qc, codes, K[kb, g], V[kb, g], n, mb,
                                  n_sink, n_local, dense=dense, exclusive=exclusive)
    return res
