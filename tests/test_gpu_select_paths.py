"""Every selection kernel instantiation the library launches, against the oracle.

The fused selection (32-bit codes; more than four query heads per KV head run as
virtual groups of at most four) runs a scan kernel and an emit kernel over
ranges of 8,192 tokens, with the ranges of a sequence combined by the scan's
last CTA; the cases vary the number of ranges, where the windows and the tie
boundary fall among them, and the budget rules. The two-kernel path (codes
wider than 32 bits in the decode; the selection entry point with more than four
query heads per KV head) has SCORE/TOPK instantiations for 4, 8, 16 and 32
tokens per thread. Each case asserts which plan the shape takes
(hash_attn_selection_plan) and then compares the selected sets bit for bit and
the attention within tolerance on the selected heads.
"""
import numpy as np
import pytest
import torch

import gpu_helpers as GH
from oracle import hashattn_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from long_context_sparse_score_gb300 import _build
    _build.build()
    from long_context_sparse_score_gb300 import hashattn
    hashattn.lib()


def W():
    from long_context_sparse_score_gb300 import workloads
    return workloads


def _codes(w, kind, seed):
    """Replace the workload's codes: 'random' keeps the projection codes, 'pool'
    draws from a few codes near the query (the threshold bin holds thousands of
    ties), 'far' makes every key the complement of every query (all distances 32)."""
    if kind == "random":
        return
    q0 = 0x0F0F0F0F
    if kind == "pool":
        gen = torch.Generator(device="cuda").manual_seed(seed)
        pool = torch.tensor([q0, q0 ^ 1, q0 ^ 3, q0 ^ 0x70000000, q0 ^ 0x0000FFFF], dtype=torch.int32,
                            device="cuda")
        w.k_sig = pool[torch.randint(0, 5, w.k_sig.shape, generator=gen, device="cuda")].contiguous()
    elif kind == "far":
        w.k_sig = torch.full_like(w.k_sig, ~q0)
    w.q_sig = torch.full_like(w.q_sig, q0)


def _check(w, heads, *, exclusive=False, m_per_head=None, code_words=1, att_heads=4):
    res = GH.run_decode(w, exclusive=exclusive, m_per_head=m_per_head, code_words=code_words)
    assert res["status"] == 0, hex(res["flags"])
    hc = GH.HostCopy(w, exclusive=exclusive, m_per_head=m_per_head)
    GH.check_selection(res, hc, heads, w.m)
    GH.check_attention(res, hc, heads[:att_heads], w.m)
    return res


def _check_two_kernel(w, heads, *, exclusive=False, m_per_head=None, att_heads=4):
    """The selection entry point (the two-kernel SCORE/TOPK on the caller's shape,
    which takes any number of query heads per KV head) and GATHER-ATT on its lists,
    against the oracle."""
    H = GH.ha()
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig, batch=w.B)
    opts = H.select_opts(m_per_head, exclusive, 1) if (exclusive or m_per_head is not None) else None
    ws = torch.empty(H.hash_attn_workspace_size_ex(shape, w.m, w.n_sink, w.n_local, opts), dtype=torch.uint8,
                     device="cuda")
    H.hash_attn_workspace_init(ws)
    B, Hq, d = w.q.shape
    cap = H.hash_attn_select_capacity(w.n_cap, w.m, w.n_sink, w.n_local)
    idx = torch.full((B, Hq, cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, Hq), -7, dtype=torch.int32, device="cuda")
    H.hash_attn_select_ex(shape, w.q_sig, w.k_sig, w.seq_lens, w.m_per_seq, w.m, w.n_sink, w.n_local, opts, idx,
                          cnt, workspace=ws)
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    H.hash_attn_gather_att(shape, w.q, w.K, w.V, w.seq_lens, idx, cap, cnt, out, lse, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, hex(flags)
    res = dict(out=out, lse=lse, sel_idx=idx, sel_cnt=cnt, cap=cap)
    hc = GH.HostCopy(w, exclusive=exclusive, m_per_head=m_per_head)
    GH.check_selection(res, hc, heads, w.m)
    GH.check_attention(res, hc, heads[:att_heads], w.m)


def _plan(w, code_words=1):
    H = GH.ha()
    return H.hash_attn_selection_plan(H.make_shape(w.q, w.K, w.V, w.k_sig), code_words)


# ---------------------------------------------------------------- fused selection: ranges, windows, ties

FUSED = [
    # name, B, Hq, Hkv, n_cap, lens, m, S, Lw, codes
    ("one_range", 2, 8, 2, 8192, [8192, 5000], 300, 16, 64, "pool"),
    ("two_ranges_ragged", 2, 4, 1, 12000, [12000, 7000], 700, 40, 500, "random"),
    ("four_ranges_g3", 1, 3, 1, 30000, [30000], 2000, 128, 128, "pool"),
    ("windows_span_ranges_g2", 2, 4, 2, 60000, [60000, 33333], 1500, 9000, 9000, "pool"),
    ("g1_long_local_window", 1, 1, 1, 65536, [65535], 4000, 7, 20000, "random"),
    ("many_pairs_ragged", 40, 8, 8, 16000, [16000 - 7 * i for i in range(40)], 1000, 16, 32, "random"),
    ("empty_and_one_token", 20, 8, 8, 30000, [30000] * 10 + [1, 0] + [29000] * 8, 1000, 16, 32, "pool"),
    ("sixteen_ranges", 5, 32, 8, 131072, [131072, 5, 131071, 0, 70000], 4096, 128, 256, "pool"),
    ("windows_span_ranges_long", 1, 4, 1, 262144, [250000], 5000, 70000, 40000, "pool"),
    ("sixty_four_ranges", 1, 2, 1, 524288, [524288], 16000, 128, 256, "pool"),
    ("all_distances_32", 1, 4, 1, 20000, [20000], 900, 16, 16, "far"),
    ("budget_zero_windows_only", 1, 4, 1, 20000, [20000], 0, 9000, 100, "pool"),
]


@pytest.mark.parametrize("case", FUSED, ids=[c[0] for c in FUSED])
def test_fused_selection(case):
    name, B, Hq, Hkv, n_cap, lens, m, S, Lw, codes = case
    w = W().make_gqa(31, B=B, Hq=Hq, Hkv=Hkv, d=128, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S, n_local=Lw,
                     device="cuda", name=name)
    _codes(w, codes, 41)
    plan = _plan(w)
    assert plan["fused"] == 1 and plan["ranges"] == -(-n_cap // 8192), plan
    heads = [(b, h) for b in range(B) for h in range(Hq)]
    if len(heads) > 16:
        heads = _sample(B, Hq, 16, 5)
    _check(w, heads)


FUSED_VARIANTS = [
    # name, n_cap, lens, m, S, Lw, codes, exclusive, per-head budgets
    ("exclusive_quota_across_ranks", 60000, [60000, 41000], 3000, 9000, 12000, "pool", True, False),
    ("per_head_budgets_cl8", 60000, [60000, 20000], 2500, 64, 128, "random", False, True),
    ("exclusive_per_head_cl16", 100000, [100000, 77777], 3000, 128, 20000, "pool", True, True),
]


@pytest.mark.parametrize("case", FUSED_VARIANTS, ids=[c[0] for c in FUSED_VARIANTS])
def test_fused_selection_variants(case):
    """Exclusive windows and per-head budgets where the windows and the tie
    boundary fall in different ranges."""
    name, n_cap, lens, m, S, Lw, codes, exclusive, per_head = case
    w = W().make_gqa(32, B=2, Hq=4, Hkv=1, d=128, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S, n_local=Lw,
                     device="cuda", name=name)
    _codes(w, codes, 42)
    assert _plan(w)["ranges"] >= 8
    mph = None
    if per_head:
        gen = torch.Generator(device="cuda").manual_seed(9)
        mph = torch.randint(0, m + 1, (2, 4), generator=gen, device="cuda", dtype=torch.int32)
        mph[0, 0], mph[1, 3] = 0, m
    res = _check(w, [(b, h) for b in range(2) for h in range(4)], exclusive=exclusive, m_per_head=mph)
    if exclusive:
        cnt = res["sel_cnt"].cpu().numpy()
        for b, n in enumerate(lens):
            nw = len(O.window_positions(n, S, Lw))
            for h in range(4):
                mb = int(mph[b, h]) if per_head else m
                assert int(cnt[b, h]) == min(n, mb + nw)


def test_fused_select_entry_point_pads_and_matches_decode():
    H = GH.ha()
    w = W().make_gqa(33, B=2, Hq=4, Hkv=1, d=128, n_cap=60000, seq_lens=[60000, 100], m=2000, n_sink=64,
                     n_local=64, device="cuda")
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig)
    ws = GH.workspace(shape, w.m, w.n_sink, w.n_local)
    cap = H.hash_attn_select_capacity(60000, 2000, 64, 64)
    sel = torch.full((2, 4, cap), 77, dtype=torch.int32, device="cuda")
    cnt = torch.full((2, 4), 77, dtype=torch.int32, device="cuda")
    H.hash_attn_select(shape, w.q_sig, w.k_sig, w.seq_lens, None, 2000, 64, 64, sel, cnt, workspace=ws)
    res = {"sel_idx": sel, "sel_cnt": cnt, "cap": cap}
    GH.check_selection(res, GH.HostCopy(w), [(b, h) for b in range(2) for h in range(4)], 2000)
    dec = GH.run_decode(w)
    assert torch.equal(dec["sel_idx"], sel) and torch.equal(dec["sel_cnt"], cnt)


# ---------------------------------------------------------------- two-kernel path: every TPT
# Eight query heads per KV head: the selection entry point takes the two-kernel
# path (its chunk, hence its tokens per thread, set by the shape); the decode runs
# two virtual groups of four per KV head on the fused selection and the group
# kernel. Both against the oracle.

TWO_KERNEL = [
    # name, B, Hq, Hkv, n_cap, lens, m, S, Lw, codes, expected chunk
    ("g8_tpt4", 2, 64, 8, 10000, [10000, 6000], 500, 32, 64, "pool", 1024),
    ("g8_tpt8", 2, 64, 8, 40000, [40000, 25000], 1200, 128, 128, "random", 2048),
    ("g8_tpt16", 2, 64, 8, 80000, [80000, 79999], 2500, 128, 256, "pool", 4096),
    ("g8_tpt32", 2, 64, 8, 150000, [150000, 99999], 4096, 128, 256, "random", 8192),
]


def _sample(B, Hq, k, seed):
    rng = np.random.default_rng(seed)
    heads = [(b, h) for b in range(B) for h in range(Hq)]
    pick = rng.choice(len(heads), size=min(k, len(heads)), replace=False)
    return sorted(heads[i] for i in pick)


@pytest.mark.parametrize("case", TWO_KERNEL, ids=[c[0] for c in TWO_KERNEL])
def test_two_kernel_selection(case):
    name, B, Hq, Hkv, n_cap, lens, m, S, Lw, codes, chunk = case
    w = W().make_gqa(34, B=B, Hq=Hq, Hkv=Hkv, d=128, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S, n_local=Lw,
                     device="cuda", name=name)
    _codes(w, codes, 43)
    plan = _plan(w)
    assert plan["fused"] == 1 and plan["chunk"] == chunk, plan
    heads = _sample(B, Hq, 12, 1)
    _check_two_kernel(w, heads)
    res = _check(w, heads)
    GH.check_decode_step_path(w, res, GH.HostCopy(w), heads[:4], w.m, ws=res["ws"])


@pytest.mark.parametrize("chunk,exclusive", [(8192, True), (2048, True), (8192, False)])
def test_two_kernel_variants(chunk, exclusive):
    """Exclusive windows and per-head budgets on the two-kernel path (eight query
    heads per KV head), at the largest and a small chunk, and on the decode's
    virtual groups of four."""
    n_cap = 150000 if chunk == 8192 else 40000
    w = W().make_gqa(35, B=2, Hq=64, Hkv=8, d=128, n_cap=n_cap, seq_lens=[n_cap, n_cap - 1234], m=2000,
                     n_sink=3000, n_local=5000, device="cuda")
    _codes(w, "pool", 44)
    assert _plan(w)["chunk"] == chunk
    gen = torch.Generator(device="cuda").manual_seed(10)
    mph = torch.randint(0, 2001, (2, 64), generator=gen, device="cuda", dtype=torch.int32)
    heads = _sample(2, 64, 10, 2)
    _check_two_kernel(w, heads, exclusive=exclusive, m_per_head=mph)
    _check(w, heads, exclusive=exclusive, m_per_head=mph)


@pytest.mark.parametrize("Wd", [2, 4, 16])
def test_wide_codes_at_the_largest_chunk(Wd):
    """Codes of Wd words at the 8,192-token chunk (the shape of the bench's
    128-bit measurement), random codes."""
    B, Hq, Hkv, n_cap = 2, 32, 8, 160000
    w = W().make_gqa(36, B=B, Hq=Hq, Hkv=Hkv, d=128, n_cap=n_cap, seq_lens=[n_cap, 150001], m=4096,
                     n_sink=128, n_local=256, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(20 + Wd)
    w.k_sig = torch.randint(-2 ** 31, 2 ** 31 - 1, (B, Hkv, n_cap, Wd), generator=gen, device="cuda",
                            dtype=torch.int64).to(torch.int32).contiguous()
    w.q_sig = torch.randint(-2 ** 31, 2 ** 31 - 1, (B, Hq, Wd), generator=gen, device="cuda",
                            dtype=torch.int64).to(torch.int32).contiguous()
    plan = _plan(w, Wd)
    assert plan["fused"] == 0 and plan["chunk"] == 8192
    _check(w, _sample(B, Hq, 8, 3), code_words=Wd)


@pytest.mark.parametrize("n_cap,B,Hkv,chunk", [(10000, 2, 2, 1024), (40000, 2, 8, 2048), (80000, 2, 8, 4096),
                                                (150000, 2, 8, 8192)])
def test_score_entry_point_every_chunk(n_cap, B, Hkv, chunk):
    """hash_attn_score (distances and histograms) at each SCORE instantiation."""
    H = GH.ha()
    Hq = 4 * Hkv
    w = W().make_gqa(37, B=B, Hq=Hq, Hkv=Hkv, d=128, n_cap=n_cap, seq_lens=[n_cap, n_cap // 2 + 3], m=64,
                     n_sink=0, n_local=0, device="cuda")
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig)
    assert H.hash_attn_selection_plan(shape)["chunk"] == chunk
    ws = GH.workspace(shape, w.m, 0, 0)
    dist = torch.full((B, Hq, n_cap), 255, dtype=torch.uint8, device="cuda")
    hist = torch.zeros((B, Hq, 33), dtype=torch.int32, device="cuda")
    H.hash_attn_score(shape, w.q_sig, w.k_sig, w.seq_lens, dist, hist, workspace=ws)
    torch.cuda.synchronize()
    dist = dist.cpu().numpy()
    hist = hist.cpu().numpy()
    qs = w.q_sig.cpu().numpy()
    lens = w.seq_lens.cpu().numpy()
    for b, h in _sample(B, Hq, 6, 4):
        n = int(lens[b])
        ref = O.hamming_distances(int(qs[b, h]), w.k_sig[b, h // 4, :n].cpu().numpy())
        assert np.array_equal(dist[b, h, :n], ref)
        assert np.all(dist[b, h, n:] == 255)
        assert np.array_equal(hist[b, h], O.distance_histogram(ref))


def test_single_sequence_of_two_million_tokens():
    """One (sequence, KV head) of 2^21 tokens with four query heads: 256 ranges of
    the fused selection."""
    n = 1 << 21
    w = W().make_gqa(38, B=1, Hq=4, Hkv=1, d=128, n_cap=n, seq_lens=[n], m=65536, n_sink=128, n_local=256,
                     device="cuda")
    plan = _plan(w)
    assert plan["fused"] == 1 and plan["ranges"] == 256
    res = _check(w, [(0, h) for h in range(4)], att_heads=2)
    # the decode step without selection outputs: 256 ranges merged per head
    GH.check_decode_step_path(w, res, GH.HostCopy(w), [(0, 0), (0, 3)], w.m, ws=res["ws"])


def test_single_sequence_two_kernel_path_long():
    """One (sequence, KV head) of 2^21 tokens with eight query heads: the two-kernel
    path with its chunk raised so the segments fit GATHER-ATT's table, and the
    decode's two virtual groups of four over 256 ranges."""
    n = 1 << 21
    w = W().make_gqa(40, B=1, Hq=8, Hkv=1, d=128, n_cap=n, seq_lens=[n - 5], m=30000, n_sink=128, n_local=256,
                     device="cuda")
    plan = _plan(w)
    assert plan["fused"] == 1 and (n + plan["chunk"] - 1) // plan["chunk"] * 8 <= 4096
    heads = [(0, h) for h in range(0, 8, 3)]
    _check_two_kernel(w, heads, att_heads=2)
    res = _check(w, heads, att_heads=2)
    GH.check_decode_step_path(w, res, GH.HostCopy(w), heads[:2], w.m, ws=res["ws"])


# ---------------------------------------------------------------- dense path: one read per GQA group

DENSE_GROUP = [
    # name, B, Hq, Hkv, d, n_cap, lens, shared, kv dtype
    ("many_splits_ragged", 3, 8, 2, 128, 40000, [40000, 1, 0], False, "bf16"),
    ("d64_odd_lengths", 2, 4, 1, 64, 700, [700, 333], False, "bf16"),
    ("one_split", 2, 8, 2, 128, 50, [50, 17], False, "bf16"),
    ("shared_cache", 4, 8, 2, 128, 5000, [5000, 4999, 3, 2500], True, "bf16"),
    # one, two and three query heads per KV head; range boundaries and ragged tails
    ("g1_two_ranges", 2, 4, 4, 128, 9000, [9000, 8193], False, "bf16"),
    ("g2_d64_three_ranges", 2, 4, 2, 64, 17000, [17000, 123], False, "bf16"),
    ("g3_ragged_tail", 1, 6, 2, 128, 20000, [19999], False, "bf16"),
    # spans of 2,048 rows over 16 ranges of a long sequence (64 partials per head)
    ("long_sequence", 4, 8, 2, 128, 131072, [131072, 131071, 65536, 8191], False, "bf16"),
    # float32 K/V: the per-head kernel
    ("fp32_per_head", 2, 8, 2, 64, 3000, [3000, 1500], False, "f32"),
]


@pytest.mark.parametrize("case", DENSE_GROUP, ids=[c[0] for c in DENSE_GROUP])
def test_dense_group_kernel(case):
    """The dense path (m >= n_cap) reads each row once for the GQA group on
    bf16 K/V (1 to 4 query heads per KV head); every head must equal full
    attention over its sequence."""
    name, B, Hq, Hkv, d, n_cap, lens, shared, kvd = case
    w = W().make_gqa(39, B=B, Hq=Hq, Hkv=Hkv, d=d, n_cap=n_cap, seq_lens=lens, m=0, n_sink=0, n_local=0,
                     device="cuda", shared=shared, name=name,
                     kv_dtype=torch.bfloat16 if kvd == "bf16" else torch.float32)
    if kvd == "f32":
        w.q = w.q.float()
    res = GH.run_decode(w, m=n_cap, dense=True, m_per_seq=None, sel=False)
    assert res["status"] == 0, hex(res["flags"])
    hc = GH.HostCopy(w)
    GH.check_attention(res, hc, [(b, h) for b in range(B) for h in range(Hq)], n_cap, dense=True)
