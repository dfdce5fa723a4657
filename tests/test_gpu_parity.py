"""CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Selected index sets and Hamming distances/histograms must match bit for bit;
outputs within 2e-3 * (1 + |ref|) and lse within 1e-4 * (1 + |ref|).
"""
import math

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


def all_heads(w):
    return [(b, h) for b in range(w.B) for h in range(w.Hq)]


# ---------------------------------------------------------------- small shapes, many edge cases

SMALL = [
    # name, B, Hq, Hkv, d, n_cap, lens, m, S, Lw, kv dtype
    ("g1_d64_bf16", 1, 2, 2, 64, 1500, [1500], 64, 4, 16, torch.bfloat16),
    ("g4_ragged_tail", 2, 8, 2, 128, 5000, [5000, 3333], 300, 32, 64, torch.bfloat16),
    ("g8_two_passes", 1, 8, 1, 128, 3000, [2999], 100, 8, 8, torch.bfloat16),
    ("g2_d64", 3, 4, 2, 64, 2100, [2100, 1, 1025], 50, 3, 5, torch.bfloat16),
    ("fp32_d128", 1, 4, 1, 128, 1200, [1200], 77, 5, 9, torch.float32),
    ("fp32_d64", 1, 1, 1, 64, 1024, [1024], 64, 4, 16, torch.float32),
    ("windows_overlap", 2, 4, 1, 128, 200, [200, 150], 64, 128, 128, torch.bfloat16),
    ("budget_zero", 1, 4, 2, 128, 900, [900], 0, 16, 16, torch.bfloat16),
    ("empty_everything", 2, 4, 2, 128, 900, [900, 0], 0, 0, 0, torch.bfloat16),
    ("budget_at_n", 1, 4, 2, 128, 704, [700], 700, 0, 0, torch.bfloat16),
    ("budget_above_n", 2, 4, 2, 128, 704, [500, 704], 600, 8, 8, torch.bfloat16),
    ("chunk_edges", 3, 4, 1, 128, 8196, [8192, 8193, 1024], 512, 1, 1, torch.bfloat16),
    ("long_rows_many_splits", 1, 4, 1, 128, 40000, [40000], 9000, 64, 64, torch.bfloat16),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes(case):
    name, B, Hq, Hkv, d, n_cap, lens, m, S, Lw, kvdt = case
    w = W().make_gqa(7, B=B, Hq=Hq, Hkv=Hkv, d=d, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S,
                     n_local=Lw, device="cuda", kv_dtype=kvdt, name=name)
    if kvdt == torch.float32:
        w.q = w.q.float()
    res = GH.run_decode(w)
    assert res["status"] == 0, res["flags"]
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), m)
    GH.check_attention(res, hc, all_heads(w), m)
    # the decode step without selection outputs (the group kernel where it applies)
    GH.check_decode_step_path(w, res, hc, all_heads(w), m, ws=res["ws"])


def test_tie_heavy_codes():
    """Few distinct codes: the threshold bin holds most tokens; the index tie rule decides."""
    w = W().make_gqa(8, B=2, Hq=8, Hkv=2, d=128, n_cap=20000, seq_lens=[20000, 17001], m=1500,
                     n_sink=16, n_local=16, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(99)
    pool = torch.tensor([0x0F0F0F0F, 0x0F0F0F0E, 0x7F0F0F0F], dtype=torch.int64, device="cuda")
    pool = torch.where(pool >= 2**31, pool - 2**32, pool).to(torch.int32)
    pick = torch.randint(0, 3, w.k_sig.shape, generator=gen, device="cuda")
    w.k_sig = pool[pick].contiguous()
    w.q_sig = torch.full_like(w.q_sig, 0x0F0F0F0F)
    res = GH.run_decode(w)
    assert res["status"] == 0
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), w.m)
    GH.check_attention(res, hc, all_heads(w), w.m)
    GH.check_decode_step_path(w, res, hc, all_heads(w), w.m, ws=res["ws"])


def test_all_codes_equal_take_first_m():
    w = W().make_gqa(9, B=1, Hq=4, Hkv=1, d=128, n_cap=5000, seq_lens=[5000], m=333, n_sink=0,
                     n_local=0, device="cuda")
    w.k_sig = torch.full_like(w.k_sig, 12345)
    res = GH.run_decode(w)
    idx = res["sel_idx"].cpu().numpy()
    for h in range(4):
        assert int(res["sel_cnt"][0, h]) == 333
        assert np.array_equal(idx[0, h, :333], np.arange(333))


WINDOW_CASES = [
    # name, n, m, S, Lw, code pattern
    ("quota_ends_in_sink_window", 5000, 700, 1000, 300, "equal"),
    ("quota_ends_in_local_window", 5000, 900, 8, 300, "far_then_equal"),
    ("windows_span_many_chunks", 20000, 500, 7000, 9000, "random"),
    ("windows_meet_exactly", 6000, 100, 2500, 3500, "random"),
    ("windows_and_ties_random_pool", 9000, 1200, 1500, 2500, "pool"),
]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=[c[0] for c in WINDOW_CASES])
def test_windows_across_chunks_and_tie_boundary(case):
    """Windows that cover several chunks, and a tie quota that runs out inside a
    chunk the sink or the local window reaches (chunks are 1,024 tokens here)."""
    name, n, m, S, Lw, pattern = case
    w = W().make_gqa(17, B=2, Hq=4, Hkv=1, d=128, n_cap=n, seq_lens=[n, n - 333], m=m, n_sink=S,
                     n_local=Lw, device="cuda", name=name)
    q0 = 0x0F0F0F0F
    w.q_sig = torch.full_like(w.q_sig, q0)
    if pattern == "equal":
        w.k_sig = torch.full_like(w.k_sig, q0)
    elif pattern == "far_then_equal":
        ks = torch.full_like(w.k_sig, q0)
        ks[..., :4000] = ~torch.tensor(q0, dtype=torch.int32)
        w.k_sig = ks.contiguous()
    elif pattern == "pool":
        gen = torch.Generator(device="cuda").manual_seed(5)
        pool = torch.tensor([q0, q0 ^ 1, q0 ^ 3, q0 ^ 0x70000000], dtype=torch.int32, device="cuda")
        w.k_sig = pool[torch.randint(0, 4, w.k_sig.shape, generator=gen, device="cuda")].contiguous()
    res = GH.run_decode(w)
    assert res["status"] == 0, res["flags"]
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), m)
    GH.check_attention(res, hc, all_heads(w)[:4], m)
    GH.check_decode_step_path(w, res, hc, all_heads(w)[:4], m, ws=res["ws"])


VARIANT_CASES = [
    # name, n_cap, lens, m, S, Lw, codes ("random" | "pool"), exclusive, per-head budgets
    ("exclusive_random", 9000, [9000, 7001], 700, 64, 128, "random", True, False),
    ("exclusive_tie_pool", 9000, [9000, 8500], 1200, 1500, 2500, "pool", True, False),
    ("exclusive_quota_in_window_chunks", 5000, [5000, 4667], 900, 1000, 300, "pool", True, False),
    ("per_head_budgets", 6000, [6000, 3001], 500, 16, 32, "random", False, True),
    ("per_head_budgets_exclusive", 6000, [6000, 4444], 500, 300, 200, "pool", True, True),
]


@pytest.mark.parametrize("case", VARIANT_CASES, ids=[c[0] for c in VARIANT_CASES])
def test_selection_variants(case):
    """Exclusive windows (top-m over the tokens outside the windows) and per-head
    budgets through hash_attn_decode_ex, against the oracle."""
    name, n_cap, lens, m, S, Lw, codes, exclusive, per_head = case
    w = W().make_gqa(23, B=2, Hq=8, Hkv=2, d=128, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S, n_local=Lw,
                     device="cuda", name=name)
    if codes == "pool":
        q0 = 0x0F0F0F0F
        gen = torch.Generator(device="cuda").manual_seed(6)
        pool = torch.tensor([q0, q0 ^ 1, q0 ^ 3, q0 ^ 0x70000000], dtype=torch.int32, device="cuda")
        w.k_sig = pool[torch.randint(0, 4, w.k_sig.shape, generator=gen, device="cuda")].contiguous()
        w.q_sig = torch.full_like(w.q_sig, q0)
    mph = None
    if per_head:
        gen = torch.Generator(device="cuda").manual_seed(7)
        mph = torch.randint(0, m + 1, (2, 8), generator=gen, device="cuda", dtype=torch.int32)
        mph[0, 0], mph[1, 7] = 0, m
    res = GH.run_decode(w, exclusive=exclusive, m_per_head=mph)
    assert res["status"] == 0, res["flags"]
    hc = GH.HostCopy(w, exclusive=exclusive, m_per_head=mph)
    GH.check_selection(res, hc, all_heads(w), m)
    GH.check_attention(res, hc, all_heads(w)[::3], m)
    if exclusive:
        cnt = res["sel_cnt"].cpu().numpy()
        for b, n in enumerate(lens):
            W_ = len(O.window_positions(n, S, Lw))
            for h in range(8):
                mb = int(mph[b, h]) if per_head else m
                assert int(cnt[b, h]) == min(n, mb + W_)


@pytest.mark.parametrize("Wd,n_cap,lens,m,S,Lw,pool", [
    (2, 9000, [9000, 7001], 700, 16, 32, False),
    (4, 6000, [6000, 4321], 300, 64, 64, True),
    (16, 5000, [5000, 2500], 900, 8, 8, False),
])
def test_wide_codes(Wd, n_cap, lens, m, S, Lw, pool):
    """Codes of Wd 32-bit words through hash_attn_decode_ex against the oracle
    (the distance sums over the words; b + 1 bins)."""
    w = W().make_gqa(25, B=2, Hq=8, Hkv=2, d=128, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S, n_local=Lw,
                     device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(8 + Wd)
    if pool:   # few distinct codes: ties across chunks
        base = torch.randint(-2 ** 31, 2 ** 31 - 1, (5, Wd), generator=gen, device="cuda", dtype=torch.int64)
        pick = torch.randint(0, 5, (2, 2, n_cap), generator=gen, device="cuda")
        w.k_sig = base[pick].to(torch.int32).contiguous()
        w.q_sig = base[torch.zeros((2, 8), dtype=torch.int64, device="cuda")].to(torch.int32).contiguous()
    else:
        w.k_sig = torch.randint(-2 ** 31, 2 ** 31 - 1, (2, 2, n_cap, Wd), generator=gen, device="cuda",
                                dtype=torch.int64).to(torch.int32).contiguous()
        w.q_sig = torch.randint(-2 ** 31, 2 ** 31 - 1, (2, 8, Wd), generator=gen, device="cuda",
                                dtype=torch.int64).to(torch.int32).contiguous()
    res = GH.run_decode(w, code_words=Wd)
    assert res["status"] == 0, res["flags"]
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), m)
    GH.check_attention(res, hc, all_heads(w)[::3], m)


def test_per_head_budget_above_bound_is_flagged():
    H = GH.ha()
    w = W().make_gqa(24, B=1, Hq=4, Hkv=1, d=128, n_cap=3000, seq_lens=[3000], m=100, n_sink=4, n_local=4,
                     device="cuda")
    mph = torch.tensor([[100, 150, -3, 7]], dtype=torch.int32, device="cuda")
    res = GH.run_decode(w, m_per_head=mph)
    assert res["status"] == H.HA_ERR_DEVICE and res["flags"] & H.HA_DEVERR_BUDGET
    hc = GH.HostCopy(w, m_per_head=torch.tensor([[100, 100, 0, 7]], dtype=torch.int32))
    GH.check_selection(res, hc, all_heads(w), 100)
    # the decode step without selection outputs clamps and flags the same way
    grp = GH.run_decode(w, m_per_head=mph, sel=False)
    assert grp["status"] == H.HA_ERR_DEVICE and grp["flags"] & H.HA_DEVERR_BUDGET
    GH.check_attention(grp, hc, all_heads(w), 100)


def test_ragged_per_sequence_budget():
    lens = [4096, 9000, 1, 0, 12000, 6000]
    wl = W()
    mb = wl.ragged_budget(torch.tensor(lens, dtype=torch.int32))
    w = wl.make_gqa(5, B=6, Hq=8, Hkv=2, d=128, n_cap=12000, seq_lens=lens, m=int(mb.max()),
                    n_sink=64, n_local=128, device="cuda", m_per_seq=mb)
    res = GH.run_decode(w)
    assert res["status"] == 0
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), w.m)
    GH.check_attention(res, hc, all_heads(w), w.m)
    lse = res["lse"].cpu().numpy()
    assert np.all(lse[3] == -math.inf) and np.all(res["out"][3].cpu().numpy() == 0)


def test_shared_cache_batch_stride_zero():
    w = W().make_gqa(4, B=5, Hq=8, Hkv=2, d=128, n_cap=6000, seq_lens=6000, m=512, n_sink=128,
                     n_local=0, device="cuda", shared=True)
    assert w.K.shape[0] == 1
    res = GH.run_decode(w)
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), w.m)
    GH.check_attention(res, hc, all_heads(w), w.m)


def test_strided_views():
    """K/V and codes as views into larger buffers (padded token and head strides)."""
    base = W().make_gqa(10, B=2, Hq=4, Hkv=2, d=128, n_cap=3000, seq_lens=[2900, 3000], m=200,
                        n_sink=8, n_local=8, device="cuda")
    Kb = torch.zeros((2, 2, 3100, 136), dtype=torch.bfloat16, device="cuda")
    Vb = torch.zeros((2, 2, 3072, 128), dtype=torch.bfloat16, device="cuda")
    Kb[:, :, :3000, :128] = base.K
    Vb[:, :, :3000] = base.V
    Cb = torch.zeros((2, 2, 3004), dtype=torch.int32, device="cuda")
    Cb[:, :, :3000] = base.k_sig
    K = Kb[:, :, :3000, :128]
    V = Vb[:, :, :3000]
    base.k_sig = Cb[:, :, :3000]
    res = GH.run_decode(base, K=K, V=V)
    assert res["status"] == 0
    hc = GH.HostCopy(base, K=K, V=V)
    GH.check_selection(res, hc, all_heads(base), base.m)
    GH.check_attention(res, hc, all_heads(base), base.m)
    GH.check_decode_step_path(base, res, hc, all_heads(base), base.m, ws=res["ws"], K=K, V=V)


def test_dense_path_equals_full_attention():
    w = W().make_gqa(11, B=2, Hq=8, Hkv=2, d=128, n_cap=3000, seq_lens=[3000, 2222], m=0,
                     n_sink=0, n_local=0, device="cuda")
    res = GH.run_decode(w, m=3000, dense=True, m_per_seq=None)
    assert res["status"] == 0
    hc = GH.HostCopy(w)
    GH.check_attention(res, hc, all_heads(w), 3000, dense=True)


def test_repeated_calls_are_identical():
    w = W().make_gqa(12, B=2, Hq=8, Hkv=2, d=128, n_cap=9000, seq_lens=[9000, 8000], m=700,
                     n_sink=16, n_local=16, device="cuda")
    a = GH.run_decode(w)
    b = GH.run_decode(w, ws=a["ws"])
    c = GH.run_decode(w, ws=a["ws"])
    for r in (b, c):
        assert torch.equal(a["out"], r["out"]) and torch.equal(a["lse"], r["lse"])
        assert torch.equal(a["sel_idx"], r["sel_idx"])


# ---------------------------------------------------------------- stage entry points

def test_score_entry_point():
    H = GH.ha()
    w = W().make_gqa(13, B=2, Hq=8, Hkv=2, d=128, n_cap=7000, seq_lens=[7000, 4321], m=64,
                     n_sink=0, n_local=0, device="cuda")
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig)
    ws = GH.workspace(shape, w.m, 0, 0)
    dist = torch.full((2, 8, 7000), 255, dtype=torch.uint8, device="cuda")
    hist = torch.zeros((2, 8, 33), dtype=torch.int32, device="cuda")
    H.hash_attn_score(shape, w.q_sig, w.k_sig, w.seq_lens, dist, hist, workspace=ws)
    torch.cuda.synchronize()
    dist = dist.cpu().numpy()
    hist = hist.cpu().numpy()
    qs = w.q_sig.cpu().numpy()
    for b, n in [(0, 7000), (1, 4321)]:
        for h in range(8):
            ref = O.hamming_distances(int(qs[b, h]), w.k_sig[b, h // 4, :n].cpu().numpy())
            assert np.array_equal(dist[b, h, :n], ref)
            assert np.all(dist[b, h, n:] == 255)
            assert np.array_equal(hist[b, h], O.distance_histogram(ref))


def test_select_entry_point_matches_decode():
    H = GH.ha()
    w = W().make_gqa(14, B=2, Hq=8, Hkv=2, d=128, n_cap=10000, seq_lens=[10000, 7777], m=600,
                     n_sink=32, n_local=48, device="cuda")
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig)
    ws = GH.workspace(shape, w.m, w.n_sink, w.n_local)
    cap = H.hash_attn_select_capacity(10000, 600, 32, 48)
    sel = torch.empty((2, 8, cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((2, 8), dtype=torch.int32, device="cuda")
    H.hash_attn_select(shape, w.q_sig, w.k_sig, w.seq_lens, None, 600, 32, 48, sel, cnt, workspace=ws)
    res = {"sel_idx": sel, "sel_cnt": cnt, "cap": cap}
    GH.check_selection(res, GH.HostCopy(w), all_heads(w), 600)
    dec = GH.run_decode(w)
    assert torch.equal(dec["sel_idx"], sel) and torch.equal(dec["sel_cnt"], cnt)


def test_gather_att_entry_point_with_given_lists():
    H = GH.ha()
    w = W().make_gqa(15, B=2, Hq=4, Hkv=2, d=128, n_cap=5000, seq_lens=[5000, 3000], m=0,
                     n_sink=0, n_local=0, device="cuda")
    rng = np.random.default_rng(0)
    cap = 700
    idx = np.full((2, 4, cap), -1, dtype=np.int32)
    cnt = np.zeros((2, 4), dtype=np.int32)
    lists = {}
    for b, n in [(0, 5000), (1, 3000)]:
        for h in range(4):
            k = int(rng.integers(0, cap + 1))
            sel = rng.choice(n, size=k, replace=False)       # unsorted on purpose
            idx[b, h, :k] = sel
            cnt[b, h] = k
            lists[(b, h)] = np.sort(sel)
    shape = H.make_shape(w.q, w.K, w.V)
    ws = GH.workspace(shape, cap, 0, 0)
    out = torch.empty((2, 4, 128), device="cuda")
    lse = torch.empty((2, 4), device="cuda")
    H.hash_attn_gather_att(shape, w.q, w.K, w.V, w.seq_lens, torch.from_numpy(idx).cuda(), cap,
                           torch.from_numpy(cnt).cuda(), out, lse, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, flags
    hc = GH.HostCopy(w)
    for (b, h), sel in lists.items():
        Kh, Vh = hc.kv(b, h // 2)
        ro, rl = O.attend(hc.q[b, h], Kh, Vh, sel)
        GH.assert_out_close(out[b, h].cpu().numpy(), ro, f"({b},{h})")
        GH.assert_lse_close(float(lse[b, h]), rl, f"({b},{h})")
    # an index outside [0, seq_len) is skipped and flagged
    idx[1, 0, 0] = 3000
    cnt[1, 0] = max(cnt[1, 0], 1)
    H.hash_attn_gather_att(shape, w.q, w.K, w.V, w.seq_lens, torch.from_numpy(idx).cuda(), cap,
                           torch.from_numpy(cnt).cuda(), out, lse, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    assert st == H.HA_ERR_DEVICE and flags & H.HA_DEVERR_INDEX


def test_merge_entry_point():
    H = GH.ha()
    rng = np.random.default_rng(1)
    rows, d = 37, 128
    oa = rng.standard_normal((rows, d)).astype(np.float32)
    ob = rng.standard_normal((rows, d)).astype(np.float32)
    la = (rng.standard_normal(rows) * 3).astype(np.float32)
    lb = (rng.standard_normal(rows) * 3).astype(np.float32)
    la[3] = -np.inf
    lb[5] = -np.inf
    la[7] = lb[7] = -np.inf
    t = lambda a: torch.from_numpy(a).cuda()
    out = torch.empty((rows, d), device="cuda")
    lse = torch.empty(rows, device="cuda")
    H.hash_attn_merge(t(oa), t(la), t(ob), t(lb), out, lse, rows, d)
    torch.cuda.synchronize()
    for r in range(rows):
        ro, rl = O.merge(oa[r], float(la[r]), ob[r], float(lb[r]))
        GH.assert_out_close(out[r].cpu().numpy(), ro, f"row {r}")
        GH.assert_lse_close(float(lse[r]), rl, f"row {r}")
    # in place (out aliases out_a)
    A, LA = t(oa.copy()), t(la.copy())
    H.hash_attn_merge(A, LA, t(ob), t(lb), A, LA, rows, d)
    torch.cuda.synchronize()
    assert torch.allclose(A, out) and torch.equal(LA.isinf(), lse.isinf())


@pytest.mark.parametrize("nseg,d", [(1, 128), (2, 64), (3, 128), (5, 128)])
def test_merge_n_entry_point(nseg, d):
    """Multi-segment merge against the oracle: empty segments and empty rows, a
    padded segment stride, and the output aliasing segment 0."""
    H = GH.ha()
    rng = np.random.default_rng(10 + nseg)
    rows = 41
    outs = rng.standard_normal((nseg, rows + 3, d)).astype(np.float32)  # 3 padding rows per segment
    lses = (rng.standard_normal((nseg, rows + 5)) * 4).astype(np.float32)
    lses[0, 2] = -np.inf
    lses[:, 9] = -np.inf
    if nseg > 1:
        lses[nseg - 1, 11:20] = -np.inf
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    O_d, L_d = t(outs), t(lses)
    ov, lv = O_d[:, :rows], L_d[:, :rows]   # views with segment strides (rows + 3) * d and rows + 5
    out = torch.empty((rows, d), device="cuda")
    lse = torch.empty(rows, device="cuda")
    H.hash_attn_merge_n(ov, lv, out, lse)
    torch.cuda.synchronize()
    for r in range(rows):
        ro, rl = O.merge_segments(outs[:, r], lses[:, r])
        GH.assert_out_close(out[r].cpu().numpy(), ro, f"row {r}")
        GH.assert_lse_close(float(lse[r]), rl, f"row {r}")
    assert torch.all(out[9] == 0) and bool(lse[9].isneginf())
    # in place: the result overwrites segment 0
    H.hash_attn_merge_n(ov, lv, ov[0], lv[0])
    torch.cuda.synchronize()
    assert torch.allclose(ov[0], out) and torch.equal(lv[0].isinf(), lse.isinf())


@pytest.mark.parametrize("d,q_dtype", [(128, torch.float32), (128, torch.bfloat16), (64, torch.bfloat16)])
def test_encode_queries_and_keys(d, q_dtype):
    """Sign-projection codes against the oracle: every bit that float32 rounding
    cannot flip must match; appended keys land at their positions only."""
    H = GH.ha()
    B, Hq, Hkv, n_cap = 3, 8, 2, 64
    gen = torch.Generator(device="cuda").manual_seed(19 + d)
    q = torch.randn((B, Hq, d), generator=gen, device="cuda").to(q_dtype)
    K = torch.randn((B, Hkv, n_cap, d), generator=gen, device="cuda").to(torch.bfloat16)
    V = torch.zeros_like(K)
    W = torch.randn((Hkv, 32, d), generator=gen, device="cuda")
    k_sig = torch.full((B, Hkv, n_cap), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    shape = H.make_shape(q, K, V, k_sig)
    q_sig = torch.zeros((B, Hq), dtype=torch.int32, device="cuda")
    H.hash_attn_encode_queries(shape, q, W, q_sig)
    pos = torch.tensor([17, -1, n_cap - 1], dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = k_sig.clone()
    H.hash_attn_encode_keys(shape, K, W, pos, k_sig, flags)
    torch.cuda.synchronize()
    Wn = W.cpu().numpy().astype(np.float64)
    qn = q.float().cpu().numpy()
    Kn = K.float().cpu().numpy()
    G = Hq // Hkv
    got_q = q_sig.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    for b in range(B):
        for h in range(Hq):
            ref = O.encode(qn[b, h], Wn[h // G])
            amb = O.encode_ambiguous(qn[b, h], Wn[h // G])
            assert (int(got_q[b, h]) ^ ref) & ~amb & 0xFFFFFFFF == 0, (b, h, hex(int(got_q[b, h])), hex(ref))
    got_k = k_sig.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    exp_k = before.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    for b, p_ in enumerate([17, -1, n_cap - 1]):
        for g in range(Hkv):
            if p_ < 0:
                continue
            ref = O.encode(Kn[b, g, p_], Wn[g])
            amb = O.encode_ambiguous(Kn[b, g, p_], Wn[g])
            assert (int(got_k[b, g, p_]) ^ ref) & ~amb & 0xFFFFFFFF == 0, (b, g)
            exp_k[b, g, p_] = got_k[b, g, p_]
    assert np.array_equal(got_k, exp_k), "codes outside the appended positions changed"
    assert int(flags.item()) & H.HA_DEVERR_INDEX


@pytest.mark.parametrize("mode", ["sparse", "budgets", "dense", "packed"])
def test_decode_host_buffers_equal_device_decode(mode):
    """hash_attn_decode_host (inputs and results in pinned host memory) gives the
    outputs of hash_attn_decode on device copies of the same inputs, bit for bit,
    for the sparse path, per-sequence budgets and the dense path (no codes); in
    "packed" the inputs sit back to back in one host buffer at the staging offsets
    (merged copies) and out / lse in another."""
    H = GH.ha()
    w = W().make_gqa(47, B=3, Hq=8, Hkv=2, d=128, n_cap=3000, seq_lens=[3000, 1999, 2500], m=200, n_sink=16,
                     n_local=16, device="cuda", m_per_seq=[200, 150, 64] if mode == "budgets" else None)
    m = 4000 if mode == "dense" else w.m
    res = GH.run_decode(w, m=m, sel=False, dense=(mode == "dense"))
    assert res["status"] == 0
    q_strided = torch.empty((3, 8, 256), dtype=w.q.dtype, device="cuda")[:, :, :128]
    q_strided.copy_(w.q)                         # the host call ignores the shape's q strides
    shape = H.make_shape(q_strided, w.K, w.V, w.k_sig)
    ws = GH.workspace(shape, m, w.n_sink, w.n_local)
    staging = torch.empty(H.hash_attn_host_staging_size(shape), dtype=torch.uint8, device="cuda")
    pin = lambda t: t.cpu().contiguous().pin_memory()
    q_h, sig_h, sl_h = pin(w.q), pin(w.q_sig), pin(w.seq_lens)
    mps_h = pin(w.m_per_seq) if w.m_per_seq is not None else None
    out_h = torch.full((3, 8, 128), float("nan")).pin_memory()
    lse_h = torch.full((3, 8), float("nan")).pin_memory()
    if mode == "packed":
        # q (6,144 bytes), q_sig (96 bytes) and seq_lens (12 bytes) back to back: the
        # first two and the lengths follow each other at 16-byte staging boundaries
        qb, sb = w.q.numel() * 2, w.q_sig.numel() * 4
        buf = torch.empty(qb + sb + 12, dtype=torch.uint8).pin_memory()
        buf[:qb].copy_(w.q.cpu().contiguous().view(torch.uint8).view(-1))
        buf[qb:qb + sb].copy_(w.q_sig.cpu().contiguous().view(torch.uint8).view(-1))
        buf[qb + sb:].copy_(w.seq_lens.cpu().contiguous().view(torch.uint8).view(-1))
        q_h, sig_h, sl_h = buf[:qb], buf[qb:qb + sb], buf[qb + sb:]
        res_buf = torch.full((3 * 8 * 128 + 3 * 8,), float("nan")).pin_memory()
        out_h, lse_h = res_buf[:3 * 8 * 128].view(3, 8, 128), res_buf[3 * 8 * 128:].view(3, 8)
    H.hash_attn_decode_host(shape, q_h, None if mode == "dense" else sig_h, sl_h, mps_h,
                            None if mode == "dense" else w.k_sig, w.K, w.V, m, w.n_sink, w.n_local, out_h, lse_h,
                            staging=staging, workspace=ws)
    torch.cuda.current_stream().synchronize()
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, flags
    assert torch.equal(out_h, res["out"].cpu()) and torch.equal(lse_h, res["lse"].cpu())


@pytest.mark.parametrize("d,q_dtype,hidden", [(128, torch.float32, 128), (64, torch.bfloat16, 64),
                                              (128, torch.bfloat16, 32)])
def test_encode_mlp_queries_and_keys(d, q_dtype, hidden):
    """MLP-map codes against the oracle: every bit outside the float32 error bound
    of the three layers must match; appended keys land at their positions only;
    20 query vectors per KV head leave a ragged last CTA."""
    H = GH.ha()
    B, Hq, Hkv, n_cap = 5, 8, 2, 64
    gen = torch.Generator(device="cuda").manual_seed(61 + d + hidden)
    q = torch.randn((B, Hq, d), generator=gen, device="cuda").to(q_dtype)
    K = torch.randn((B, Hkv, n_cap, d), generator=gen, device="cuda").to(torch.bfloat16)
    wts = W().mlp_weights(29, Hkv, d, hidden, device="cuda")
    mw = H.mlp(*wts)
    k_sig = torch.full((B, Hkv, n_cap), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    shape = H.make_shape(q, K, torch.zeros_like(K), k_sig)
    q_sig = torch.zeros((B, Hq), dtype=torch.int32, device="cuda")
    H.hash_attn_encode_queries_mlp(shape, q, mw, q_sig)
    pos_l = [17, -1, n_cap - 1, 0, 40]
    pos = torch.tensor(pos_l, dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = k_sig.clone()
    H.hash_attn_encode_keys_mlp(shape, K, mw, pos, k_sig, flags)
    torch.cuda.synchronize()
    wn = [t.double().cpu().numpy() for t in wts]
    qn, Kn = q.double().cpu().numpy(), K.double().cpu().numpy()
    G = Hq // Hkv
    got_q = q_sig.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    for b in range(B):
        for h in range(Hq):
            args = [t[h // G] for t in wn]
            ref, amb = O.encode_mlp(qn[b, h], *args), O.encode_mlp_ambiguous(qn[b, h], *args)
            assert (int(got_q[b, h]) ^ ref) & ~amb & 0xFFFFFFFF == 0, (b, h, hex(int(got_q[b, h])), hex(ref))
    got_k = k_sig.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    exp_k = before.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    for b, p_ in enumerate(pos_l):
        for g in range(Hkv):
            if p_ < 0:
                continue
            args = [t[g] for t in wn]
            ref, amb = O.encode_mlp(Kn[b, g, p_], *args), O.encode_mlp_ambiguous(Kn[b, g, p_], *args)
            assert (int(got_k[b, g, p_]) ^ ref) & ~amb & 0xFFFFFFFF == 0, (b, g)
            exp_k[b, g, p_] = got_k[b, g, p_]
    assert np.array_equal(got_k, exp_k), "codes outside the appended positions changed"
    assert int(flags.item()) & H.HA_DEVERR_INDEX


@pytest.mark.parametrize("kind,exclusive,Hq", [("sign", False, 8), ("mlp", False, 8), ("mlp", True, 8),
                                               ("sign", False, 16)])
def test_decode_mapped_runs_the_map_ahead_of_score(kind, exclusive, Hq):
    """One decode step from raw q: the map writes the appended tokens' key codes
    and the query codes (as the stand-alone encoders give them, and matching the
    oracle's unambiguous bits), and the rest of the step equals
    hash_attn_decode on those codes, bit for bit (four and eight query heads per
    KV head: groups of two, and of four, per KV head on this small grid)."""
    import copy
    H = GH.ha()
    w = W().make_gqa(41, B=3, Hq=Hq, Hkv=2, d=128, n_cap=4000, seq_lens=[4000, 3001, 1234], m=300, n_sink=16,
                     n_local=32, device="cuda")
    pos = (w.seq_lens - 1).to(torch.int32)
    k_sig = w.k_sig.clone()
    for b, p_ in enumerate(pos.tolist()):
        k_sig[b, :, p_] = 0x5A5A5A5A            # stale: the map must rewrite it
    stale = k_sig.clone()
    gen = torch.Generator(device="cuda").manual_seed(43)
    if kind == "sign":
        Wp = torch.randn((2, 32, 128), generator=gen, device="cuda")
        map_ = H.sign_map(Wp)
    else:
        wts = W().mlp_weights(31, 2, 128, 128, device="cuda")
        mw = H.mlp(*wts)
        map_ = H.mlp_map(mw)
    shape = H.make_shape(w.q, w.K, w.V, k_sig)
    ws = GH.workspace(shape, w.m, w.n_sink, w.n_local)
    B, Hq, d = w.q.shape
    q_sig = torch.zeros((B, Hq), dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    cap = H.hash_attn_select_capacity(4000, w.m, w.n_sink, w.n_local)
    sel_idx = torch.full((B, Hq, cap), -7, dtype=torch.int32, device="cuda")
    sel_cnt = torch.full((B, Hq), -7, dtype=torch.int32, device="cuda")
    opts = H.select_opts(None, True) if exclusive else None
    H.hash_attn_decode_mapped(shape, w.q, map_, pos, q_sig, k_sig, w.K, w.V, w.seq_lens, None, w.m, w.n_sink,
                              w.n_local, opts, out, lse, sel_idx, sel_cnt, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, flags
    q_ref = torch.zeros_like(q_sig)
    k_ref = stale.clone()
    if kind == "sign":
        H.hash_attn_encode_queries(shape, w.q, Wp, q_ref)
        H.hash_attn_encode_keys(shape, w.K, Wp, pos, k_ref)
    else:
        H.hash_attn_encode_queries_mlp(shape, w.q, mw, q_ref)
        H.hash_attn_encode_keys_mlp(shape, w.K, mw, pos, k_ref)
    torch.cuda.synchronize()
    assert torch.equal(q_sig, q_ref) and torch.equal(k_sig, k_ref)
    changed = (k_sig != stale).nonzero().tolist()
    assert all(i == pos[b].item() for b, _, i in changed)
    Kn = w.K.double().cpu().numpy()
    for b, p_ in enumerate(pos.tolist()):     # the appended keys against the oracle
        for g in range(2):
            x = Kn[b, g, p_]
            if kind == "sign":
                Wn = Wp[g].double().cpu().numpy()
                ref, amb = O.encode(x, Wn), O.encode_ambiguous(x, Wn)
            else:
                args = [t[g].double().cpu().numpy() for t in wts]
                ref, amb = O.encode_mlp(x, *args), O.encode_mlp_ambiguous(x, *args)
            assert (int(k_sig[b, g, p_].item()) & 0xFFFFFFFF ^ ref) & ~amb & 0xFFFFFFFF == 0, (b, g)
    w2 = copy.copy(w)
    w2.q_sig, w2.k_sig = q_sig, k_sig
    res = GH.run_decode(w2, exclusive=exclusive)
    assert res["status"] == 0
    assert torch.equal(res["out"], out) and torch.equal(res["lse"], lse)
    assert torch.equal(res["sel_cnt"], sel_cnt) and torch.equal(res["sel_idx"], sel_idx)


@pytest.mark.parametrize("d,kv_dtype,m", [(128, torch.bfloat16, 100), (128, torch.bfloat16, 2500),
                                           (64, torch.float32, 37), (128, torch.bfloat16, 5000)])
def test_topk_exact_and_recall(d, kv_dtype, m):
    """Exact top-m by dot score against the oracle (tokens inside the float32 band
    around the boundary may go either way, the count is exact), then the recall of
    the hashed selection against it."""
    H = GH.ha()
    w = W().make_gqa(21, B=2, Hq=8, Hkv=2, d=d, n_cap=3000, seq_lens=[3000, 2222], m=300, n_sink=16,
                     n_local=16, device="cuda", kv_dtype=kv_dtype)
    if kv_dtype == torch.float32:
        w.q = w.q.float()
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig)
    ws = torch.empty(H.hash_attn_topk_exact_workspace_size(shape), dtype=torch.uint8, device="cuda")
    cap = min(m, 3000)
    idx = torch.full((2, 8, cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((2, 8), -7, dtype=torch.int32, device="cuda")
    H.hash_attn_topk_exact(shape, w.q, w.K, w.seq_lens, m, idx, cnt, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, flags
    qn, Kn = w.q.float().cpu().numpy(), w.K.float().cpu().numpy()
    idx_h, cnt_h = idx.cpu().numpy(), cnt.cpu().numpy()
    for b, n in enumerate([3000, 2222]):
        for h in range(8):
            k = min(m, n)
            assert int(cnt_h[b, h]) == k
            got = idx_h[b, h, :k]
            assert np.all(np.diff(got) > 0) and np.all(idx_h[b, h, k:] == -1)
            sure, band = O.top_m_band(qn[b, h], Kn[b, h // 4], n, m)
            assert set(sure) <= set(got) <= set(sure) | set(band), (b, h)
    # recall of the hashed selection against the exact top-m
    res = GH.run_decode(w)
    rec = torch.empty(16, device="cuda")
    H.hash_attn_recall(res["sel_idx"], res["sel_cnt"], idx, cnt, rec)
    torch.cuda.synchronize()
    sel_h, scnt_h = res["sel_idx"].cpu().numpy(), res["sel_cnt"].cpu().numpy()
    for b in range(2):
        for h in range(8):
            want = O.recall(sel_h[b, h, :scnt_h[b, h]], idx_h[b, h, :cnt_h[b, h]])
            assert abs(float(rec[b * 8 + h]) - want) < 1e-6


def test_topk_exact_timed_equals_untimed():
    """The events variant records its three events and returns the same selection."""
    H = GH.ha()
    w = W().make_gqa(24, B=2, Hq=8, Hkv=2, d=128, n_cap=5000, seq_lens=[5000, 4100], m=256, n_sink=0,
                     n_local=0, device="cuda")
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig)
    ws = torch.empty(H.hash_attn_topk_exact_workspace_size(shape), dtype=torch.uint8, device="cuda")
    outs = []
    for timed in (False, True):
        idx = torch.full((2, 8, 256), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((2, 8), -7, dtype=torch.int32, device="cuda")
        if timed:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            for e in ev:
                e.record()
            H.hash_attn_topk_exact_timed(shape, w.q, w.K, w.seq_lens, 256, idx, cnt, ev, workspace=ws)
        else:
            H.hash_attn_topk_exact(shape, w.q, w.K, w.seq_lens, 256, idx, cnt, workspace=ws)
        torch.cuda.synchronize()
        outs.append((idx.cpu(), cnt.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert ev[0].elapsed_time(ev[1]) > 0 and ev[1].elapsed_time(ev[2]) > 0


def test_topk_exact_ties_take_smaller_indices():
    H = GH.ha()
    w = W().make_gqa(22, B=1, Hq=4, Hkv=1, d=128, n_cap=2048, seq_lens=[2048], m=64, n_sink=0, n_local=0,
                     device="cuda")
    w.K[:] = w.K[:, :, :1]                       # every row equal: every score ties
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig)
    ws = torch.empty(H.hash_attn_topk_exact_workspace_size(shape), dtype=torch.uint8, device="cuda")
    idx = torch.empty((1, 4, 300), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    H.hash_attn_topk_exact(shape, w.q, w.K, w.seq_lens, 300, idx, cnt, workspace=ws)
    torch.cuda.synchronize()
    for h in range(4):
        assert int(cnt[0, h]) == 300 and torch.equal(idx[0, h].cpu(), torch.arange(300, dtype=torch.int32))


def _exact_call(H, shape, q, K, seq_lens, m, B, Hq, n_cap):
    """Run the exact comparator; returns (scores [B, Hq, n_cap] from the
    workspace, idx, cnt). The scores follow the 256-byte error word."""
    ws = torch.empty(H.hash_attn_topk_exact_workspace_size(shape), dtype=torch.uint8, device="cuda")
    cap = min(m, n_cap)
    idx = torch.full((B, Hq, cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, Hq), -7, dtype=torch.int32, device="cuda")
    H.hash_attn_topk_exact(shape, q, K, seq_lens, m, idx, cnt, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, flags
    z = ws[256:256 + B * Hq * n_cap * 4].view(torch.float32).view(B, Hq, n_cap)
    return z.cpu(), idx.cpu().numpy(), cnt.cpu().numpy()


# (Hq, Hkv, d, q dtype, kv dtype): groups of 1, 4, 8, 10, 16 and 21 heads take
# the tensor-core kernel for bf16 keys (3 G <= 64 columns: N = 16, 32, 48, 64),
# 24 heads and float32 keys the CUDA-core one
EXACT_SHAPES = [(8, 2, 128, torch.float32, torch.bfloat16), (8, 8, 64, torch.float32, torch.bfloat16),
                (16, 2, 128, torch.float32, torch.bfloat16), (20, 2, 64, torch.bfloat16, torch.bfloat16),
                (32, 2, 128, torch.float32, torch.bfloat16), (21, 1, 64, torch.float32, torch.bfloat16),
                (24, 1, 128, torch.float32, torch.bfloat16), (8, 2, 128, torch.float32, torch.float32)]


@pytest.mark.parametrize("Hq,Hkv,d,q_dtype,kv_dtype", EXACT_SHAPES)
def test_exact_scores_one_hot_keys_are_exact(Hq, Hkv, d, q_dtype, kv_dtype):
    """Keys with one non-zero entry, a power of two, make every score a single
    product: z[b, h, i] = 2^e_i q[b, h, j_i] exactly, in any summation order, so
    the scores must match bit for bit (this pins the dimension order, the head
    order and, for a float32 query, the split of q into three bf16 parts). Equal
    scores recur, so the top-m also checks that ties go to the smaller index."""
    H = GH.ha()
    B, n_cap, lens, m = 2, 1000, [1000, 333], 150
    g_ = torch.Generator().manual_seed(31)
    q = torch.randn((B, Hq, d), generator=g_).to(q_dtype)
    i = torch.arange(n_cap)
    scale = torch.pow(2.0, (i % 5).double() - 2.0)
    K = torch.zeros((B, Hkv, n_cap, d), dtype=torch.float64)
    col = torch.empty((B, Hkv, n_cap), dtype=torch.int64)
    for b in range(B):
        for g in range(Hkv):
            col[b, g] = (7 * i + 3 * g + b) % d
            K[b, g, i, col[b, g]] = scale
    Kd, qd = K.to(kv_dtype).cuda(), q.cuda()
    V = torch.zeros_like(Kd)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    shape = H.make_shape(qd, Kd, V)
    z, idx, cnt = _exact_call(H, shape, qd, Kd, seq, m, B, Hq, n_cap)
    G = Hq // Hkv
    q64 = q.double()
    for b, n in enumerate(lens):
        for h in range(Hq):
            want = (q64[b, h, col[b, h // G, :n]] * scale[:n]).float()
            assert torch.equal(z[b, h, :n], want), (b, h)
            assert int(cnt[b, h]) == min(m, n)
            ref = O.top_m_by_dot(q64[b, h].numpy(), K[b, h // G].numpy(), n, m)
            assert np.array_equal(idx[b, h, :min(m, n)], ref), (b, h)


@pytest.mark.parametrize("n_cap,lens,shared", [(100, [100, 37], False), (8, [8, 5], False),
                                              (700, [700, 640], True)])
def test_exact_scores_small_and_shared_caches(n_cap, lens, shared):
    """Caches shorter than one 128-row tile (the tile reads past n_cap as zeros
    and nothing past n is written), and one cache shared by every batch entry
    (batch stride 0): one-hot keys make the scores exact."""
    H = GH.ha()
    B, Hq, Hkv, d, m = 2, 8, 2, 128, 20
    g_ = torch.Generator().manual_seed(41)
    q = torch.randn((B, Hq, d), generator=g_)
    i = torch.arange(n_cap)
    Bk = 1 if shared else B
    K = torch.zeros((Bk, Hkv, n_cap, d), dtype=torch.float64)
    col = torch.empty((Bk, Hkv, n_cap), dtype=torch.int64)
    for b in range(Bk):
        for g in range(Hkv):
            col[b, g] = (3 * i + 5 * g + b) % d
            K[b, g, i, col[b, g]] = torch.pow(2.0, (i % 4).double() - 1.0)
    Kd, qd = K.to(torch.bfloat16).cuda(), q.cuda()
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    shape = H.make_shape(qd, Kd, torch.zeros_like(Kd))
    assert (shape.k_sb == 0) == shared
    ws = torch.full((H.hash_attn_topk_exact_workspace_size(shape),), 0x7F, dtype=torch.uint8, device="cuda")
    cap = min(m, n_cap)
    idx = torch.full((B, Hq, cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, Hq), -7, dtype=torch.int32, device="cuda")
    H.hash_attn_topk_exact(shape, qd, Kd, seq, m, idx, cnt, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, flags
    z = ws[256:256 + B * Hq * n_cap * 4].view(torch.float32).view(B, Hq, n_cap).cpu()
    untouched = torch.full((1,), 0x7F7F7F7F, dtype=torch.int32).view(torch.float32)
    G = Hq // Hkv
    for b, n in enumerate(lens):
        bk = 0 if shared else b
        for h in range(Hq):
            want = (q.double()[b, h, col[bk, h // G, :n]] * torch.pow(2.0, (i[:n] % 4).double() - 1.0)).float()
            assert torch.equal(z[b, h, :n], want), (b, h)
            assert torch.all(z[b, h, n:].view(torch.int32) == untouched.view(torch.int32)), (b, h)
            ref = O.top_m_by_dot(q.double()[b, h].numpy(), K[bk, h // G].numpy(), n, m)
            assert int(cnt[b, h]) == min(m, n)
            assert np.array_equal(idx[b, h, :min(m, n)].cpu().numpy(), ref), (b, h)


@pytest.mark.parametrize("Hq,Hkv,d,q_dtype,kv_dtype", EXACT_SHAPES)
def test_exact_scores_within_float32_bound(Hq, Hkv, d, q_dtype, kv_dtype):
    """Random keys and queries: every score within d 2^-22 sum_k |q_k k_ik| of the
    float64 dot product (the band the selection check uses), and the top-m inside
    the oracle's band."""
    H = GH.ha()
    lens, m = [3000, 2222], 300
    w = W().make_gqa(23, B=2, Hq=Hq, Hkv=Hkv, d=d, n_cap=3000, seq_lens=lens, m=m, n_sink=0, n_local=0,
                     device="cuda", kv_dtype=kv_dtype)
    q = w.q.to(q_dtype)
    shape = H.make_shape(q, w.K, w.V, w.k_sig)
    z, idx, cnt = _exact_call(H, shape, q, w.K, w.seq_lens, m, 2, Hq, 3000)
    qn, Kn = q.double().cpu().numpy(), w.K.double().cpu().numpy()
    G = Hq // Hkv
    for b, n in enumerate(lens):
        for h in range(Hq):
            Kh = Kn[b, h // G, :n]
            exact = O.dot_scores(qn[b, h], Kh, n)
            bound = d * 2.0 ** -22 * (np.abs(Kh) @ np.abs(qn[b, h]))
            assert np.all(np.abs(z[b, h, :n].double().numpy() - exact) <= bound), (b, h)
            k = min(m, n)
            assert int(cnt[b, h]) == k
            sure, band = O.top_m_band(qn[b, h], Kn[b, h // G], n, m)
            assert set(sure) <= set(idx[b, h, :k]) <= set(sure) | set(band), (b, h)


@pytest.mark.parametrize("n_cap,pattern", [(131072, "sampled_high"), (131072, "sampled_low"),
                                            (131072, "random"), (300000, "random"), (131072, "outliers"),
                                            (131072, "clustered")])
def test_topk_exact_at_length(n_cap, pattern):
    """The top-m at full context length. The selection estimates its threshold
    from blocks of 8 tokens out of every 136 (n = 131072); keys whose scores are
    large exactly on those tokens (or exactly off them) make the estimate miss
    in both directions, and 300000 tokens exceed the bitmap, so the general
    radix path is checked at length too. A few huge keys put the largest score
    far above the rest (past the reach of the one-pass 16-bit histograms), and
    clustered scores put thousands of tokens in the k-th key's 16-bit prefix,
    so the shared-memory radix fallbacks run as well. One-hot keys give exact
    scores; random keys are checked against the oracle's float32 band."""
    H = GH.ha()
    B, Hq, Hkv, d, m = 1, 4, 1, 64, 4096
    g_ = torch.Generator().manual_seed(37)
    if pattern == "random":
        K = torch.randn((B, Hkv, n_cap, d), generator=g_).to(torch.bfloat16)
        q = torch.randn((B, Hq, d), generator=g_)
    elif pattern == "outliers":
        # exact one-hot scores, three of them 2^60 times larger than the rest
        i = torch.arange(n_cap)
        K = torch.zeros((B, Hkv, n_cap, d), dtype=torch.float64)
        K[0, 0, i, (5 * i) % d] = torch.pow(2.0, (i % 3).double())
        K[0, 0, [5, 70000, 131000]] *= 2.0 ** 60
        K = K.to(torch.bfloat16)
        q = torch.rand((B, Hq, d), generator=g_) + 0.5
    elif pattern == "clustered":
        # exact scores q[c] * 2^e with q[c] = 1 + c / 4096, tokens spread over four groups by a
        # fixed permutation: 3000 spread over 16 prefixes, then 2500 in one prefix (where the
        # 4096th lies: more than the 1024 keys the in-prefix rank takes), then 3000 over 6
        # prefixes (where the sampled threshold lies: about 6500 candidates), then the rest
        i = torch.arange(n_cap)
        grp = (i * 7919) % n_cap
        e = torch.where(grp < 3000, 4 + grp % 8, torch.where(grp < 5500, torch.full_like(i, 2),
                        torch.where(grp < 8500, -1 - grp % 3, torch.full_like(i, -8))))
        col = torch.where((grp >= 3000) & (grp < 5500), i % 32, i % 64)
        K = torch.zeros((B, Hkv, n_cap, d), dtype=torch.float64)
        K[0, 0, i, col] = torch.pow(2.0, e.double())
        K = K.to(torch.bfloat16)
        q = (1.0 + torch.arange(d, dtype=torch.float64) / 4096.0).float().expand(B, Hq, d).contiguous()
    else:
        i = torch.arange(n_cap)
        on = (i % 136) < 8
        big = on if pattern == "sampled_high" else ~on
        scale = torch.where(big, 8.0, 0.125).double() * torch.pow(2.0, (i % 3).double())   # exact products
        K = torch.zeros((B, Hkv, n_cap, d), dtype=torch.float64)
        K[0, 0, i, (5 * i) % d] = scale
        K = K.to(torch.bfloat16)
        q = torch.rand((B, Hq, d), generator=g_) + 0.5      # positive: the scale decides the order
    Kd, qd = K.cuda(), q.cuda()
    seq = torch.tensor([n_cap], dtype=torch.int32, device="cuda")
    shape = H.make_shape(qd, Kd, torch.zeros_like(Kd))
    z, idx, cnt = _exact_call(H, shape, qd, Kd, seq, m, B, Hq, n_cap)
    qn, Kn = q.double().numpy(), K.double().numpy()
    for h in range(Hq):
        assert int(cnt[0, h]) == m
        got = idx[0, h, :m]
        assert np.all(np.diff(got) > 0)
        if pattern == "random":
            sure, band = O.top_m_band(qn[0, h], Kn[0, 0], n_cap, m)
            assert set(sure) <= set(got) <= set(sure) | set(band), h
        else:
            assert np.array_equal(got, O.top_m_by_dot(qn[0, h], Kn[0, 0], n_cap, m)), h


def test_device_errors_are_flagged_not_faulted():
    H = GH.ha()
    w = W().make_gqa(16, B=3, Hq=4, Hkv=2, d=128, n_cap=2000, seq_lens=[2000, 1500, 2000], m=100,
                     n_sink=4, n_local=4, device="cuda")
    w.seq_lens = torch.tensor([2000, 2001, -5], dtype=torch.int32, device="cuda")  # 2 bad entries
    res = GH.run_decode(w)
    assert res["status"] == H.HA_ERR_DEVICE and res["flags"] & H.HA_DEVERR_SEQLEN
    assert torch.all(res["lse"][1:].isneginf()) and torch.all(res["out"][1:] == 0)
    assert torch.all(res["sel_cnt"][1:] == 0)
    hc = GH.HostCopy(w)
    GH.check_attention(res, hc, [(0, h) for h in range(4)], w.m)
    # the same on the decode step without selection outputs (scan + group kernel)
    grp = GH.run_decode(w, sel=False)
    assert grp["status"] == H.HA_ERR_DEVICE and grp["flags"] & H.HA_DEVERR_SEQLEN
    assert torch.all(grp["lse"][1:].isneginf()) and torch.all(grp["out"][1:] == 0)
    GH.check_attention(grp, hc, [(0, h) for h in range(4)], w.m)
    # a per-sequence budget above the bound is clamped and flagged
    w.seq_lens = torch.tensor([2000, 1500, 2000], dtype=torch.int32, device="cuda")
    w.m_per_seq = torch.tensor([100, 150, 50], dtype=torch.int32, device="cuda")
    res = GH.run_decode(w, m=100)
    assert res["status"] == H.HA_ERR_DEVICE and res["flags"] & H.HA_DEVERR_BUDGET
    assert int(res["sel_cnt"][1, 0]) == len(O.selected_set(int(w.q_sig[1, 0]),
                                                              w.k_sig[1, 0].cpu().numpy(), 1500, 100, 4, 4))
    grp = GH.run_decode(w, m=100, sel=False)
    assert grp["status"] == H.HA_ERR_DEVICE and grp["flags"] & H.HA_DEVERR_BUDGET
    w.m_per_seq = torch.tensor([100, 100, 50], dtype=torch.int32, device="cuda")  # as clamped
    GH.check_attention(grp, GH.HostCopy(w), [(b, h) for b in range(3) for h in range(4)], 100)
    # the next call on the same workspace reports clean
    w.m_per_seq = None
    res = GH.run_decode(w, ws=res["ws"])
    assert res["status"] == 0


# ---------------------------------------------------------------- the five workloads at full size

def test_workload1_tiny_full():
    w = W().make_workload(1, "cuda")
    res = GH.run_decode(w)
    assert res["status"] == 0
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), w.m)
    GH.check_attention(res, hc, all_heads(w), w.m)


def test_workload2_gqa_32k_full():
    w = W().make_workload(2, "cuda")
    res = GH.run_decode(w)
    assert res["status"] == 0
    hc = GH.HostCopy(w)
    GH.check_selection(res, hc, all_heads(w), w.m)
    GH.check_attention(res, hc, all_heads(w), w.m)
    GH.check_decode_step_path(w, res, hc, all_heads(w), w.m, ws=res["ws"])


def _sample_heads(w, k, seed):
    rng = np.random.default_rng(seed)
    pairs = all_heads(w)
    pick = rng.choice(len(pairs), size=min(k, len(pairs)), replace=False)
    return sorted(pairs[i] for i in pick)


def test_workload3_batch16_128k_sampled():
    w = W().make_workload(3, "cuda")
    res = GH.run_decode(w)
    assert res["status"] == 0
    hc = GH.HostCopy(w)
    heads = _sample_heads(w, 24, 3)
    GH.check_selection(res, hc, heads, w.m)
    GH.check_attention(res, hc, heads[:12], w.m)
    # properties that hold for every head: |I| within [min(n, m), m + S + Lw], ascending, windows in
    cnt = res["sel_cnt"].cpu().numpy()
    assert cnt.min() >= 4096 and cnt.max() <= 4096 + 128 + 256
    idx = res["sel_idx"].cpu().numpy()
    assert np.all(np.diff(idx[:, :, :4096], axis=-1) > 0)
    assert np.all(idx[:, :, :128] == np.arange(128))
    # the path the bench times, in its launch configuration (full grid, same workspace)
    GH.check_decode_step_path(w, res, hc, heads[:12], w.m, ws=res["ws"])
    del w, res


def test_workload4_shared_document_full():
    H = GH.ha()
    w = W().make_workload(4, "cuda")
    doc = GH.run_decode(w)
    assert doc["status"] == 0
    B, Hq, d = w.q.shape
    from types import SimpleNamespace
    loc_w = SimpleNamespace(q=w.q, q_sig=None, k_sig=None, K=w.K_loc, V=w.V_loc, B=B, Hq=Hq,
                            Hkv=8, m=512, n_sink=0, n_local=0, m_per_seq=None,
                            seq_lens=torch.full((B,), 512, dtype=torch.int32, device="cuda"))
    loc = GH.run_decode(loc_w, dense=True, m_per_seq=None)
    assert loc["status"] == 0
    out = torch.empty_like(doc["out"])
    lse = torch.empty_like(doc["lse"])
    H.hash_attn_merge(doc["out"], doc["lse"], loc["out"], loc["lse"], out, lse, B * Hq, d)
    torch.cuda.synchronize()
    hc = GH.HostCopy(w)
    heads = _sample_heads(w, 16, 4)
    GH.check_selection(doc, hc, heads, w.m)
    GH.check_decode_step_path(w, doc, hc, heads[:8], w.m, ws=doc["ws"])
    q = w.q.float().cpu().numpy()
    for b, h in heads[:8]:
        _, _, od, ld = hc.head(b, h, w.m)
        Kl = w.K_loc[b, h // 4].float().cpu().numpy()
        Vl = w.V_loc[b, h // 4].float().cpu().numpy()
        ol, ll = O.attend(q[b, h], Kl, Vl, np.arange(512))
        ro, rl = O.merge(od, ld, ol, ll)
        GH.assert_out_close(out[b, h].cpu().numpy(), ro, f"merged ({b},{h})")
        GH.assert_lse_close(float(lse[b, h]), rl, f"merged ({b},{h})")


def test_workload5_ragged_full_sparse_and_dense():
    w = W().make_workload(5, "cuda")
    res = GH.run_decode(w)
    assert res["status"] == 0
    hc = GH.HostCopy(w)
    heads = _sample_heads(w, 24, 5)
    GH.check_selection(res, hc, heads, w.m)
    GH.check_attention(res, hc, heads[:12], w.m)
    GH.check_decode_step_path(w, res, hc, heads[:12], w.m, ws=res["ws"])
    dense = GH.run_decode(w, m=w.n_cap, m_per_seq=None, dense=True, sel=False)
    assert dense["status"] == 0
    GH.check_attention(dense, hc, heads[:6], w.n_cap, dense=True)
