"""The decode step without selection outputs: k_sel_scan, then one kernel per
GQA group (k_group_att) that rebuilds every head's mask from the codes and
attends over the union of the group's rows with tensor-core products.

hash_attn_decode takes this path when the caller asks for no selected indices
(sel_idx = NULL), the query and K/V are bf16, d is 64 or 128 and the fused
selection applies (32-bit codes, at most four query heads per KV head). Every
case compares the outputs and log-normalisers of all (or 16 sampled) heads with
the oracle, and with the same call that also returns the selection (which takes
the emit kernel and the per-head GATHER-ATT)."""
import numpy as np
import pytest
import torch

import gpu_helpers as GH
from test_gpu_select_paths import FUSED, FUSED_VARIANTS, _codes, _sample

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


def _both(w, heads, *, exclusive=False, m_per_head=None):
    """The group path against the oracle and against the path with selection outputs."""
    grp = GH.run_decode(w, sel=False, exclusive=exclusive, m_per_head=m_per_head)
    assert grp["status"] == 0, hex(grp["flags"])
    hc = GH.HostCopy(w, exclusive=exclusive, m_per_head=m_per_head)
    GH.check_attention(grp, hc, heads, w.m)
    ref = GH.run_decode(w, sel=True, exclusive=exclusive, m_per_head=m_per_head)
    assert ref["status"] == 0, hex(ref["flags"])
    go, ro = grp["out"].cpu().numpy(), ref["out"].cpu().numpy()
    gl, rl = grp["lse"].cpu().numpy(), ref["lse"].cpu().numpy()
    assert np.all(np.isfinite(go)), "non-finite output"
    GH.assert_out_close(go, ro, "group vs per-head path")
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.all(np.abs(gl[fin] - rl[fin]) <= 2 * GH.LSE_ATOL * (1 + np.abs(rl[fin])))
    return grp


@pytest.mark.parametrize("case", FUSED, ids=[c[0] for c in FUSED])
def test_group_path_fused_cases(case):
    """Ranges, windows across ranges, tie-heavy codes, G = 1, 2, 3, 4, empty and
    one-token sequences, all distances 32, windows only."""
    name, B, Hq, Hkv, n_cap, lens, m, S, Lw, codes = case
    w = W().make_gqa(31, B=B, Hq=Hq, Hkv=Hkv, d=128, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S, n_local=Lw,
                     device="cuda", name=name)
    _codes(w, codes, 41)
    heads = [(b, h) for b in range(B) for h in range(Hq)]
    if len(heads) > 16:
        heads = _sample(B, Hq, 16, 6)
    _both(w, heads)


@pytest.mark.parametrize("case", FUSED_VARIANTS, ids=[c[0] for c in FUSED_VARIANTS])
def test_group_path_variants(case):
    """Exclusive windows and per-head budgets (0 and m included)."""
    name, n_cap, lens, m, S, Lw, codes, exclusive, per_head = case
    w = W().make_gqa(32, B=2, Hq=4, Hkv=1, d=128, n_cap=n_cap, seq_lens=lens, m=m, n_sink=S, n_local=Lw,
                     device="cuda", name=name)
    _codes(w, codes, 42)
    mph = None
    if per_head:
        gen = torch.Generator(device="cuda").manual_seed(9)
        mph = torch.randint(0, m + 1, (2, 4), generator=gen, device="cuda", dtype=torch.int32)
        mph[0, 0], mph[1, 3] = 0, m
    _both(w, [(b, h) for b in range(2) for h in range(4)], exclusive=exclusive, m_per_head=mph)


@pytest.mark.parametrize("d", [64, 128])
def test_group_path_head_dims_and_ragged_budgets(d):
    """d = 64 and 128; ragged lengths with per-sequence budgets (the ragged recipe)."""
    lens = [9000, 4096, 20000, 17, 16385, 8192]
    lt = torch.tensor(lens, dtype=torch.int32)
    mb = W().ragged_budget(lt)
    w = W().make_gqa(33, B=6, Hq=8, Hkv=2, d=d, n_cap=20000, seq_lens=lens, m=int(mb.max()), n_sink=64,
                     n_local=128, device="cuda", m_per_seq=mb, name=f"ragged-d{d}")
    _both(w, [(b, h) for b in range(6) for h in range(8)])


def test_group_path_shared_cache():
    """One cached document for the whole batch (K/V and codes with batch stride 0)."""
    w = W().make_gqa(34, B=6, Hq=8, Hkv=2, d=128, n_cap=30000, seq_lens=30000, m=1000, n_sink=128, n_local=0,
                     device="cuda", shared=True, name="shared")
    _both(w, [(b, h) for b in range(6) for h in range(8)])


def test_group_path_batch16_slice():
    """Two sequences of the 16 x 131,072-token workload (16 ranges per sequence)."""
    w = W().make_gqa(3, B=2, Hq=32, Hkv=8, d=128, n_cap=131072, seq_lens=131072, m=4096, n_sink=128,
                     n_local=256, device="cuda", name="batch2-128k")
    _both(w, _sample(2, 32, 16, 7))


# ---------------------------------------------------------------- calls back to back

BACK_TO_BACK = [
    # name, B, n (32 / 8 heads, d = 128): one CTA per SM or less, and several waves
    ("one_sequence_32k", 1, 32768),
    ("four_sequences_40000", 4, 40000),
    ("eight_sequences_128k", 8, 131072),
]


@pytest.mark.parametrize("case", BACK_TO_BACK, ids=[c[0] for c in BACK_TO_BACK])
def test_back_to_back_calls_with_different_inputs(case):
    """Calls on one stream and one workspace issued with nothing between them (no
    host synchronisation, no other kernel), each with inputs and a budget of its
    own, as successive layers of a model make them; the decode step (selection
    scan + group kernel), the path that also returns the selection and the dense
    path interleaved. Each kernel lets the next one start early, so a call's
    kernels run beside the previous call's: every output, log-normaliser and
    selection must equal, bit for bit, those of the same call made alone, and
    the calls alone meet the oracle on sampled heads."""
    name, B, n = case
    H = GH.ha()
    wl = [W().make_gqa(50 + k, B=B, Hq=32, Hkv=8, d=128, n_cap=n, seq_lens=n, m=(1024, 2048, 700)[k],
                       n_sink=128, n_local=(128, 256, 0)[k], device="cuda", name=f"{name}_{k}")
          for k in range(3)]
    shape = H.make_shape(wl[0].q, wl[0].K, wl[0].V, wl[0].k_sig, batch=B)
    # one workspace for every call, sized for the largest use (the dense path)
    ws = GH.workspace(shape, n, 0, 0)
    caps = [H.hash_attn_select_capacity(n, w.m, w.n_sink, w.n_local) for w in wl]

    def buffers(k):
        return {"out": torch.full((B, 32, 128), float("nan"), device="cuda"),
                "lse": torch.full((B, 32), float("nan"), device="cuda"),
                "idx": torch.full((B, 32, caps[k]), -7, dtype=torch.int32, device="cuda"),
                "cnt": torch.full((B, 32), -7, dtype=torch.int32, device="cuda")}

    def call(k, mode, bf):
        w = wl[k]
        if mode == "dense":
            H.hash_attn_decode(shape, w.q, None, None, w.K, w.V, w.seq_lens, None, n, 0, 0, bf["out"], bf["lse"],
                               workspace=ws)
        elif mode == "sel":
            H.hash_attn_decode(shape, w.q, w.q_sig, w.k_sig, w.K, w.V, w.seq_lens, None, w.m, w.n_sink,
                               w.n_local, bf["out"], bf["lse"], bf["idx"], bf["cnt"], workspace=ws)
        else:
            H.hash_attn_decode(shape, w.q, w.q_sig, w.k_sig, w.K, w.V, w.seq_lens, None, w.m, w.n_sink,
                               w.n_local, bf["out"], bf["lse"], workspace=ws)

    kinds = [(k, "group") for k in range(3)] + [(k, "sel") for k in range(3)] + [(1, "dense")]
    alone = {}
    for k, mode in kinds:
        bf = buffers(k)
        call(k, mode, bf)
        torch.cuda.synchronize()
        alone[(k, mode)] = bf
    seq = [(0, "group"), (1, "group"), (2, "group"), (0, "group"), (1, "dense"), (2, "group"), (1, "group"),
           (0, "sel"), (2, "group"), (1, "sel"), (0, "group"), (2, "sel"), (1, "group"), (0, "group")]
    bufs = [buffers(k) for k, _ in seq]
    torch.cuda.synchronize()
    for (k, mode), bf in zip(seq, bufs):  # nothing else enters the stream between the calls
        call(k, mode, bf)
    torch.cuda.synchronize()
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, hex(flags)
    for i, ((k, mode), bf) in enumerate(zip(seq, bufs)):
        ref = alone[(k, mode)]
        what = f"call {i} (workload {k}, {mode})"
        assert torch.equal(bf["out"], ref["out"]), f"{what}: output differs from the call alone"
        assert torch.equal(bf["lse"], ref["lse"]), f"{what}: lse differs from the call alone"
        if mode == "sel":
            assert torch.equal(bf["idx"], ref["idx"]) and torch.equal(bf["cnt"], ref["cnt"]), what
    heads = [(b, h) for b in range(min(B, 2)) for h in (0, 5, 18, 31)]
    for k in range(3):
        w = wl[k]
        hc = GH.HostCopy(w)
        for mode in ("group", "sel"):
            GH.check_attention(alone[(k, mode)], hc, heads, w.m)
        sel = {"sel_idx": alone[(k, "sel")]["idx"], "sel_cnt": alone[(k, "sel")]["cnt"], "cap": caps[k]}
        GH.check_selection(sel, hc, heads, w.m)
    GH.check_attention(alone[(1, "dense")], GH.HostCopy(wl[1]), heads, n, dense=True)
