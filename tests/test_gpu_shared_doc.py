"""One cached document shared by a batch of queries (K, V and key codes with
batch stride 0), against the oracle.

The group kernel serves each (query, KV head, range) from the one document;
its CTAs for the batch's queries run together so that the document's rows come
from L2. The cases vary what that touches: several ranges, ragged lengths per
query (ranges past a query's end), windows, exclusive windows, per-query and
per-head budgets with ties at the threshold, G = 1 to 4, d = 64 and 128, a
capacity that is not a multiple of 128, and batches of 10 to 40 queries. Every
case checks the path the call takes, then compares the output and
log-normaliser of every head with the oracle; the selected sets are checked
through the call that returns them (another path), whose outputs the decode
step must also match.
"""
import numpy as np
import pytest
import torch

import gpu_helpers as GH

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from long_context_sparse_score_gb300 import _build
    _build.build()
    from long_context_sparse_score_gb300 import hashattn
    hashattn.lib()


def _workload(seed, B, Hq, Hkv, d, n_cap, lens, m, n_sink, n_local, codes="random", m_per_seq=None):
    from long_context_sparse_score_gb300 import workloads as W
    w = W.make_gqa(900 + seed, B=B, Hq=Hq, Hkv=Hkv, d=d, n_cap=n_cap, seq_lens=lens, m=m, n_sink=n_sink,
                   n_local=n_local, device="cuda", shared=True, m_per_seq=m_per_seq, name=f"doc{seed}")
    if codes == "pool":
        # few distinct key and query codes: every threshold bin holds many ties, and
        # the heads' thresholds differ
        gen = torch.Generator(device="cuda").manual_seed(seed)
        c0 = 0x0F0F0F0F
        kpool = torch.tensor([c0, c0 ^ 1, c0 ^ 3, c0 ^ 0x70000000, c0 ^ 0x0000FFFF, c0 ^ 0x00F00000],
                             dtype=torch.int32, device="cuda")
        qpool = torch.tensor([c0, c0 ^ 2, c0 ^ 0x100, c0 ^ 0x30000000], dtype=torch.int32, device="cuda")
        w.k_sig = kpool[torch.randint(0, 6, w.k_sig.shape, generator=gen, device="cuda")].contiguous()
        w.q_sig = qpool[torch.randint(0, 4, w.q_sig.shape, generator=gen, device="cuda")].contiguous()
    return w


RAGGED = [17000, 9000, 8192, 8191, 100, 0, 16384, 16385, 5000, 17000, 12000, 1]

# name, B, Hq, Hkv, d, n_cap, lengths, m, n_sink, n_local, codes, mode
CASES = [
    ("g4_three_ranges", 16, 8, 2, 128, 20000, 20000, 1024, 64, 128, "random", "plain"),
    ("g4_ragged_lengths", 12, 8, 2, 128, 17000, RAGGED, 800, 32, 64, "random", "plain"),
    ("g4_ties", 16, 8, 2, 128, 24000, 24000, 1500, 64, 128, "pool", "plain"),
    ("g4_ties_exclusive", 16, 8, 2, 128, 24000, [24000] * 8 + [20000] * 8, 1500, 700, 900, "pool", "exclusive"),
    ("g4_per_head", 16, 8, 2, 128, 18000, 18000, 1200, 16, 300, "pool", "per_head"),
    ("g4_per_seq", 16, 8, 2, 128, 18000, 18000, 1200, 16, 300, "random", "per_seq"),
    ("g2_d64", 16, 4, 2, 64, 12000, 12000, 900, 32, 32, "random", "plain"),
    ("g3", 10, 6, 2, 128, 9000, 9000, 1100, 16, 64, "pool", "plain"),
    ("g1_d64", 32, 2, 2, 64, 9000, 9000, 400, 8, 16, "random", "plain"),
    ("batch40_one_kv_head", 40, 4, 1, 128, 9000, 9000, 500, 32, 32, "random", "plain"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_shared_document_against_oracle(case):
    name, B, Hq, Hkv, d, n_cap, lens, m, n_sink, n_local, codes, mode = case
    H = GH.ha()
    rng = np.random.default_rng(len(name))
    mps = [int(x) for x in rng.integers(0, m + 1, size=B)] if mode == "per_seq" else None
    w = _workload(CASES.index(case), B, Hq, Hkv, d, n_cap, lens, m, n_sink, n_local, codes, mps)
    mph = None
    if mode == "per_head":
        mph = torch.as_tensor(rng.integers(0, m + 1, size=(B, Hq)), dtype=torch.int32, device="cuda")
    excl = mode == "exclusive"
    shape = H.make_shape(w.q, w.K, w.V, w.k_sig, batch=B)
    opts = H.select_opts(mph, excl, 1) if (excl or mph is not None) else None
    assert H.hash_attn_decode_path(shape, m, w.m_per_seq, opts) == "group"
    assert H.hash_attn_decode_path(shape, m, w.m_per_seq, opts, with_selection=True) == "fused_lists"

    step = GH.run_decode(w, sel=False, exclusive=excl, m_per_head=mph)
    assert step["status"] == 0, hex(step["flags"])
    hc = GH.HostCopy(w, exclusive=excl, m_per_head=mph)
    heads = [(b, h) for b in range(B) for h in range(Hq)]
    GH.check_attention(step, hc, heads, m)

    full = GH.run_decode(w, sel=True, exclusive=excl, m_per_head=mph)
    assert full["status"] == 0, hex(full["flags"])
    GH.check_selection(full, hc, heads[::3], m)
    GH.assert_out_close(step["out"].cpu().numpy(), full["out"].cpu().numpy(), "decode step vs the lists path")


def test_shared_document_back_to_back():
    """Two batches over two documents of one shape, decoded back to back on one
    workspace with nothing between the calls: each output equals that of its call
    alone, bit for bit."""
    H = GH.ha()
    ws_a = [_workload(40 + i, 16, 8, 2, 128, 20000, 20000, 1024, 64, 128) for i in range(2)]
    shape = H.make_shape(ws_a[0].q, ws_a[0].K, ws_a[0].V, ws_a[0].k_sig, batch=16)
    ws = GH.workspace(shape, 1024, 64, 128)
    outs = [(torch.empty((16, 8, 128), device="cuda"), torch.empty((16, 8), device="cuda")) for _ in range(4)]

    def call(w, o):
        H.hash_attn_decode(shape, w.q, w.q_sig, w.k_sig, w.K, w.V, w.seq_lens, None, w.m, w.n_sink, w.n_local,
                           o[0], o[1], workspace=ws)

    for i in range(2):  # alone
        call(ws_a[i], outs[i])
        torch.cuda.synchronize()
    for _ in range(3):  # back to back, repeated
        call(ws_a[0], outs[2])
        call(ws_a[1], outs[3])
    torch.cuda.synchronize()
    st, flags = H.hash_attn_device_status(ws)
    assert st == 0, hex(flags)
    for i in range(2):
        assert torch.equal(outs[i][0], outs[2 + i][0]) and torch.equal(outs[i][1], outs[2 + i][1])
    hc = GH.HostCopy(ws_a[1])
    GH.check_attention(dict(out=outs[3][0], lse=outs[3][1]), hc, [(b, h) for b in (0, 15) for h in range(8)], 1024)
