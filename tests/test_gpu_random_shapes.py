"""Seeded random decode shapes against the oracle.

Each case draws a shape (batch, KV heads, query heads per KV head, head dim,
cache capacity, ragged lengths) and a selection (budget, sink and local
windows, optionally per-sequence or per-head budgets and exclusive windows)
from its seed, then runs the decode step without selection outputs (the
selection scan and the GQA-group kernel for up to four query heads per KV head,
the two-kernel selection above; or the dense path) and the call that also
returns the selection (the per-head path), and compares both with the
oracle: selected sets bit for bit, outputs and log-normalisers within the
tolerances of gpu_helpers, on every head of the first two sequences.
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


def _draw(seed):
    rng = np.random.default_rng(7000 + seed)
    B = int(rng.integers(1, 5))
    Hkv = int(rng.integers(1, 4))
    G = int(rng.integers(1, 9))  # above 4: the two-kernel selection and per-head GATHER-ATT
    d = int(rng.choice([64, 128]))
    # code rows start on 16-byte boundaries (a documented requirement): capacities in
    # whole 4-token groups; the lengths stay ragged
    n_cap = 4 * int(rng.choice([int(rng.integers(1, 1000)), int(rng.integers(1000, 17500))]))
    lens = [int(x) for x in rng.integers(0, n_cap + 1, size=B)]
    lens[0] = n_cap
    dense = rng.random() < 0.15
    m = n_cap if dense else int(rng.integers(0, max(1, n_cap // 4) + 1))
    n_sink = int(rng.integers(0, 200))
    n_local = int(rng.integers(0, 300))
    mode = "plain" if dense else str(rng.choice(["plain", "per_seq", "per_head", "exclusive"]))
    return dict(B=B, Hkv=Hkv, G=G, d=d, n_cap=n_cap, lens=lens, m=m, n_sink=n_sink, n_local=n_local,
                dense=dense, mode=mode, rng=rng)


@pytest.mark.parametrize("seed", range(32))
def test_random_shape_against_oracle(seed):
    c = _draw(seed)
    from long_context_sparse_score_gb300 import workloads as W
    B, Hkv, G, n_cap, m = c["B"], c["Hkv"], c["G"], c["n_cap"], c["m"]
    Hq = Hkv * G
    mps = None
    if c["mode"] == "per_seq":
        mps = [int(x) for x in c["rng"].integers(0, m + 1, size=B)]
    w = W.make_gqa(300 + seed, B=B, Hq=Hq, Hkv=Hkv, d=c["d"], n_cap=n_cap, seq_lens=c["lens"], m=m,
                   n_sink=c["n_sink"], n_local=c["n_local"], device="cuda", m_per_seq=mps,
                   name=f"random{seed}")
    mph = None
    if c["mode"] == "per_head":
        mph = torch.as_tensor(c["rng"].integers(0, m + 1, size=(B, Hq)), dtype=torch.int32, device="cuda")
    excl = c["mode"] == "exclusive"
    heads = [(b, h) for b in range(min(B, 2)) for h in range(Hq)]
    hc = GH.HostCopy(w, exclusive=excl, m_per_head=mph)
    if c["dense"]:
        res = GH.run_decode(w, m=m, m_per_seq=None, dense=True, sel=False)
        assert res["status"] == 0, hex(res["flags"])
        GH.check_attention(res, hc, heads, m, dense=True)
        return
    step = GH.run_decode(w, sel=False, exclusive=excl, m_per_head=mph)
    assert step["status"] == 0, hex(step["flags"])
    GH.check_attention(step, hc, heads, m)
    full = GH.run_decode(w, sel=True, exclusive=excl, m_per_head=mph)
    assert full["status"] == 0, hex(full["flags"])
    GH.check_selection(full, hc, heads, m)
    GH.check_attention(full, hc, heads, m)
