"""Helpers of the GPU parity tests: run the C ABI on a workload, run the oracle on
the same inputs (copied to the host), compare."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import hashattn_oracle as O

OUT_RTOL = OUT_ATOL = 2e-3   # |gpu - ref| <= 2e-3 * (1 + |ref|), fp32 output
LSE_RTOL = LSE_ATOL = 1e-4   # |gpu - ref| <= 1e-4 * (1 + |ref|)


def ha():
    from long_context_sparse_score_gb300 import hashattn
    return hashattn


def workspace(shape, m, n_sink, n_local, device="cuda"):
    H = ha()
    nbytes = H.hash_attn_workspace_size(shape, m, n_sink, n_local)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    H.hash_attn_workspace_init(ws)
    return ws


def run_decode(w, *, m=None, m_per_seq="workload", sel=True, K=None, V=None, ws=None, dense=False,
               exclusive=False, m_per_head=None, code_words=1):
    """Decode a workload through the C ABI; returns a dict of outputs and the device status.
    ``exclusive`` / ``m_per_head`` / ``code_words`` go through hash_attn_decode_ex."""
    H = ha()
    K = w.K if K is None else K
    V = w.V if V is None else V
    m = w.m if m is None else m
    mps = w.m_per_seq if m_per_seq == "workload" else m_per_seq
    k_sig = None if dense else w.k_sig
    q_sig = None if dense else w.q_sig
    shape = H.make_shape(w.q, K, V, w.k_sig, batch=w.B)
    opts = None
    if exclusive or m_per_head is not None or code_words > 1:
        opts = H.select_opts(m_per_head, exclusive, code_words)
    if ws is None:
        if opts is None:
            ws = workspace(shape, m, w.n_sink, w.n_local)
        else:
            ws = torch.empty(H.hash_attn_workspace_size_ex(shape, m, w.n_sink, w.n_local, opts),
                             dtype=torch.uint8, device=w.q.device)
            H.hash_attn_workspace_init(ws)
    B, Hq, d = w.q.shape
    out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=w.q.device)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=w.q.device)
    cap = H.hash_attn_select_capacity(K.shape[2], m, w.n_sink, w.n_local)
    sel_idx = sel_cnt = None
    if sel and not (m >= K.shape[2] and mps is None):
        sel_idx = torch.full((B, Hq, max(cap, 1)), -7, dtype=torch.int32, device=w.q.device)
        sel_cnt = torch.full((B, Hq), -7, dtype=torch.int32, device=w.q.device)
    if opts is not None:
        H.hash_attn_decode_ex(shape, w.q, q_sig, k_sig, K, V, w.seq_lens, mps, m, w.n_sink, w.n_local, opts,
                              out, lse, sel_idx, sel_cnt, workspace=ws)
    else:
        H.hash_attn_decode(shape, w.q, q_sig, k_sig, K, V, w.seq_lens, mps, m, w.n_sink, w.n_local,
                           out, lse, sel_idx, sel_cnt, workspace=ws)
    st, flags = H.hash_attn_device_status(ws)
    return dict(out=out, lse=lse, sel_idx=sel_idx, sel_cnt=sel_cnt, status=st, flags=flags, ws=ws,
                cap=cap)


class HostCopy:
    """Per-(batch, KV head) host copies of a workload, made on demand."""

    def __init__(self, w, K=None, V=None, exclusive=False, m_per_head=None):
        self.w = w
        self.exclusive = exclusive
        self.mph = None if m_per_head is None else m_per_head.cpu().numpy()
        self.K = w.K if K is None else K
        self.V = w.V if V is None else V
        self.q = w.q.float().cpu().numpy()
        self.q_sig = w.q_sig.cpu().numpy().astype(np.int64)
        self.lens = w.seq_lens.cpu().numpy()
        self.mps = None if w.m_per_seq is None else w.m_per_seq.cpu().numpy()
        self._kv = {}
        self._codes = {}

    def kv(self, b, g):
        bk = 0 if self.K.shape[0] == 1 else b
        key = (bk, g)
        if key not in self._kv:
            if len(self._kv) > 8:
                self._kv.clear()
            self._kv[key] = (self.K[bk, g].float().cpu().numpy(), self.V[bk, g].float().cpu().numpy())
        return self._kv[key]

    def codes(self, b, g):
        bk = 0 if self.w.k_sig.shape[0] == 1 else b
        key = (bk, g)
        if key not in self._codes:
            self._codes[key] = self.w.k_sig[bk, g].cpu().numpy().astype(np.int64)
        return self._codes[key]

    def qcode(self, b, h):
        """The query code: an int (32-bit codes) or its words (wider codes)."""
        return int(self.q_sig[b, h]) if self.q_sig.ndim == 2 else self.q_sig[b, h]

    def budget(self, b, m, h=None):
        if self.mph is not None and h is not None:
            return int(self.mph[b, h])
        return int(self.mps[b]) if self.mps is not None else m

    def select(self, b, h, m):
        G = self.w.Hq // self.w.Hkv
        n = int(self.lens[b])
        return O.selected_set(self.qcode(b, h), self.codes(b, h // G), n, self.budget(b, m, h),
                              self.w.n_sink, self.w.n_local, exclusive=self.exclusive)

    def head(self, b, h, m, dense=False):
        G = self.w.Hq // self.w.Hkv
        g = h // G
        Kh, Vh = self.kv(b, g)
        n = int(self.lens[b])
        codes = None if dense else self.codes(b, g)
        return O.decode_head(self.q[b, h], None if dense else self.qcode(b, h), codes, Kh, Vh, n,
                             self.budget(b, m, h), self.w.n_sink, self.w.n_local, dense=dense,
                             exclusive=self.exclusive)


def assert_out_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3g}, worst ratio {(err / bound).max():.3g}"


def assert_lse_close(got, ref, what=""):
    if ref == -math.inf:
        assert got == -math.inf, f"{what}: lse {got} != -inf"
        return
    assert abs(got - ref) <= LSE_ATOL + LSE_RTOL * abs(ref), f"{what}: lse {got} vs {ref}"


def check_selection(res, hc, heads, m):
    sel_idx = res["sel_idx"].cpu().numpy()
    sel_cnt = res["sel_cnt"].cpu().numpy()
    for b, h in heads:
        want = hc.select(b, h, m)
        c = int(sel_cnt[b, h])
        assert c == len(want), f"(b={b}, h={h}) count {c} vs {len(want)}"
        assert np.array_equal(sel_idx[b, h, :c], want), f"(b={b}, h={h}) selected set differs"
        assert np.all(sel_idx[b, h, c:res["cap"]] == -1), f"(b={b}, h={h}) padding"


def check_attention(res, hc, heads, m, dense=False):
    out = res["out"].cpu().numpy()
    lse = res["lse"].cpu().numpy()
    for b, h in heads:
        _, _, ref_out, ref_lse = hc.head(b, h, m, dense=dense)
        assert_out_close(out[b, h], ref_out, f"out (b={b}, h={h})")
        assert_lse_close(float(lse[b, h]), ref_lse, f"lse (b={b}, h={h})")


def check_decode_step_path(w, res_sel, hc, heads, m, ws=None, K=None, V=None):
    """The decode call without selection outputs (the path the bench times: the
    selection scan, then the GQA-group kernel when the shape allows it) on the same
    workload: against the oracle on ``heads`` and against ``res_sel`` (the call that
    also returned the selection) on every head."""
    grp = run_decode(w, m=m, sel=False, ws=ws, K=K, V=V)
    assert grp["status"] == 0, hex(grp["flags"])
    check_attention(grp, hc, heads, m)
    go, ro = grp["out"].cpu().numpy(), res_sel["out"].cpu().numpy()
    assert np.all(np.isfinite(go)), "non-finite output"
    assert_out_close(go, ro, "decode step vs the call with selection outputs")
    gl, rl = grp["lse"].cpu().numpy(), res_sel["lse"].cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.all(np.abs(gl[fin] - rl[fin]) <= 2 * LSE_ATOL * (1 + np.abs(rl[fin])))
    return grp
