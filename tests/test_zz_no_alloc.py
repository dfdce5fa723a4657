"""The allocation-free GATHER-ATT entry point against the workspace one and the oracle.

hash_attn_gather_att_noalloc serves callers that may not allocate device
memory (a plugin whose host application owns every device allocation through
its own pool, or a latency-critical path where cudaMalloc's implicit
synchronisation would stall other work): its scratch is a fixed array inside
the library. Two calls in a row must each match hash_attn_gather_att and the
CPU oracle within the parity tolerances, and report a clean error word. The
first call of this file runs on a side stream (non-blocking with respect to the
legacy default stream), so the per-device set-up must not rely on the default
stream. This file is collected last so that a failure here leaves every other
test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import gpu_helpers as GH
from oracle import hashattn_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def H():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from long_context_sparse_score_gb300 import _build
    _build.build()
    from long_context_sparse_score_gb300 import hashattn
    hashattn.lib()
    return hashattn


def _lists(B, Hq, lens, cap, seed):
    rng = np.random.default_rng(seed)
    idx = np.full((B, Hq, cap), -1, dtype=np.int32)
    cnt = np.zeros((B, Hq), dtype=np.int32)
    for b in range(B):
        for h in range(Hq):
            k = int(rng.integers(1, cap + 1))
            idx[b, h, :k] = rng.choice(lens[b], size=k, replace=False)
            cnt[b, h] = k
    return idx, cnt


def test_noalloc_matches_workspace_entry_point_and_oracle_twice(H):
    from long_context_sparse_score_gb300 import workloads as W
    lens = [6000, 4500, 6000]
    B, Hq, Hkv, d = 3, 8, 2, 128
    G = Hq // Hkv
    w = W.make_gqa(21, B=B, Hq=Hq, Hkv=Hkv, d=d, n_cap=6000, seq_lens=lens, m=0, n_sink=0, n_local=0,
                   device="cuda")
    cap = 1500
    shape = H.make_shape(w.q, w.K, w.V)
    idx_h, cnt_h = _lists(B, Hq, lens, cap, 5)
    idx, cnt = torch.from_numpy(idx_h).cuda(), torch.from_numpy(cnt_h).cuda()
    # the first calls run on a side stream that does not synchronise with the legacy default stream
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    flags = torch.full((1,), 0xFF, dtype=torch.int32, device="cuda")
    outs = []
    with torch.cuda.stream(side):
        for call in range(2):
            out = torch.full((B, Hq, d), float("nan"), device="cuda")
            lse = torch.full((B, Hq), float("nan"), device="cuda")
            H.hash_attn_gather_att_noalloc(shape, w.q, w.K, w.V, w.seq_lens, idx, cap, cnt, out, lse,
                                           dev_flags=flags, stream=side)
            outs.append((out, lse, flags.clone()))
    side.synchronize()
    ws = GH.workspace(shape, cap, 0, 0)
    ref_out = torch.empty((B, Hq, d), device="cuda")
    ref_lse = torch.empty((B, Hq), device="cuda")
    H.hash_attn_gather_att(shape, w.q, w.K, w.V, w.seq_lens, idx, cap, cnt, ref_out, ref_lse, workspace=ws)
    torch.cuda.synchronize()
    ref_o = ref_out.cpu().numpy()
    ref_l = ref_lse.cpu().numpy()
    q = w.q.float().cpu().numpy()
    Kh = w.K.float().cpu().numpy()
    Vh = w.V.float().cpu().numpy()
    for call, (out, lse, fl) in enumerate(outs):
        assert int(fl.item()) == 0, f"call {call}: error word {int(fl.item()):#x}"
        got_o = out.cpu().numpy()
        got_l = lse.cpu().numpy()
        for b in range(B):
            for h in range(Hq):
                # against the workspace entry point
                GH.assert_out_close(got_o[b, h], ref_o[b, h], f"call {call} ({b},{h}) vs workspace path")
                GH.assert_lse_close(float(got_l[b, h]), float(ref_l[b, h]), f"call {call} ({b},{h})")
                # against the oracle on the same lists
                rows = idx_h[b, h, :cnt_h[b, h]]
                o_ref, l_ref = O.attend(q[b, h], Kh[b, h // G], Vh[b, h // G], rows)
                GH.assert_out_close(got_o[b, h], o_ref, f"call {call} ({b},{h}) vs oracle")
                GH.assert_lse_close(float(got_l[b, h]), float(l_ref), f"call {call} ({b},{h}) vs oracle")


def test_noalloc_flags_bad_index_and_rejects_oversized_shapes(H):
    from long_context_sparse_score_gb300 import workloads as W
    w = W.make_gqa(22, B=1, Hq=4, Hkv=1, d=128, n_cap=2000, seq_lens=[2000], m=0, n_sink=0, n_local=0,
                   device="cuda")
    shape = H.make_shape(w.q, w.K, w.V)
    idx = torch.tensor([[[5, 2000, 7, 9]] * 4], dtype=torch.int32, device="cuda")  # 2000 is out of range
    cnt = torch.full((1, 4), 4, dtype=torch.int32, device="cuda")
    out = torch.empty((1, 4, 128), device="cuda")
    lse = torch.empty((1, 4), device="cuda")
    flags = torch.zeros((1,), dtype=torch.int32, device="cuda")
    H.hash_attn_gather_att_noalloc(shape, w.q, w.K, w.V, w.seq_lens, idx, 4, cnt, out, lse, dev_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) & H.HA_DEVERR_INDEX
    # the next call starts with a clean error word
    idx[0, :, 1] = 11
    H.hash_attn_gather_att_noalloc(shape, w.q, w.K, w.V, w.seq_lens, idx, 4, cnt, out, lse, dev_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    # A shape whose scratch exceeds the built-in array is refused before any launch.
    # 2^17 query heads need 2^17 * (d + 2) * 4 = 68 MB of partials even with one
    # split per head, four times the 16 MiB array, so no split policy can make it fit.
    # Its pointers are those of the small tensors above: it must never launch.
    big = H.HAShape()
    ctypes.pointer(big)[0] = shape
    big.batch = 1 << 15
    big.q_sb = 0
    big.k_sb = big.v_sb = 0
    assert big.batch * big.h_q * (big.d + 2) * 4 > 4 * H.HA_NOALLOC_SCRATCH_BYTES
    st = H.lib().hash_attn_gather_att_noalloc(ctypes.byref(big), w.q.data_ptr(), w.K.data_ptr(),
                                              w.V.data_ptr(), w.seq_lens.data_ptr(), idx.data_ptr(), 4,
                                              cnt.data_ptr(), out.data_ptr(), lse.data_ptr(), None, None)
    assert st == H.HA_ERR_WORKSPACE and "scratch" in H.last_error()
