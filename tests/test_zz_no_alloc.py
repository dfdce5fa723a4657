"""The allocation-free GATHER-ATT entry point against the workspace one.

hash_attn_gather_att_noalloc serves callers that may not allocate device
memory (a host application that owns every device allocation through its own
pool, or a path that cannot afford cudaMalloc's implicit synchronisation): its
scratch is a fixed array inside the library. Two calls in a row must each match
hash_attn_gather_att within the parity tolerances, and report a clean error
word. This file is collected last so that a failure here leaves every other
test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import gpu_helpers as GH

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
    return torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()


def test_noalloc_matches_workspace_entry_point_twice(H):
    from long_context_sparse_score_gb300 import workloads as W
    lens = [6000, 4500, 6000]
    w = W.make_gqa(21, B=3, Hq=8, Hkv=2, d=128, n_cap=6000, seq_lens=lens, m=0, n_sink=0, n_local=0,
                   device="cuda")
    cap = 1500
    shape = H.make_shape(w.q, w.K, w.V)
    ws = GH.workspace(shape, cap, 0, 0)
    idx, cnt = _lists(3, 8, lens, cap, 5)
    ref_out = torch.empty((3, 8, 128), device="cuda")
    ref_lse = torch.empty((3, 8), device="cuda")
    H.hash_attn_gather_att(shape, w.q, w.K, w.V, w.seq_lens, idx, cap, cnt, ref_out, ref_lse, workspace=ws)
    flags = torch.full((1,), 0xFF, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        H.hash_attn_gather_att_noalloc(shape, w.q, w.K, w.V, w.seq_lens, idx, cap, cnt, out, lse,
                                       dev_flags=flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0, f"call {call}: error word {int(flags.item()):#x}"
        ref_o = ref_out.cpu().numpy()
        ref_l = ref_lse.cpu().numpy()
        got_o = out.cpu().numpy()
        got_l = lse.cpu().numpy()
        for b in range(3):
            for h in range(8):
                GH.assert_out_close(got_o[b, h], ref_o[b, h], f"call {call} ({b},{h})")
                GH.assert_lse_close(float(got_l[b, h]), float(ref_l[b, h]), f"call {call} ({b},{h})")


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
    # a shape whose scratch exceeds the built-in array is refused before any launch
    big = H.HAShape()
    ctypes.pointer(big)[0] = shape
    big.batch = 4096
    big.q_sb = 0
    big.k_sb = big.v_sb = 0
    st = H.lib().hash_attn_gather_att_noalloc(ctypes.byref(big), w.q.data_ptr(), w.K.data_ptr(),
                                              w.V.data_ptr(), w.seq_lens.data_ptr(), idx.data_ptr(), 2000,
                                              cnt.data_ptr(), out.data_ptr(), lse.data_ptr(), None, None)
    assert st == H.HA_ERR_WORKSPACE and "scratch" in H.last_error()
