"""Python binding of libhashattn.so (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls and forwards
device pointers taken from torch tensors plus the current CUDA stream. No step
of the computation runs in Python or torch. Loading fails loudly when the
library has not been built: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH

HA_OK = 0
HA_ERR_INVALID_ARG = -1
HA_ERR_UNSUPPORTED = -2
HA_ERR_WORKSPACE = -3
HA_ERR_CUDA = -4
HA_ERR_DEVICE = -5
HA_ERR_TIMEOUT = -6

HA_F32 = 0
HA_BF16 = 1

HA_DEVERR_SEQLEN = 0x1
HA_DEVERR_BUDGET = 0x2
HA_DEVERR_INDEX = 0x4
HA_DEVERR_COUNT = 0x8
HA_DEVERR_TIMEOUT = 0x10
HA_DEVERR_STATE = 0x20

HA_NBINS = 33
HA_NOALLOC_SCRATCH_BYTES = 16 << 20

# Entry points declared in include/hashattn.h (checked by the tests).
EXPORTED = [
    "hash_attn_workspace_size", "hash_attn_workspace_init", "hash_attn_select_capacity",
    "hash_attn_decode", "hash_attn_decode_ex", "hash_attn_decode_timed", "hash_attn_decode_host",
    "hash_attn_host_staging_size", "hash_attn_score", "hash_attn_select",
    "hash_attn_select_ex", "hash_attn_workspace_size_ex", "hash_attn_selection_plan", "hash_attn_decode_path",
    "hash_attn_gather_att", "hash_attn_gather_att_noalloc", "hash_attn_merge", "hash_attn_merge_n",
    "hash_attn_encode_queries", "hash_attn_encode_keys", "hash_attn_encode_queries_mlp",
    "hash_attn_encode_keys_mlp", "hash_attn_decode_mapped", "hash_attn_topk_exact_workspace_size",
    "hash_attn_topk_exact", "hash_attn_topk_exact_timed", "hash_attn_recall",
    "hash_attn_device_status",
    "hash_attn_status_string", "hash_attn_last_error",
]


class HASelectOpts(ctypes.Structure):
    """Mirror of ``ha_select_opts``."""

    _fields_ = [("m_per_head", ctypes.c_void_p), ("exclusive_windows", ctypes.c_int32),
                ("code_words", ctypes.c_int32), ("reserved", ctypes.c_int32 * 2)]


def select_opts(m_per_head=None, exclusive_windows=False, code_words=1) -> HASelectOpts:
    o = HASelectOpts()
    o.m_per_head = _ptr(m_per_head)
    o.exclusive_windows = 1 if exclusive_windows else 0
    o.code_words = int(code_words)
    return o


class HAMlp(ctypes.Structure):
    """Mirror of ``ha_mlp`` (the MLP signature map's weights, device pointers)."""

    _fields_ = [("W1", ctypes.c_void_p), ("b1", ctypes.c_void_p), ("W2", ctypes.c_void_p),
                ("b2", ctypes.c_void_p), ("W3", ctypes.c_void_p), ("b3", ctypes.c_void_p),
                ("hidden", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def mlp(W1, b1, W2, b2, W3, b3) -> HAMlp:
    """HAMlp over float32 device tensors W1 [h_kv, H, d], b1 [h_kv, H], W2 [h_kv, H, H],
    b2 [h_kv, H], W3 [h_kv, 32, H], b3 [h_kv, 32]. The struct holds raw pointers:
    keep the tensors alive while it is used."""
    m = HAMlp()
    m.W1, m.b1, m.W2, m.b2, m.W3, m.b3 = (_ptr(t) for t in (W1, b1, W2, b2, W3, b3))
    m.hidden = int(W1.shape[1])
    return m


class HAMap(ctypes.Structure):
    """Mirror of ``ha_map``: exactly one of W (sign projection) and mlp."""

    _fields_ = [("W", ctypes.c_void_p), ("mlp", ctypes.POINTER(HAMlp))]


def sign_map(W) -> HAMap:
    m = HAMap()
    m.W = _ptr(W)
    return m


def mlp_map(weights: HAMlp) -> HAMap:
    m = HAMap()
    m.mlp = ctypes.pointer(weights)
    return m


class HAShape(ctypes.Structure):
    """Mirror of ``ha_shape`` (all strides in elements)."""

    _fields_ = [
        ("batch", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
        ("d", ctypes.c_int32), ("n_cap", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("q_sb", ctypes.c_int64), ("q_sh", ctypes.c_int64),
        ("k_sb", ctypes.c_int64), ("k_sh", ctypes.c_int64), ("k_sn", ctypes.c_int64),
        ("v_sb", ctypes.c_int64), ("v_sh", ctypes.c_int64), ("v_sn", ctypes.c_int64),
        ("ks_sb", ctypes.c_int64), ("ks_sh", ctypes.c_int64),
    ]


class HashAttnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{status_string(status)} ({status}): {detail}")
        self.status = status
        self.detail = detail


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded library (raises if libhashattn.so has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libhashattn.so not built at {LIB_PATH}; run __graft_entry__.build() "
                          "or python long_context_sparse_score_gb300/_build.py")
    L = ctypes.CDLL(LIB_PATH)
    SP = ctypes.POINTER(HAShape)
    L.hash_attn_workspace_size.argtypes = [SP, _I32, _I32, _I32, ctypes.POINTER(_SZ)]
    L.hash_attn_workspace_init.argtypes = [_P, _SZ, _P]
    L.hash_attn_select_capacity.argtypes = [_I32, _I32, _I32, _I32]
    L.hash_attn_select_capacity.restype = _I32
    dec = [SP, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P]
    L.hash_attn_decode.argtypes = dec
    OP = ctypes.POINTER(HASelectOpts)
    L.hash_attn_decode_ex.argtypes = dec[:11] + [OP] + dec[11:]
    L.hash_attn_select_ex.argtypes = [SP, _P, _P, _P, _P, _I32, _I32, _I32, OP, _P, _P, _P, _SZ, _P]
    L.hash_attn_workspace_size_ex.argtypes = [SP, _I32, _I32, _I32, OP, ctypes.POINTER(_SZ)]
    L.hash_attn_decode_timed.argtypes = dec + [ctypes.POINTER(_P)]
    IP = ctypes.POINTER(_I32)
    L.hash_attn_selection_plan.argtypes = [SP, _I32, IP, IP, IP, IP]
    L.hash_attn_decode_path.argtypes = [SP, _I32, _P, OP, _I32, IP]
    L.hash_attn_host_staging_size.argtypes = [SP, ctypes.POINTER(_SZ)]
    L.hash_attn_decode_host.argtypes = [SP, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _SZ, _P, _SZ,
                                        _P]
    L.hash_attn_score.argtypes = [SP, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.hash_attn_select.argtypes = [SP, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _SZ, _P]
    L.hash_attn_gather_att.argtypes = [SP, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _SZ, _P]
    L.hash_attn_gather_att_noalloc.argtypes = [SP, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P]
    L.hash_attn_merge.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _I32, _P]
    L.hash_attn_merge_n.argtypes = [_P, ctypes.c_int64, _P, ctypes.c_int64, _I32, _P, _P, _I32, _I32, _P]
    L.hash_attn_encode_queries.argtypes = [SP, _P, _P, _P, _P]
    L.hash_attn_encode_keys.argtypes = [SP, _P, _P, _P, _P, _P, _P]
    L.hash_attn_encode_queries_mlp.argtypes = [SP, _P, ctypes.POINTER(HAMlp), _P, _P]
    L.hash_attn_encode_keys_mlp.argtypes = [SP, _P, ctypes.POINTER(HAMlp), _P, _P, _P, _P]
    L.hash_attn_decode_mapped.argtypes = [SP, _P, ctypes.POINTER(HAMap), _P, _P, _P, _P, _P, _P, _P, _I32, _I32,
                                          _I32, OP, _P, _P, _P, _P, _P, _SZ, _P, _P]
    L.hash_attn_topk_exact_workspace_size.argtypes = [SP, ctypes.POINTER(_SZ)]
    L.hash_attn_topk_exact.argtypes = [SP, _P, _P, _P, _I32, _P, _I32, _P, _P, _SZ, _P]
    L.hash_attn_topk_exact_timed.argtypes = [SP, _P, _P, _P, _I32, _P, _I32, _P, _P, _SZ, _P, ctypes.POINTER(_P)]
    L.hash_attn_recall.argtypes = [_P, _P, _I32, _P, _P, _I32, _I32, _P, _P]
    L.hash_attn_device_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_uint32)]
    L.hash_attn_status_string.argtypes = [_I32]
    L.hash_attn_status_string.restype = ctypes.c_char_p
    L.hash_attn_last_error.argtypes = []
    L.hash_attn_last_error.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name not in ("hash_attn_select_capacity", "hash_attn_status_string", "hash_attn_last_error"):
            getattr(L, name).restype = _I32
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().hash_attn_status_string(status).decode()


def last_error() -> str:
    return lib().hash_attn_last_error().decode()


def _check(status: int) -> None:
    if status != HA_OK:
        raise HashAttnError(status, last_error())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return HA_F32
    if t.dtype == torch.bfloat16:
        return HA_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def make_shape(q, K, V, k_sig=None, *, n_cap=None, batch=None, share_kv=None) -> HAShape:
    """ha_shape from tensors: q [B, Hq, d], K/V [Bk, Hkv, n_cap, d], k_sig [Bk, Hkv, n_cap].

    A batch extent of 1 in K/V/k_sig with B > 1 is read as one cache shared by
    every batch entry (batch stride 0).
    """
    B, Hq, d = q.shape
    Bk, Hkv, ncap, dk = K.shape
    assert dk == d and V.shape == K.shape
    s = HAShape()
    s.batch, s.h_q, s.h_kv, s.d, s.n_cap = B, Hq, Hkv, d, ncap if n_cap is None else n_cap
    s.q_dtype, s.kv_dtype = _dtype_code(q), _dtype_code(K)
    s.q_sb, s.q_sh = q.stride(0), q.stride(1)
    shared = (Bk == 1 and B > 1) if share_kv is None else share_kv
    s.k_sb = 0 if shared else K.stride(0)
    s.k_sh, s.k_sn = K.stride(1), K.stride(2)
    s.v_sb = 0 if shared else V.stride(0)
    s.v_sh, s.v_sn = V.stride(1), V.stride(2)
    if k_sig is not None:
        s.ks_sb = 0 if (k_sig.shape[0] == 1 and B > 1) else k_sig.stride(0)
        s.ks_sh = k_sig.stride(1)
    return s


def hash_attn_workspace_size(shape: HAShape, m_max: int, n_sink: int, n_local: int) -> int:
    out = _SZ(0)
    _check(lib().hash_attn_workspace_size(ctypes.byref(shape), m_max, n_sink, n_local, ctypes.byref(out)))
    return out.value


def hash_attn_workspace_init(workspace, stream=None) -> None:
    _check(lib().hash_attn_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream)))


def hash_attn_select_capacity(n_cap: int, m: int, n_sink: int, n_local: int) -> int:
    return lib().hash_attn_select_capacity(n_cap, m, n_sink, n_local)


def _ws(workspace):
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def hash_attn_decode(shape, q, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local,
                     out, lse, sel_idx=None, sel_cnt=None, *, workspace, stream=None) -> None:
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_decode(ctypes.byref(shape), _ptr(q), _ptr(q_sig), _ptr(k_sig), _ptr(K),
                                  _ptr(V), _ptr(seq_lens), _ptr(m_per_seq), m, n_sink, n_local,
                                  _ptr(out), _ptr(lse), _ptr(sel_idx), _ptr(sel_cnt), ws, nb,
                                  _stream(stream)))


def hash_attn_host_staging_size(shape) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hash_attn_host_staging_size(ctypes.byref(shape), ctypes.byref(out)))
    return out.value


def hash_attn_decode_host(shape, q_host, q_sig_host, seq_lens_host, m_per_seq_host, k_sig, K, V, m, n_sink, n_local,
                          out_host, lse_host, *, staging, workspace, stream=None) -> None:
    """hash_attn_decode with q / q_sig / seq_lens / m_per_seq and out / lse in host
    memory (pinned tensors or raw addresses), staged through the device buffer
    ``staging`` (hash_attn_host_staging_size bytes)."""
    ws, nb = _ws(workspace)
    sp, sn = _ws(staging)
    _check(lib().hash_attn_decode_host(ctypes.byref(shape), _ptr(q_host), _ptr(q_sig_host), _ptr(seq_lens_host),
                                       _ptr(m_per_seq_host), _ptr(k_sig), _ptr(K), _ptr(V), m, n_sink, n_local,
                                       _ptr(out_host), _ptr(lse_host), sp, sn, ws, nb, _stream(stream)))


def hash_attn_workspace_size_ex(shape, m_max: int, n_sink: int, n_local: int, opts) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hash_attn_workspace_size_ex(ctypes.byref(shape), m_max, n_sink, n_local,
                                             None if opts is None else ctypes.byref(opts), ctypes.byref(out)))
    return out.value


def hash_attn_selection_plan(shape, code_words: int = 1) -> dict:
    """{"fused", "ranges", "range", "chunk"}: the selection path the library takes for a shape."""
    v = [ctypes.c_int32(0) for _ in range(4)]
    _check(lib().hash_attn_selection_plan(ctypes.byref(shape), int(code_words), *(ctypes.byref(x) for x in v)))
    return dict(zip(("fused", "ranges", "range", "chunk"), (x.value for x in v)))


# decode paths (hash_attn_decode_path)
PATHS = {1: "dense_group", 2: "dense_heads", 3: "group", 4: "fused_lists", 5: "two_kernel"}


def hash_attn_decode_path(shape, m: int, m_per_seq=None, opts=None, with_selection: bool = False) -> str:
    """The kernels a decode call with this shape, budget and options runs (a name of PATHS)."""
    out = ctypes.c_int32(0)
    _check(lib().hash_attn_decode_path(ctypes.byref(shape), int(m), _ptr(m_per_seq),
                                       None if opts is None else ctypes.byref(opts), 1 if with_selection else 0,
                                       ctypes.byref(out)))
    return PATHS[out.value]


def hash_attn_decode_ex(shape, q, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local, opts,
                        out, lse, sel_idx=None, sel_cnt=None, *, workspace, stream=None) -> None:
    """``opts``: an HASelectOpts (see ``select_opts``) or None."""
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_decode_ex(ctypes.byref(shape), _ptr(q), _ptr(q_sig), _ptr(k_sig), _ptr(K), _ptr(V),
                                     _ptr(seq_lens), _ptr(m_per_seq), m, n_sink, n_local,
                                     None if opts is None else ctypes.byref(opts), _ptr(out), _ptr(lse),
                                     _ptr(sel_idx), _ptr(sel_cnt), ws, nb, _stream(stream)))


def hash_attn_decode_timed(shape, q, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local,
                           out, lse, events, sel_idx=None, sel_cnt=None, *, workspace,
                           stream=None) -> None:
    """``events``: four torch.cuda.Event(enable_timing=True)."""
    ws, nb = _ws(workspace)
    arr = (_P * 4)(*[e.cuda_event for e in events])
    _check(lib().hash_attn_decode_timed(ctypes.byref(shape), _ptr(q), _ptr(q_sig), _ptr(k_sig),
                                        _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(m_per_seq), m,
                                        n_sink, n_local, _ptr(out), _ptr(lse), _ptr(sel_idx),
                                        _ptr(sel_cnt), ws, nb, _stream(stream), arr))


def hash_attn_score(shape, q_sig, k_sig, seq_lens, dist=None, hist=None, *, workspace,
                    stream=None) -> None:
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_score(ctypes.byref(shape), _ptr(q_sig), _ptr(k_sig), _ptr(seq_lens),
                                 _ptr(dist), _ptr(hist), ws, nb, _stream(stream)))


def hash_attn_select(shape, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink, n_local, sel_idx, sel_cnt,
                     *, workspace, stream=None) -> None:
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_select(ctypes.byref(shape), _ptr(q_sig), _ptr(k_sig), _ptr(seq_lens),
                                  _ptr(m_per_seq), m, n_sink, n_local, _ptr(sel_idx), _ptr(sel_cnt),
                                  ws, nb, _stream(stream)))


def hash_attn_select_ex(shape, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink, n_local, opts, sel_idx, sel_cnt,
                        *, workspace, stream=None) -> None:
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_select_ex(ctypes.byref(shape), _ptr(q_sig), _ptr(k_sig), _ptr(seq_lens),
                                     _ptr(m_per_seq), m, n_sink, n_local,
                                     None if opts is None else ctypes.byref(opts), _ptr(sel_idx), _ptr(sel_cnt),
                                     ws, nb, _stream(stream)))


def hash_attn_gather_att(shape, q, K, V, seq_lens, idx, idx_cap, cnt, out, lse, *, workspace,
                         stream=None) -> None:
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_gather_att(ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(V), _ptr(seq_lens),
                                      _ptr(idx), idx_cap, _ptr(cnt), _ptr(out), _ptr(lse), ws, nb,
                                      _stream(stream)))


def hash_attn_gather_att_noalloc(shape, q, K, V, seq_lens, idx, idx_cap, cnt, out, lse, dev_flags=None,
                                 stream=None) -> None:
    """hash_attn_gather_att without a workspace: the library's built-in scratch
    serves (for callers that may not allocate device memory)."""
    _check(lib().hash_attn_gather_att_noalloc(ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(V),
                                              _ptr(seq_lens), _ptr(idx), idx_cap, _ptr(cnt), _ptr(out),
                                              _ptr(lse), _ptr(dev_flags), _stream(stream)))


def hash_attn_merge(out_a, lse_a, out_b, lse_b, out, lse, rows: int, d: int, stream=None) -> None:
    _check(lib().hash_attn_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out),
                                 _ptr(lse), rows, d, _stream(stream)))


def hash_attn_merge_n(outs, lses, out, lse, stream=None) -> None:
    """``outs`` [nseg, rows, d] and ``lses`` [nseg, rows] float32 (rows contiguous
    within a segment; any segment stride); ``out`` [rows, d], ``lse`` [rows]."""
    nseg, rows, d = outs.shape
    if tuple(lses.shape) != (nseg, rows) or outs.stride(1) != d or outs.stride(2) != 1 or lses.stride(1) != 1:
        raise ValueError("outs must be [nseg, rows, d] with contiguous rows and lses [nseg, rows]")
    _check(lib().hash_attn_merge_n(_ptr(outs), outs.stride(0), _ptr(lses), lses.stride(0), nseg, _ptr(out),
                                   _ptr(lse), rows, d, _stream(stream)))


def hash_attn_encode_queries(shape, q, W, q_sig, stream=None) -> None:
    """q_sig[b, h] = sign-projection code of q[b, h] under W[h // G] (W float32 [h_kv, 32, d])."""
    _check(lib().hash_attn_encode_queries(ctypes.byref(shape), _ptr(q), _ptr(W), _ptr(q_sig), _stream(stream)))


def hash_attn_encode_keys(shape, K, W, pos, k_sig, dev_flags=None, stream=None) -> None:
    """k_sig[b, g, pos[b]] = code of K[b, g, pos[b]] under W[g], for pos[b] in [0, n_cap)."""
    _check(lib().hash_attn_encode_keys(ctypes.byref(shape), _ptr(K), _ptr(W), _ptr(pos), _ptr(k_sig),
                                       _ptr(dev_flags), _stream(stream)))


def hash_attn_encode_queries_mlp(shape, q, weights: HAMlp, q_sig, stream=None) -> None:
    """q_sig[b, h] = code of q[b, h] under the MLP map of KV head h / G."""
    _check(lib().hash_attn_encode_queries_mlp(ctypes.byref(shape), _ptr(q), ctypes.byref(weights), _ptr(q_sig),
                                              _stream(stream)))


def hash_attn_encode_keys_mlp(shape, K, weights: HAMlp, pos, k_sig, dev_flags=None, stream=None) -> None:
    """k_sig[b, g, pos[b]] = code of K[b, g, pos[b]] under the MLP map of KV head g."""
    _check(lib().hash_attn_encode_keys_mlp(ctypes.byref(shape), _ptr(K), ctypes.byref(weights), _ptr(pos),
                                           _ptr(k_sig), _ptr(dev_flags), _stream(stream)))


def hash_attn_decode_mapped(shape, q, map_, pos, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local,
                            opts, out, lse, sel_idx=None, sel_cnt=None, *, workspace, dev_flags=None,
                            stream=None) -> None:
    """One decode step with the signature map (``sign_map`` / ``mlp_map``) ahead of SCORE."""
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_decode_mapped(ctypes.byref(shape), _ptr(q), ctypes.byref(map_), _ptr(pos), _ptr(q_sig),
                                         _ptr(k_sig), _ptr(K), _ptr(V), _ptr(seq_lens), _ptr(m_per_seq), m,
                                         n_sink, n_local, None if opts is None else ctypes.byref(opts), _ptr(out),
                                         _ptr(lse), _ptr(sel_idx), _ptr(sel_cnt), ws, nb, _ptr(dev_flags),
                                         _stream(stream)))


def hash_attn_topk_exact_workspace_size(shape) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().hash_attn_topk_exact_workspace_size(ctypes.byref(shape), ctypes.byref(out)))
    return out.value


def hash_attn_topk_exact(shape, q, K, seq_lens, m, idx, cnt, *, workspace, stream=None) -> None:
    """idx [B, Hq, cap] / cnt [B, Hq]: the min(m, n) largest <q, k_i> per head, ascending."""
    ws, nb = _ws(workspace)
    _check(lib().hash_attn_topk_exact(ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(seq_lens), m, _ptr(idx),
                                      idx.shape[-1], _ptr(cnt), ws, nb, _stream(stream)))


def hash_attn_topk_exact_timed(shape, q, K, seq_lens, m, idx, cnt, events, *, workspace, stream=None) -> None:
    """hash_attn_topk_exact with ``events``: three torch.cuda.Event(enable_timing=True),
    recorded before the scores, between the scores and the top-m, and after."""
    ws, nb = _ws(workspace)
    arr = (_P * 3)(*[e.cuda_event for e in events])
    _check(lib().hash_attn_topk_exact_timed(ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(seq_lens), m, _ptr(idx),
                                            idx.shape[-1], _ptr(cnt), ws, nb, _stream(stream), arr))


def hash_attn_recall(sel_idx, sel_cnt, ref_idx, ref_cnt, recall, stream=None) -> None:
    """recall[h] = |sel_h & ref_h| / |ref_h| over [heads, cap] index lists (any leading shape)."""
    heads = sel_cnt.numel()
    _check(lib().hash_attn_recall(_ptr(sel_idx), _ptr(sel_cnt), sel_idx.shape[-1], _ptr(ref_idx), _ptr(ref_cnt),
                                  ref_idx.shape[-1], heads, _ptr(recall), _stream(stream)))


def hash_attn_device_status(workspace, stream=None) -> tuple[int, int]:
    """(status, raw flags); synchronises the stream and clears the error word."""
    flags = ctypes.c_uint32(0)
    st = lib().hash_attn_device_status(_ptr(workspace), _stream(stream), ctypes.byref(flags))
    return st, flags.value
