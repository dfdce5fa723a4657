"""Host-side tests of the C ABI that need no GPU.

The library must build, load and export every entry point that
include/hashattn.h declares; argument errors must come back as status codes
before anything is enqueued (so these calls never touch a device).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ha():
    from long_context_sparse_score_gb300 import _build
    _build.build()
    from long_context_sparse_score_gb300 import hashattn
    return hashattn


def _declared():
    text = open(os.path.join(ROOT, "include", "hashattn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:ha_status|size_t|int32_t|const char\*)\s+(hash_attn_\w+)\(",
                                 text, re.M)))


def test_header_declares_the_binding_names(ha):
    assert _declared() == sorted(ha.EXPORTED)


def test_library_exports_every_declared_symbol(ha):
    L = ha.lib()
    for name in _declared():
        assert hasattr(L, name), name


def _shape(ha, **kw):
    s = ha.HAShape()
    s.batch, s.h_q, s.h_kv, s.d, s.n_cap = 2, 8, 2, 128, 4096
    s.q_dtype = s.kv_dtype = ha.HA_BF16
    s.q_sb, s.q_sh = 8 * 128, 128
    s.k_sb, s.k_sh, s.k_sn = 2 * 4096 * 128, 4096 * 128, 128
    s.v_sb, s.v_sh, s.v_sn = s.k_sb, s.k_sh, s.k_sn
    s.ks_sb, s.ks_sh = 2 * 4096, 4096
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def _ws_size(ha, s, m=256, S=16, L=16):
    out = ctypes.c_size_t(0)
    st = ha.lib().hash_attn_workspace_size(ctypes.byref(s), m, S, L, ctypes.byref(out))
    return st, out.value


def test_workspace_size_and_capacity(ha):
    st, nbytes = _ws_size(ha, _shape(ha))
    assert st == ha.HA_OK and nbytes > 0 and nbytes % 256 == 0
    # the budget arithmetic of the pages: 16,384 tokens, m=1,024, 128 + 128 -> 1,280 reads
    assert ha.hash_attn_select_capacity(16384, 1024, 128, 128) == 1280
    assert ha.hash_attn_select_capacity(1000, 1024, 128, 128) == 1000
    assert ha.hash_attn_select_capacity(4096, 0, 0, 0) == 0
    # a dense-sized workspace (m >= n_cap) is at least as large as a sparse one
    assert _ws_size(ha, _shape(ha), m=4096)[1] >= nbytes


def _plan(ha, B, Hq, Hkv, n_cap, code_words=1):
    s = _shape(ha, batch=B, h_q=Hq, h_kv=Hkv, n_cap=n_cap, q_sb=Hq * 128, k_sb=Hkv * n_cap * 128,
               k_sh=n_cap * 128, v_sb=Hkv * n_cap * 128, v_sh=n_cap * 128, ks_sb=Hkv * n_cap, ks_sh=n_cap)
    return ha.hash_attn_selection_plan(s, code_words)


def test_selection_plan_of_the_workloads(ha):
    """32-bit codes take the fused selection (each distance computed once, one CTA
    per 8,192 tokens) at any context length: with more than four query heads per
    KV head the decode splits each KV head's heads into groups of at most four
    (virtual KV heads reading the same codes and rows). Wider codes take the
    two-kernel path, as does the selection entry point for more than four heads
    per KV head (the plan's chunk is that path's)."""
    for name, shape in {"tiny": (1, 1, 1, 1024), "gqa32k": (1, 32, 8, 32768), "batch16_128k": (16, 32, 8, 131072),
                        "shared_doc": (32, 32, 8, 61440), "ragged": (64, 32, 8, 65536),
                        "2m": (1, 4, 1, 1 << 21)}.items():
        p = _plan(ha, *shape)
        assert p["fused"] == 1 and p["range"] == 8192 and p["ranges"] == -(-shape[3] // 8192), (name, p)
    # 5, 6, 7, 8, 12 and 16 query heads per KV head: virtual groups of at most four
    for Hq in (40, 48, 56, 64, 96, 128):
        p = _plan(ha, 2, Hq, 8, 131072)
        assert p["fused"] == 1 and p["ranges"] == 16, (Hq, p)
    assert _plan(ha, 16, 32, 8, 131072, code_words=4)["fused"] == 0  # 128-bit codes
    # a single long sequence on the two-kernel path keeps within its segment table
    for n in (1 << 21, 1 << 22):
        p = _plan(ha, 1, 8, 1, n)
        assert -(-n // p["chunk"]) * 8 <= 4096, (n, p)
    with pytest.raises(ha.HashAttnError):
        _plan(ha, 1, 4, 1, 4096, code_words=3)


def test_decode_path_reports_the_kernels(ha):
    """hash_attn_decode_path (host only: nothing is launched). The batch-16 128K
    shape and the shared 61,440-token document take the GQA-group kernel; with
    selection outputs the fused lists; 128-bit codes the two-kernel path; m >=
    n_cap the dense group kernel, or the per-head one for an fp32 cache; a
    per-sequence budget keeps the selection even at m = n_cap."""
    n = 131072
    s = _shape(ha, batch=16, h_q=32, h_kv=8, n_cap=n, q_sb=32 * 128, k_sb=8 * n * 128, k_sh=n * 128,
               v_sb=8 * n * 128, v_sh=n * 128, ks_sb=8 * n, ks_sh=n)
    P = ha.hash_attn_decode_path
    assert P(s, 4096) == "group"
    assert P(s, 4096, with_selection=True) == "fused_lists"
    assert P(s, 4096, opts=ha.select_opts(None, False, 4)) == "two_kernel"
    assert P(s, n) == "dense_group"
    assert P(s, n, m_per_seq=1 << 20) == "group"
    s32 = _shape(ha, batch=16, h_q=32, h_kv=8, n_cap=n, q_sb=32 * 128, k_sb=8 * n * 128, k_sh=n * 128,
                 v_sb=8 * n * 128, v_sh=n * 128, ks_sb=8 * n, ks_sh=n, kv_dtype=ha.HA_F32)
    assert P(s32, n) == "dense_heads"
    nd = 61440
    doc = _shape(ha, batch=32, h_q=32, h_kv=8, n_cap=nd, q_sb=32 * 128, k_sb=0, k_sh=nd * 128, v_sb=0,
                 v_sh=nd * 128, ks_sb=0, ks_sh=nd)
    assert P(doc, 2048) == "group"
    # eight query heads per KV head: virtual groups of four on the group kernel
    s8 = _shape(ha, batch=2, h_q=64, h_kv=8, n_cap=n, q_sb=64 * 128, k_sb=8 * n * 128, k_sh=n * 128,
                v_sb=8 * n * 128, v_sh=n * 128, ks_sb=8 * n, ks_sh=n)
    assert P(s8, 4096) == "group"
    with pytest.raises(ha.HashAttnError):
        P(s, -1)


def test_fused_workspace_is_sized_by_the_budget_not_the_context(ha):
    """With the fused kernel the token lists take heads x (m + n_sink + n_local) ints,
    not heads x n_cap: at the 16 x 131,072-token shape well under 100 MB."""
    s = _shape(ha, batch=16, h_q=32, h_kv=8, n_cap=131072, q_sb=32 * 128, k_sb=8 * 131072 * 128,
               k_sh=131072 * 128, v_sb=8 * 131072 * 128, v_sh=131072 * 128, ks_sb=8 * 131072, ks_sh=131072)
    st, nbytes = _ws_size(ha, s, m=4096, S=128, L=256)
    assert st == ha.HA_OK and nbytes < 100 * 2 ** 20, nbytes


@pytest.mark.parametrize("field,value,status", [
    ("d", 96, -2), ("d", 256, -2), ("h_q", 7, -1), ("h_kv", 0, -1), ("batch", 0, -1),
    ("n_cap", 0, -1), ("kv_dtype", 5, -2), ("q_dtype", -1, -2), ("k_sn", 0, -1), ("q_sh", -3, -1),
])
def test_bad_shape_is_rejected(ha, field, value, status):
    st, _ = _ws_size(ha, _shape(ha, **{field: value}))
    assert st == status
    assert ha.last_error() != ""


def _decode(ha, s, *, q=512, q_sig=512, k_sig=512, K=512, V=512, seq=512, m=256, S=16, L=16,
            out=512, lse=512, ws=1024, ws_bytes=None, sel=None, cnt=None):
    if ws_bytes is None:
        ws_bytes = 1 << 40
    return ha.lib().hash_attn_decode(ctypes.byref(s), q, q_sig, k_sig, K, V, seq, None, m, S, L,
                                     out, lse, sel, cnt, ws, ws_bytes, None)


def test_decode_argument_errors_before_launch(ha):
    s = _shape(ha)
    assert _decode(ha, s, q=None) == ha.HA_ERR_INVALID_ARG
    assert _decode(ha, s, K=None) == ha.HA_ERR_INVALID_ARG
    assert _decode(ha, s, out=None) == ha.HA_ERR_INVALID_ARG
    assert _decode(ha, s, k_sig=None) == ha.HA_ERR_INVALID_ARG          # sparse path needs codes
    assert _decode(ha, s, k_sig=516) == ha.HA_ERR_INVALID_ARG           # unaligned codes
    assert _decode(ha, s, K=520) == ha.HA_ERR_INVALID_ARG               # unaligned rows
    assert _decode(ha, s, m=-1) == ha.HA_ERR_INVALID_ARG
    assert _decode(ha, s, S=-4) == ha.HA_ERR_INVALID_ARG
    assert _decode(ha, s, ws=None) == ha.HA_ERR_WORKSPACE
    assert _decode(ha, s, ws=1024 + 16) == ha.HA_ERR_WORKSPACE           # not 256-aligned
    assert _decode(ha, s, ws_bytes=1024) == ha.HA_ERR_WORKSPACE          # too small
    assert _decode(ha, s, sel=512) == ha.HA_ERR_INVALID_ARG              # sel_idx without sel_cnt
    assert _decode(ha, _shape(ha, ks_sh=4095)) == ha.HA_ERR_INVALID_ARG  # code rows unaligned
    assert _decode(ha, _shape(ha, k_sn=100)) == ha.HA_ERR_INVALID_ARG    # 200-byte row stride
    assert _decode(ha, _shape(ha, d=80)) == ha.HA_ERR_UNSUPPORTED
    assert "workspace" in ha.last_error() or ha.last_error() != ""


def test_other_entry_points_reject_bad_arguments(ha):
    L = ha.lib()
    s = _shape(ha)
    sp = ctypes.byref(s)
    assert L.hash_attn_score(sp, 512, 512, 512, None, None, 1024, 1 << 40, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_select(sp, 512, 512, 512, None, 8, 0, 0, None, 512, 1024, 1 << 40,
                              None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_gather_att(sp, 512, 512, 512, 512, 512, 5000, 512, 512, 512, 1024, 1 << 40,
                                  None) == ha.HA_ERR_INVALID_ARG     # idx_cap > n_cap
    assert L.hash_attn_merge(512, 512, 512, 512, 512, 512, -1, 128, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_merge(None, 512, 512, 512, 512, 512, 4, 128, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_merge(None, None, None, None, None, None, 0, 128, None) == ha.HA_OK  # nothing to do
    # multi-segment merge: segment count, row/dim bounds, overlapping strides, nulls
    assert L.hash_attn_merge_n(512, 512, 512, 512, 0, 512, 512, 4, 128, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_merge_n(512, 4 * 128 - 1, 512, 4, 3, 512, 512, 4, 128, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_merge_n(512, 4 * 128, 512, 3, 3, 512, 512, 4, 128, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_merge_n(None, 512, 512, 4, 3, 512, 512, 4, 128, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_merge_n(512, 512, 512, 4, 2, 512, 512, 4, 0, None) == ha.HA_ERR_INVALID_ARG
    assert L.hash_attn_merge_n(None, 0, None, 0, 2, None, None, 0, 128, None) == ha.HA_OK  # nothing to do
    assert L.hash_attn_device_status(None, None, None) == ha.HA_ERR_WORKSPACE
    assert L.hash_attn_workspace_init(None, 16, None) == ha.HA_ERR_WORKSPACE
    ev3 = (ctypes.c_void_p * 3)(512, None, 512)
    assert L.hash_attn_topk_exact_timed(sp, 512, 512, 512, 8, 512, 8, 512, 1 << 20, 1 << 40, None,
                                        ev3) == ha.HA_ERR_INVALID_ARG          # events[1] is NULL
    events = (ctypes.c_void_p * 4)(None, None, None, None)
    assert L.hash_attn_decode_timed(sp, 512, 512, 512, 512, 512, 512, None, 8, 0, 0, 512, 512, None,
                                    None, 1024, 1 << 40, None, events) == ha.HA_ERR_INVALID_ARG


def test_map_entry_points_reject_bad_arguments(ha):
    """The MLP encoders and the mapped decode check the map before anything is
    enqueued (every call here fails its checks, so no device is touched)."""
    L = ha.lib()
    s = _shape(ha)
    sp = ctypes.byref(s)
    good = ha.HAMlp(512, 512, 512, 512, 512, 512, 128, 0)
    assert L.hash_attn_encode_queries_mlp(sp, 512, None, 512, None) == ha.HA_ERR_INVALID_ARG
    for bad, status in ((ha.HAMlp(512, 512, 512, 512, 512, 512, 96, 0), ha.HA_ERR_UNSUPPORTED),
                        (ha.HAMlp(512, 512, 520, 512, 512, 512, 128, 0), ha.HA_ERR_INVALID_ARG),  # W2 unaligned
                        (ha.HAMlp(512, None, 512, 512, 512, 512, 128, 0), ha.HA_ERR_INVALID_ARG),
                        (ha.HAMlp(512, 512, 512, 512, 512, 512, 128, 1), ha.HA_ERR_INVALID_ARG)):
        assert L.hash_attn_encode_queries_mlp(sp, 512, ctypes.byref(bad), 512, None) == status
        assert L.hash_attn_encode_keys_mlp(sp, 512, ctypes.byref(bad), 512, 512, None, None) == status
    assert L.hash_attn_encode_keys_mlp(sp, 512, ctypes.byref(good), None, 512, None, None) == ha.HA_ERR_INVALID_ARG

    def mapped(map_, opts=None, ws_bytes=1024, q_sig=512):
        return L.hash_attn_decode_mapped(sp, 512, map_, None, q_sig, 512, 512, 512, 512, None, 8, 0, 0, opts,
                                         512, 512, None, None, 1024, ws_bytes, None, None)
    assert mapped(None) == ha.HA_ERR_INVALID_ARG
    both = ha.HAMap()
    both.W = 512
    both.mlp = ctypes.pointer(good)
    assert mapped(ctypes.byref(both)) == ha.HA_ERR_INVALID_ARG                     # both maps given
    assert mapped(ctypes.byref(ha.HAMap())) == ha.HA_ERR_INVALID_ARG               # neither
    wide = ha.select_opts(code_words=4)
    assert mapped(ctypes.byref(_w512(ha)), ctypes.byref(wide)) == ha.HA_ERR_UNSUPPORTED
    assert mapped(ctypes.byref(_w512(ha)), q_sig=None) == ha.HA_ERR_INVALID_ARG     # no q_sig
    assert mapped(ctypes.byref(_w512(ha))) == ha.HA_ERR_WORKSPACE                  # 1 KB workspace
    bad_mlp = ha.HAMlp(512, 512, 512, 512, 512, 512, 48, 0)
    assert mapped(ctypes.byref(ha.mlp_map(bad_mlp))) == ha.HA_ERR_UNSUPPORTED


def test_host_buffer_decode_checks_before_any_copy(ha):
    """hash_attn_decode_host runs the staging check and every check of the
    decode before it enqueues its first copy (no device is touched here)."""
    L = ha.lib()
    s = _shape(ha)
    sp = ctypes.byref(s)
    need = ctypes.c_size_t(0)
    assert L.hash_attn_host_staging_size(sp, ctypes.byref(need)) == ha.HA_OK and need.value > 0

    def call(q=512, seq=512, out=512, staging=1024, st_bytes=None, ws_bytes=1024, m=8):
        return L.hash_attn_decode_host(sp, q, 512, seq, None, 512, 512, 512, m, 0, 0, out, 512, staging,
                                       need.value if st_bytes is None else st_bytes, 1024, ws_bytes, None)
    assert call(q=None) == ha.HA_ERR_INVALID_ARG
    assert call(seq=None) == ha.HA_ERR_INVALID_ARG
    assert call(out=None) == ha.HA_ERR_INVALID_ARG
    assert call(staging=1024 + 16) == ha.HA_ERR_WORKSPACE              # unaligned staging
    assert call(st_bytes=need.value - 1) == ha.HA_ERR_WORKSPACE        # staging too small
    assert call() == ha.HA_ERR_WORKSPACE                                # the decode's own workspace check
    assert call(m=-1) == ha.HA_ERR_INVALID_ARG


def _w512(ha):
    m = ha.HAMap()
    m.W = 512
    return m


def test_status_strings(ha):
    for code in range(0, -7, -1):
        assert ha.status_string(code) not in ("", "unknown status")
    assert ha.status_string(-99) == "unknown status"


def test_product_path_fails_loudly_without_the_library(ha, monkeypatch, tmp_path):
    from long_context_sparse_score_gb300 import hashattn
    monkeypatch.setattr(hashattn, "_lib", None)
    monkeypatch.setattr(hashattn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        hashattn.lib()


def test_bench_traffic_key_ignores_comments(tmp_path):
    """The bench's recorded DRAM traffic stays valid across comment edits of the
    kernel source and lapses on any code change."""
    import bench
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int* p) {  // a kernel\n    p[0] = 1;\n}\n")
    key = bench.source_code_key(str(src))
    src.write_text("// another header\n\n__global__ void k(int* p) {  // the same kernel\n    p[0] = 1;\n}\n")
    assert bench.source_code_key(str(src)) == key
    src.write_text("// header\n__global__ void k(int* p) {\n    p[0] = 2;\n}\n")
    assert bench.source_code_key(str(src)) != key
