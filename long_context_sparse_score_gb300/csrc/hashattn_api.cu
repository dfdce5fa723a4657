// C ABI of the sparse-decode library: argument checks, workspace layout and the
// stream-ordered launch sequence SCORE -> TOPK -> GATHER-ATT (+ merge).
// Every check that the host can make happens before anything is enqueued.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "ha_internal.cuh"

namespace ha {

namespace {

thread_local std::string g_last_error;

ha_status fail(ha_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

ha_status cuda_fail(cudaError_t e, const char* what) {
    return fail(HA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int dtype) { return dtype == HA_F32 ? 4 : 2; }

ha_status check_shape(const ha_shape* s) {
    if (s == nullptr) return fail(HA_ERR_INVALID_ARG, "shape is NULL");
    if (s->batch < 1 || s->h_q < 1 || s->h_kv < 1)
        return fail(HA_ERR_INVALID_ARG, "batch, h_q and h_kv must be >= 1 (got %d, %d, %d)", s->batch,
                    s->h_q, s->h_kv);
    if (s->h_q % s->h_kv != 0)
        return fail(HA_ERR_INVALID_ARG, "h_q (%d) must be a multiple of h_kv (%d)", s->h_q, s->h_kv);
    if (s->d != 64 && s->d != 128) return fail(HA_ERR_UNSUPPORTED, "d must be 64 or 128 (got %d)", s->d);
    if ((s->q_dtype != HA_F32 && s->q_dtype != HA_BF16) || (s->kv_dtype != HA_F32 && s->kv_dtype != HA_BF16))
        return fail(HA_ERR_UNSUPPORTED, "dtypes must be HA_F32 or HA_BF16 (got q %d, kv %d)", s->q_dtype,
                    s->kv_dtype);
    if (s->n_cap < 1 || (int64_t)s->n_cap > kMaxCap)
        return fail(HA_ERR_INVALID_ARG, "n_cap must be in [1, %lld] (got %d)", (long long)kMaxCap, s->n_cap);
    if ((int64_t)s->batch * s->h_q > (int64_t)1 << 26)
        return fail(HA_ERR_INVALID_ARG, "batch * h_q too large");
    if (s->q_sb < 0 || s->q_sh < 0 || s->k_sb < 0 || s->k_sh < 0 || s->k_sn < 1 || s->v_sb < 0 ||
        s->v_sh < 0 || s->v_sn < 1 || s->ks_sb < 0 || s->ks_sh < 0)
        return fail(HA_ERR_INVALID_ARG, "strides must be >= 0 (token strides >= 1)");
    return HA_OK;
}

ha_status check_kv(const ha_shape* s, const void* K, const void* V) {
    if (K == nullptr || V == nullptr) return fail(HA_ERR_INVALID_ARG, "K or V is NULL");
    const int64_t es = elem_size(s->kv_dtype);
    if (!aligned16(K) || !aligned16(V)) return fail(HA_ERR_INVALID_ARG, "K and V must be 16-byte aligned");
    const int64_t strides[6] = {s->k_sb, s->k_sh, s->k_sn, s->v_sb, s->v_sh, s->v_sn};
    for (int64_t st : strides)
        if ((st * es) % 16 != 0)
            return fail(HA_ERR_INVALID_ARG, "K/V strides times the element size must be multiples of 16 bytes");
    return HA_OK;
}

ha_status check_codes(const ha_shape* s, const uint32_t* q_sig, const uint32_t* k_sig) {
    if (q_sig == nullptr || k_sig == nullptr) return fail(HA_ERR_INVALID_ARG, "q_sig or k_sig is NULL");
    if (!aligned16(k_sig) || s->ks_sh % 4 != 0 || s->ks_sb % 4 != 0)
        return fail(HA_ERR_INVALID_ARG, "k_sig rows must start on 16-byte boundaries (pointer, ks_sh, ks_sb)");
    return HA_OK;
}

ha_status check_window(int32_t m, int32_t n_sink, int32_t n_local) {
    if (m < 0 || n_sink < 0 || n_local < 0)
        return fail(HA_ERR_INVALID_ARG, "m, n_sink and n_local must be >= 0 (got %d, %d, %d)", m, n_sink,
                    n_local);
    return HA_OK;
}

ha_status check_ws(const Layout& lay, void* ws, size_t ws_bytes) {
    if (ws == nullptr) return fail(HA_ERR_WORKSPACE, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(HA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < lay.total)
        return fail(HA_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", ws_bytes, lay.total);
    return HA_OK;
}

ha_status check_segments(const Layout& lay) {
    if (!lay.fused && lay.nseg > kMaxSegments)
        return fail(HA_ERR_UNSUPPORTED, "n_cap too large for this batch: %d selection segments per head (limit %d)",
                    lay.nseg, kMaxSegments);
    return HA_OK;
}

int64_t rows_cap_of(int32_t n_cap, int64_t m, int64_t n_sink, int64_t n_local) {
    const int64_t r = m + n_sink + n_local;
    return r < n_cap ? r : n_cap;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

struct Views {
    uint32_t* err;
    uint32_t* counters;
    uint32_t* chunk_hist;
    int32_t* seg_cnt;
    int32_t* seg_idx;
    float* part;
    uint32_t* score_cnt;
    int32_t* meta_t;
    int2* meta_qt;
    int32_t* list;
    int32_t* lcnt;
};

Views views(const Layout& lay, void* ws) {
    Views v;
    const bool seg = lay.chunk && !lay.fused;
    v.err = at<uint32_t>(ws, lay.off_err);
    v.counters = at<uint32_t>(ws, lay.off_counter);
    v.chunk_hist = lay.chunk ? at<uint32_t>(ws, lay.off_hist) : nullptr;
    v.seg_cnt = seg ? at<int32_t>(ws, lay.off_segcnt) : nullptr;
    v.seg_idx = seg ? at<int32_t>(ws, lay.off_seg) : nullptr;
    v.part = at<float>(ws, lay.off_part);
    v.score_cnt = at<uint32_t>(ws, lay.off_scnt);
    v.meta_t = lay.chunk ? at<int32_t>(ws, lay.off_meta_t) : nullptr;
    v.meta_qt = lay.chunk ? at<int2>(ws, lay.off_meta_qt) : nullptr;
    v.list = lay.fused ? at<int32_t>(ws, lay.off_list) : nullptr;
    v.lcnt = lay.fused ? at<int32_t>(ws, lay.off_lcnt) : nullptr;
    return v;
}

ScoreParams score_params(const ha_shape* s, const Layout& lay, const Views& v, const uint32_t* q_sig,
                         const uint32_t* k_sig, const int32_t* seq_lens, const int32_t* m_per_seq,
                         int32_t m, bool thresholds) {
    ScoreParams p{};
    p.q_sig = q_sig;
    p.k_sig = k_sig;
    p.ks_sb = s->ks_sb;
    p.ks_sh = s->ks_sh;
    p.seq_lens = seq_lens;
    p.B = s->batch;
    p.Hq = s->h_q;
    p.Hkv = s->h_kv;
    p.G = s->h_q / s->h_kv;
    p.n_cap = s->n_cap;
    p.chunk = lay.chunk;
    p.nchunks = lay.nchunks;
    p.chunk_hist = v.chunk_hist;
    p.counters = v.counters;
    p.dist = nullptr;
    p.err = v.err;
    p.m_per_seq = m_per_seq;
    p.m = m;
    p.score_cnt = thresholds ? v.score_cnt : nullptr;
    p.meta_t = thresholds ? v.meta_t : nullptr;
    p.meta_qt = thresholds ? v.meta_qt : nullptr;
    return p;
}

SelectParams select_params(const ha_shape* s, const Layout& lay, const Views& v, const uint32_t* q_sig,
                           const uint32_t* k_sig, const int32_t* seq_lens, int32_t n_sink, int32_t n_local) {
    SelectParams p{};
    p.q_sig = q_sig;
    p.k_sig = k_sig;
    p.ks_sb = s->ks_sb;
    p.ks_sh = s->ks_sh;
    p.seq_lens = seq_lens;
    p.n_sink = n_sink;
    p.n_local = n_local;
    p.B = s->batch;
    p.Hq = s->h_q;
    p.Hkv = s->h_kv;
    p.G = s->h_q / s->h_kv;
    p.n_cap = s->n_cap;
    p.chunk = lay.chunk;
    p.nchunks = lay.nchunks;
    p.meta_t = v.meta_t;
    p.meta_qt = v.meta_qt;
    p.seg_cnt = v.seg_cnt;
    p.seg_idx = v.seg_idx;
    p.err = v.err;
    return p;
}

GatherParams gather_params(const ha_shape* s, const Layout& lay, const Views& v, const void* q,
                           const void* K, const void* V, const int32_t* seq_lens, float* out, float* lse) {
    GatherParams p{};
    p.q = q;
    p.q_sb = s->q_sb;
    p.q_sh = s->q_sh;
    p.q_bf16 = s->q_dtype == HA_BF16;
    p.K = static_cast<const char*>(K);
    p.V = static_cast<const char*>(V);
    p.k_sb = s->k_sb;
    p.k_sh = s->k_sh;
    p.k_sn = s->k_sn;
    p.v_sb = s->v_sb;
    p.v_sh = s->v_sh;
    p.v_sn = s->v_sn;
    p.seq_lens = seq_lens;
    p.B = s->batch;
    p.Hq = s->h_q;
    p.Hkv = s->h_kv;
    p.G = s->h_q / s->h_kv;
    p.kv_mul = 0u;
    p.n_cap = s->n_cap;
    p.mode = kIdentity;
    p.seg_cap = lay.seg_cap;
    p.nseg = lay.nseg;
    p.seg_cnt = v.seg_cnt;
    p.seg_idx = v.seg_idx;
    p.splits = lay.splits;
    p.rows_per_split = lay.rows_per_split;
    p.part = v.part;
    p.counters = v.counters;
    p.err = v.err;
    p.out = out;
    p.lse = lse;
    p.qscale = (float)(1.4426950408889634 / std::sqrt((double)s->d));
    return p;
}

ha_status record(void* const* events, int i, cudaStream_t st) {
    if (events == nullptr) return HA_OK;
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st);
    return e == cudaSuccess ? HA_OK : cuda_fail(e, "cudaEventRecord");
}

#define HA_TRY(expr)                      \
    do {                                  \
        const ha_status _st = (expr);     \
        if (_st != HA_OK) return _st;     \
    } while (0)

#define HA_LAUNCH(expr, what)                              \
    do {                                                   \
        const cudaError_t _e = (expr);                     \
        if (_e != cudaSuccess) return cuda_fail(_e, what); \
    } while (0)

ha_status check_opts(const ha_select_opts* o) {
    if (o == nullptr) return HA_OK;
    if (o->exclusive_windows != 0 && o->exclusive_windows != 1)
        return fail(HA_ERR_INVALID_ARG, "exclusive_windows must be 0 or 1 (got %d)", o->exclusive_windows);
    const int w = o->code_words;
    if (w != 0 && w != 1 && w != 2 && w != 4 && w != 8 && w != 16)
        return fail(HA_ERR_UNSUPPORTED, "code_words must be 1, 2, 4, 8 or 16 (got %d)", w);
    if (w > 1 && (o->exclusive_windows || o->m_per_head != nullptr))
        return fail(HA_ERR_UNSUPPORTED, "codes wider than 32 bits take the default budget rules only");
    for (int i = 0; i < 2; ++i)
        if (o->reserved[i] != 0) return fail(HA_ERR_INVALID_ARG, "ha_select_opts.reserved must be zero");
    return HA_OK;
}

int code_words_of(const ha_select_opts* o) { return (o != nullptr && o->code_words > 1) ? o->code_words : 1; }

int nbins_of(const ha_select_opts* o) { return 32 * code_words_of(o) + 1; }

ha_status check_wide_codes(const ha_shape* s, const uint32_t* q_sig, const uint32_t* k_sig, int W) {
    if (q_sig == nullptr || k_sig == nullptr) return fail(HA_ERR_INVALID_ARG, "q_sig or k_sig is NULL");
    if (!aligned16(k_sig) || s->ks_sh % 4 != 0 || s->ks_sb % 4 != 0 || s->ks_sh < (int64_t)s->n_cap * W)
        return fail(HA_ERR_INVALID_ARG,
                    "wide k_sig rows must start on 16-byte boundaries and hold n_cap * code_words words");
    return HA_OK;
}

WideParams wide_params(const ha_shape* s, const Layout& lay, const Views& v, const uint32_t* q_sig,
                       const uint32_t* k_sig, const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m,
                       int32_t n_sink, int32_t n_local, int W) {
    WideParams p{};
    p.q_sig = q_sig;
    p.k_sig = k_sig;
    p.ks_sb = s->ks_sb;
    p.ks_sh = s->ks_sh;
    p.seq_lens = seq_lens;
    p.B = s->batch;
    p.Hq = s->h_q;
    p.Hkv = s->h_kv;
    p.G = s->h_q / s->h_kv;
    p.n_cap = s->n_cap;
    p.W = W;
    p.NB = 32 * W + 1;
    p.chunk = lay.chunk;
    p.nchunks = lay.nchunks;
    p.chunk_hist = v.chunk_hist;
    p.counters = v.counters;
    p.err = v.err;
    p.m_per_seq = m_per_seq;
    p.m = m;
    p.n_sink = n_sink;
    p.n_local = n_local;
    p.score_cnt = v.score_cnt;
    p.meta_t = v.meta_t;
    p.meta_qt = v.meta_qt;
    p.seg_cnt = v.seg_cnt;
    p.seg_idx = v.seg_idx;
    return p;
}

// The selection options into the SCORE/TOPK parameter blocks.
void apply_opts(const ha_select_opts* o, int32_t n_sink, int32_t n_local, ScoreParams* sp, SelectParams* tp) {
    sp->n_sink = n_sink;
    sp->n_local = n_local;
    sp->m_per_head = o ? o->m_per_head : nullptr;
    sp->excl = o ? o->exclusive_windows : 0;
    tp->excl = sp->excl;
}

// Parameters of the fused SCORE+TOPK kernels; the lists go to `list` (stride cap).
FusedSelParams fused_params(const ha_shape* s, const Layout& lay, void* ws, const Views& v, const uint32_t* q_sig,
                            const uint32_t* k_sig, const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m,
                            int32_t n_sink, int32_t n_local, const ha_select_opts* o, int32_t* list, int32_t* cnt,
                            int pad) {
    FusedSelParams p{};
    p.q_sig = q_sig;
    p.k_sig = k_sig;
    p.ks_sb = s->ks_sb;
    p.ks_sh = s->ks_sh;
    p.seq_lens = seq_lens;
    p.m_per_seq = m_per_seq;
    p.m_per_head = o ? o->m_per_head : nullptr;
    p.m = m;
    p.n_sink = n_sink;
    p.n_local = n_local;
    p.excl = o ? o->exclusive_windows : 0;
    p.B = s->batch;
    p.Hq = s->h_q;
    p.Hkv = s->h_kv;
    p.G = s->h_q / s->h_kv;
    p.kv_mul = 0u;
    p.n_cap = s->n_cap;
    p.nranges = lay.nranges;
    p.dist = at<uint32_t>(ws, lay.off_dist);
    p.d_sp = lay.d_sp;
    p.rh = at<uint32_t>(ws, lay.off_rh);
    p.arrive = v.score_cnt;
    p.meta_r = at<int4>(ws, lay.off_meta_r);
    p.meta_t = at<int2>(ws, lay.off_meta_tt);
    p.tot = at<uint32_t>(ws, lay.off_tot);
    p.list = list;
    p.cap = lay.rows_cap;
    p.cnt = cnt;
    p.pad = pad;
    p.err = v.err;
    return p;
}

// The tag of a call's selection ready flags: nonzero, different from the tags of
// the calls before it (a process-wide count; it wraps after 2^32 - 1 calls, long
// after any flag of an earlier call has been reset).
uint32_t next_call_tag() {
    static std::atomic<uint32_t> count{0};
    uint32_t t = count.fetch_add(1u, std::memory_order_relaxed) + 1u;
    if (t == 0u) t = count.fetch_add(1u, std::memory_order_relaxed) + 1u;
    return t;
}

// Query-head groups per KV head for the fused selection, the group kernel and the
// dense group path, which take at most kMaxHeadsPerPass query heads per KV head:
// with G = h_q / h_kv above that, each KV head's heads are split into k groups of
// G / k (the smallest such k; G itself when nothing smaller divides G), which run
// as k virtual KV heads that read the same codes and rows (kv_magic(k)). A grid so
// small that even twice its CTAs leave SMs idle splits groups of four heads once
// more, into two of two: twice the CTAs, each with half the masks and rows. Wider
// codes keep the two-kernel path, which takes any G (1).
int kv_split(const ha_shape& s, int code_words) {
    const int G = s.h_q / s.h_kv;
    if (code_words != 1) return 1;
    int k = G;
    for (int c = (G + kMaxHeadsPerPass - 1) / kMaxHeadsPerPass; c < G; ++c)
        if (G % c == 0) {
            k = c;
            break;
        }
    if (G <= kMaxHeadsPerPass) k = 1;
    if (G / k == kMaxHeadsPerPass && (int64_t)s.batch * s.h_kv * k * fused_ranges(s.n_cap) * 4 < kSMs) k *= 2;
    return k;
}

// The shape with k virtual KV heads per KV head (the strides stay those of the
// real heads; the kernels map a virtual head g to the real head g / k).
ha_shape virtual_shape(const ha_shape& s, int k) {
    ha_shape v = s;
    v.h_kv = s.h_kv * k;
    return v;
}

// The dense path runs on the group kernel for the shapes it takes (element
// strides of K/V rows below 2^30).
bool dense_group(const ha_shape& s) {
    return group_att_supported(s.d, s.kv_dtype == HA_BF16, s.q_dtype == HA_BF16, s.h_q / s.h_kv) &&
           s.k_sn < (int64_t(1) << 30) && s.v_sn < (int64_t(1) << 30);
}

// The group kernel's parameters on the dense path: the shape, the lengths and the
// error word; no codes, budgets or selection buffers.
FusedSelParams dense_sel_params(const ha_shape* s, const Views& v, const int32_t* seq_lens) {
    FusedSelParams p{};
    p.seq_lens = seq_lens;
    p.B = s->batch;
    p.Hq = s->h_q;
    p.Hkv = s->h_kv;
    p.G = s->h_q / s->h_kv;
    p.kv_mul = 0u;
    p.n_cap = s->n_cap;
    p.nranges = fused_ranges(s->n_cap);
    p.err = v.err;
    return p;
}

// The kernels a decode call runs (hash_attn_decode_path reports what decode_impl
// takes): the budget and options and whether the selection is returned. *kdiv:
// virtual KV heads per real one.
int decode_path(const ha_shape& s, int32_t m, const int32_t* m_per_seq, const ha_select_opts* opts, bool with_sel,
                int* kdiv) {
    const bool dense = (m >= s.n_cap) && (m_per_seq == nullptr) && (opts == nullptr || opts->m_per_head == nullptr);
    const int W = code_words_of(opts);
    // more than kMaxHeadsPerPass query heads per KV head: virtual KV heads
    *kdiv = kv_split(s, W);
    const ha_shape v = virtual_shape(s, *kdiv);
    if (dense) return dense_group(v) ? HA_PATH_DENSE_GROUP : HA_PATH_DENSE_HEADS;
    const bool fused = fused_selection(v, W);
    if (fused && !with_sel &&
        group_att_supported(v.d, v.kv_dtype == HA_BF16, v.q_dtype == HA_BF16, v.h_q / v.h_kv) &&
        v.k_sn < (int64_t(1) << 30) && v.v_sn < (int64_t(1) << 30))
        return HA_PATH_GROUP;
    return fused ? HA_PATH_FUSED_LISTS : HA_PATH_TWO_KERNEL;
}

// The signature map run ahead of SCORE (hash_attn_decode_mapped): the appended
// tokens' key codes (optional) and the step's query codes.
struct MapStep {
    EncodeParams queries, keys;
    bool mlp = false, with_keys = false;
};

ha_status decode_impl(const ha_shape* s, const void* q, const uint32_t* q_sig, const uint32_t* k_sig,
                      const void* K, const void* V, const int32_t* seq_lens, const int32_t* m_per_seq,
                      int32_t m, int32_t n_sink, int32_t n_local, const ha_select_opts* opts, float* out,
                      float* lse, int32_t* sel_idx, int32_t* sel_cnt, void* ws, size_t ws_bytes, void* stream,
                      void* const* events, const MapStep* map = nullptr, bool check_only = false) {
    HA_TRY(check_shape(s));
    HA_TRY(check_window(m, n_sink, n_local));
    HA_TRY(check_opts(opts));
    if (q == nullptr || seq_lens == nullptr || out == nullptr || lse == nullptr)
        return fail(HA_ERR_INVALID_ARG, "q, seq_lens, out and lse must not be NULL");
    HA_TRY(check_kv(s, K, V));
    int kdiv = 1;
    const int path = decode_path(*s, m, m_per_seq, opts, sel_idx != nullptr, &kdiv);
    const bool dense = path == HA_PATH_DENSE_GROUP || path == HA_PATH_DENSE_HEADS;
    const int W = code_words_of(opts);
    // with virtual KV heads the checks above ran on the caller's shape; strides and
    // pointers are the same
    const ha_shape vshape = virtual_shape(*s, kdiv);
    s = &vshape;
    if (!dense) HA_TRY(W > 1 ? check_wide_codes(s, q_sig, k_sig, W) : check_codes(s, q_sig, k_sig));
    if ((sel_idx == nullptr) != (sel_cnt == nullptr))
        return fail(HA_ERR_INVALID_ARG, "sel_idx and sel_cnt must both be given or both be NULL");
    const int64_t rows_cap = dense ? s->n_cap : rows_cap_of(s->n_cap, m, n_sink, n_local);
    const Layout lay = make_layout(*s, rows_cap, !dense, nbins_of(opts), W, dense);
    HA_TRY(check_segments(lay));
    HA_TRY(check_ws(lay, ws, ws_bytes));
    if (check_only) return HA_OK;
    const Views v = views(lay, ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int bhkv = s->batch * s->h_kv;
    const int heads = s->batch * s->h_q;
    if (map != nullptr) {  // every check has passed: nothing was enqueued before this point
        if (map->with_keys)
            HA_LAUNCH(map->mlp ? launch_encode_mlp(map->keys, st) : launch_encode(map->keys, st), "key map launch");
        HA_LAUNCH(map->mlp ? launch_encode_mlp(map->queries, st) : launch_encode(map->queries, st),
                  "query map launch");
    }

    GatherParams gp = gather_params(s, lay, v, q, K, V, seq_lens, out, lse);
    gp.kv_mul = kv_magic(kdiv);
    if (dense) {
        HA_TRY(record(events, 0, st));
        HA_TRY(record(events, 1, st));
        HA_TRY(record(events, 2, st));
        if (path == HA_PATH_DENSE_GROUP) {
            // one CTA per (batch entry, KV head, span of a range): each K/V row once
            // for the whole group
            GroupAttParams ga{};
            ga.sel = dense_sel_params(s, v, seq_lens);
            ga.sel.kv_mul = kv_magic(kdiv);
            ga.att = gp;
            ga.nsplit = group_dense_splits(bhkv, s->n_cap);
            HA_LAUNCH(launch_group_dense(ga, s->d, bhkv, st, true), "GATHER-ATT launch");
        } else {
            gp.mode = kIdentity;
            HA_LAUNCH(launch_gather(gp, s->d, s->kv_dtype == HA_BF16, st), "GATHER-ATT launch");
        }
        HA_TRY(record(events, 3, st));
        return HA_OK;
    }
    HA_TRY(record(events, 0, st));
    if (path == HA_PATH_GROUP) {
        // the scan's thresholds, then one kernel per GQA group that builds the masks
        // in place and attends over the union of the group's rows
        GroupAttParams ga{};
        ga.sel = fused_params(s, lay, ws, v, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink, n_local, opts, v.list,
                              v.lcnt, 0);
        ga.sel.kv_mul = kv_magic(kdiv);
        ga.sel.ready = at<uint32_t>(ws, lay.off_ready);
        ga.sel.epoch = next_call_tag();
        ga.att = gp;
        ga.nsplit = group_splits((int64_t)bhkv * lay.nranges);
        // the scan's counting may overlap the previous call's last kernel (not the
        // map kernels, whose codes it reads)
        HA_LAUNCH(launch_sel_scan(ga.sel, bhkv, st, false, map == nullptr), "SCORE+TOPK launch");
        HA_TRY(record(events, 1, st));
        HA_TRY(record(events, 2, st));
        HA_LAUNCH(launch_group_att(ga, s->d, bhkv, st, true), "GATHER-ATT launch");
        HA_TRY(record(events, 3, st));
        return HA_OK;
    }
    if (path == HA_PATH_FUSED_LISTS) {
        // SCORE and TOPK in one cluster kernel writing flat ascending lists: into the
        // caller's sel_idx (padded with -1) when given, else into the workspace
        const bool to_caller = sel_idx != nullptr;
        FusedSelParams cp = fused_params(s, lay, ws, v, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink, n_local, opts,
                                         to_caller ? sel_idx : v.list, to_caller ? sel_cnt : v.lcnt, to_caller ? 1 : 0);
        cp.kv_mul = kv_magic(kdiv);
        gp.mode = kList;
        gp.list_idx = cp.list;
        gp.list_cnt = cp.cnt;
        gp.list_cap = cp.cap;
        HA_LAUNCH(launch_select_fused(cp, bhkv, st), "SCORE+TOPK launch");
        HA_TRY(record(events, 1, st));
        HA_TRY(record(events, 2, st));
        // GATHER-ATT may start while the selection drains (it waits in the kernel)
        HA_LAUNCH(launch_gather(gp, s->d, s->kv_dtype == HA_BF16, st, true), "GATHER-ATT launch");
        HA_TRY(record(events, 3, st));
        return HA_OK;
    }
    if (W > 1) {
        const WideParams wp = wide_params(s, lay, v, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink, n_local, W);
        HA_LAUNCH(launch_score_wide(wp, bhkv, st), "SCORE launch");
        HA_TRY(record(events, 1, st));
        HA_LAUNCH(launch_select_wide(wp, bhkv, st, true), "TOPK launch");
    } else {
        ScoreParams sp = score_params(s, lay, v, q_sig, k_sig, seq_lens, m_per_seq, m, true);
        SelectParams tp = select_params(s, lay, v, q_sig, k_sig, seq_lens, n_sink, n_local);
        apply_opts(opts, n_sink, n_local, &sp, &tp);
        HA_LAUNCH(launch_score(sp, bhkv, st), "SCORE launch");
        HA_TRY(record(events, 1, st));
        // TOPK and GATHER-ATT may start while their predecessor drains (they wait in
        // the kernel before reading its output)
        HA_LAUNCH(launch_select(tp, bhkv, st, true), "TOPK launch");
    }
    HA_TRY(record(events, 2, st));
    gp.mode = kSegmented;
    HA_LAUNCH(launch_gather(gp, s->d, s->kv_dtype == HA_BF16, st, true), "GATHER-ATT launch");
    HA_TRY(record(events, 3, st));
    if (sel_idx != nullptr) {
        CompactParams cp{};
        cp.seq_lens = seq_lens;
        cp.Hq = s->h_q;
        cp.n_cap = s->n_cap;
        cp.seg_cap = lay.seg_cap;
        cp.nseg = lay.nseg;
        cp.cap = (int)rows_cap;
        cp.seg_cnt = v.seg_cnt;
        cp.seg_idx = v.seg_idx;
        cp.sel_idx = sel_idx;
        cp.sel_cnt = sel_cnt;
        cp.err = v.err;
        HA_LAUNCH(launch_compact(cp, heads, st), "compaction launch");
    }
    return HA_OK;
}

EncodeParams query_encode_params(const ha_shape* shape, const void* q, uint32_t* q_sig) {
    EncodeParams p{};
    p.x = q;
    p.x_bf16 = shape->q_dtype == HA_BF16;
    p.x_sb = shape->q_sb;
    p.x_sh = shape->q_sh;
    p.codes = q_sig;
    p.B = shape->batch;
    p.Hq = shape->h_q;
    p.Hkv = shape->h_kv;
    p.G = shape->h_q / shape->h_kv;
    p.d = shape->d;
    p.n_cap = shape->n_cap;
    p.keys = 0;
    return p;
}

EncodeParams key_encode_params(const ha_shape* shape, const void* K, const int32_t* pos, uint32_t* k_sig,
                               uint32_t* dev_flags) {
    EncodeParams p{};
    p.x = K;
    p.x_bf16 = shape->kv_dtype == HA_BF16;
    p.x_sb = shape->k_sb;
    p.x_sh = shape->k_sh;
    p.x_sn = shape->k_sn;
    p.codes = k_sig;
    p.c_sb = shape->ks_sb;
    p.c_sh = shape->ks_sh;
    p.pos = pos;
    p.flags = dev_flags;
    p.B = shape->batch;
    p.Hq = shape->h_q;
    p.Hkv = shape->h_kv;
    p.G = shape->h_q / shape->h_kv;
    p.d = shape->d;
    p.n_cap = shape->n_cap;
    p.keys = 1;
    return p;
}

ha_status check_mlp(const ha_mlp* mlp) {
    if (mlp->W1 == nullptr || mlp->b1 == nullptr || mlp->W2 == nullptr || mlp->b2 == nullptr ||
        mlp->W3 == nullptr || mlp->b3 == nullptr)
        return fail(HA_ERR_INVALID_ARG, "every MLP weight and bias must be given");
    if (mlp->hidden != 32 && mlp->hidden != 64 && mlp->hidden != 128)
        return fail(HA_ERR_UNSUPPORTED, "MLP hidden width must be 32, 64 or 128 (got %d)", mlp->hidden);
    if (!aligned16(mlp->W1) || !aligned16(mlp->W2) || !aligned16(mlp->W3))
        return fail(HA_ERR_INVALID_ARG, "MLP weight matrices must be 16-byte aligned");
    if (mlp->reserved != 0) return fail(HA_ERR_INVALID_ARG, "ha_mlp.reserved must be zero");
    return HA_OK;
}

void set_mlp(EncodeParams* p, const ha_mlp* mlp) {
    p->W1 = mlp->W1;
    p->b1 = mlp->b1;
    p->W2 = mlp->W2;
    p->b2 = mlp->b2;
    p->W3 = mlp->W3;
    p->b3 = mlp->b3;
    p->hidden = mlp->hidden;
}

// Device staging of hash_attn_decode_host: q, q_sig, seq_lens, m_per_seq (each
// 16-byte aligned, packed), then out (256-byte aligned) and lse (16-byte aligned):
// host buffers laid out the same way move in one copy each way.
struct Staging {
    size_t q = 0, q_sig = 0, seq = 0, mps = 0, out = 0, lse = 0, total = 0;
    size_t q_bytes = 0, sig_bytes = 0, seq_bytes = 0, out_bytes = 0, lse_bytes = 0;
};

Staging staging_layout(const ha_shape* s) {
    Staging L;
    const size_t heads = (size_t)s->batch * s->h_q;
    L.q_bytes = heads * s->d * (s->q_dtype == HA_F32 ? 4 : 2);
    L.sig_bytes = heads * sizeof(uint32_t);
    L.seq_bytes = (size_t)s->batch * sizeof(int32_t);
    L.out_bytes = heads * s->d * sizeof(float);
    L.lse_bytes = heads * sizeof(float);
    size_t off = 0;
    L.q = off;
    off = align_up(off + L.q_bytes, 16);
    L.q_sig = off;
    off = align_up(off + L.sig_bytes, 16);
    L.seq = off;
    off = align_up(off + L.seq_bytes, 16);
    L.mps = off;
    off = align_up(off + L.seq_bytes, 256);
    L.out = off;
    off = align_up(off + L.out_bytes, 16);
    L.lse = off;
    L.total = align_up(off + L.lse_bytes, 256);
    return L;
}

}  // namespace

// ---------------------------------------------------------------- layout policy

int choose_chunk(int64_t batch_hkv, int64_t n_cap) {
    // kScoreThreads * TPT with TPT in {32, 16, 8, 4} (the instantiated kernels)
    int chunk = kScoreThreads * 4;
    for (int tpt = 32; tpt > 4; tpt >>= 1)
        if (batch_hkv * ceil_div(n_cap, (int64_t)kScoreThreads * tpt) >= kTargetCtas) {
            chunk = kScoreThreads * tpt;
            break;
        }
    // a long single sequence: larger chunks keep the segments per head within
    // GATHER-ATT's prefix table
    while (chunk < kScoreThreads * 32 && ceil_div(n_cap, chunk) * kSegPerChunk > kMaxSegments) chunk *= 2;
    return chunk;
}

bool fused_selection(const ha_shape& s, int code_words) {
    return code_words <= 1 && s.h_q / s.h_kv <= kMaxHeadsPerPass;
}

void choose_splits(int64_t heads, int64_t rows_cap, int* splits, int* rows_per_split) {
    if (rows_cap <= 0) {
        *splits = 1;
        *rows_per_split = kTileRows;
        return;
    }
    int64_t sp = ceil_div(rows_cap, 1024);
    const int64_t fill = ceil_div(kTargetCtas, heads);       // enough CTAs for small batches
    if (fill > sp) sp = fill;
    const int64_t most = ceil_div(rows_cap, 2 * kTileRows);  // at least two tiles per CTA
    if (sp > most) sp = most;
    if (sp < 1) sp = 1;
    int64_t rps = ceil_div(ceil_div(rows_cap, sp), kTileRows) * kTileRows;
    sp = ceil_div(rows_cap, rps);
    *splits = (int)sp;
    *rows_per_split = (int)rps;
}

Layout make_layout(const ha_shape& s, int64_t rows_cap, bool with_selection, int nbins, int code_words,
                   bool dense_parts) {
    Layout L;
    L.heads = s.batch * s.h_q;
    L.rows_cap = (int)rows_cap;
    choose_splits(L.heads, rows_cap, &L.splits, &L.rows_per_split);
    size_t off = 256;  // error word + padding
    L.off_err = 0;
    // What must be zero between calls comes first, at offsets that depend on the
    // shape alone: calls with other budgets, code widths or options, the dense
    // path and the entry points with given lists lay out the scratch after it
    // differently, so one workspace serves all of them in turn.
    const int64_t pairs = (int64_t)s.batch * s.h_kv;
    L.off_counter = off;  // GATHER-ATT split-K arrival counters, per head
    off = align_up(off + (size_t)L.heads * 4, 256);
    L.off_scnt = off;     // SCORE arrival counters, per (batch entry, KV head)
    off = align_up(off + (size_t)pairs * 4, 256);
    L.off_tot = off;      // fused: per (pair, head) 36-word distance histogram
    off = align_up(off + (size_t)pairs * 4 * 36 * 4, 256);
    L.off_ready = off;    // fused: per pair, shares-complete flag
    off = align_up(off + (size_t)pairs * 4, 256);
    // scratch: written by every call before it reads it
    if (with_selection) {
        L.chunk = choose_chunk(pairs, s.n_cap);
        L.nchunks = (int)ceil_div(s.n_cap, L.chunk);
        L.seg_cap = L.chunk / kSegPerChunk;
        L.nseg = L.nchunks * kSegPerChunk;
        L.nbins = nbins;
        L.off_meta_t = off;
        off = align_up(off + (size_t)L.heads * 4, 256);
        L.off_meta_qt = off;
        off = align_up(off + (size_t)L.heads * L.nchunks * 8, 256);
        L.off_hist = off;
        off = align_up(off + (size_t)L.heads * L.nchunks * nbins * 4, 256);
        if (fused_selection(s, code_words)) {
            L.fused = true;
            L.nranges = fused_ranges(s.n_cap);
            L.d_sp = ceil_div(s.n_cap, 64) * 64;
            L.off_list = off;
            off = align_up(off + (size_t)L.heads * (size_t)rows_cap * 4, 256);
            L.off_lcnt = off;
            off = align_up(off + (size_t)L.heads * 4, 256);
            L.off_dist = off;
            off = align_up(off + (size_t)pairs * (size_t)L.d_sp * 4, 256);
            L.off_rh = off;
            off = align_up(off + (size_t)pairs * L.nranges * 3 * 4 * 36 * 4, 256);
            L.off_meta_r = off;
            off = align_up(off + (size_t)pairs * L.nranges * 4 * 16, 256);
            L.off_meta_tt = off;
            off = align_up(off + (size_t)pairs * 4 * 8, 256);
        } else {
            L.off_segcnt = off;
            off = align_up(off + (size_t)L.heads * L.nseg * 4, 256);
            L.off_seg = off;
            off = align_up(off + (size_t)L.heads * L.nseg * L.seg_cap * 4, 256);
        }
    }
    // split-K partials; the group kernel keeps one per (head, range, split) of the
    // fused plan, or per (head, range, span) on the dense path
    int64_t psplits = L.splits;
    if (L.fused) psplits = std::max<int64_t>(psplits, (int64_t)L.nranges * group_splits(pairs * L.nranges));
    if (dense_parts && dense_group(s))
        psplits = std::max<int64_t>(psplits, (int64_t)fused_ranges(s.n_cap) * group_dense_splits(pairs, s.n_cap));
    L.off_part = off;
    off = align_up(off + (size_t)L.heads * psplits * (s.d + 2) * 4, 256);
    L.total = off;
    return L;
}

// The layout a workspace is sized for: the largest that a call on this shape makes
// (the decode on virtual KV heads when G exceeds kMaxHeadsPerPass, the selection
// and SCORE entry points on the caller's shape, whose two-kernel path takes any G).
Layout workspace_layout(const ha_shape& s, int64_t rows_cap, int nbins, int code_words, bool dense) {
    const int k = kv_split(s, code_words);
    Layout L = make_layout(virtual_shape(s, k), rows_cap, true, nbins, code_words, dense);
    if (k > 1) {
        const Layout r = make_layout(s, rows_cap, true, nbins, code_words, dense);
        L.total = std::max(L.total, r.total);
    }
    return L;
}

}  // namespace ha

using namespace ha;

extern "C" {

ha_status hash_attn_workspace_size(const ha_shape* shape, int32_t m_max, int32_t n_sink, int32_t n_local,
                                   size_t* bytes) {
    HA_TRY(check_shape(shape));
    HA_TRY(check_window(m_max, n_sink, n_local));
    if (bytes == nullptr) return fail(HA_ERR_INVALID_ARG, "bytes is NULL");
    const bool dense = m_max >= shape->n_cap;
    // the selection regions are always included so that hash_attn_select and
    // hash_attn_score work with any budget on the same workspace
    const int64_t rows_cap = dense ? shape->n_cap : rows_cap_of(shape->n_cap, m_max, n_sink, n_local);
    const Layout sparse = workspace_layout(*shape, rows_cap, HA_NBINS, 1, dense);
    HA_TRY(check_segments(sparse));
    *bytes = sparse.total;
    return HA_OK;
}

ha_status hash_attn_workspace_size_ex(const ha_shape* shape, int32_t m_max, int32_t n_sink, int32_t n_local,
                                      const ha_select_opts* opts, size_t* bytes) {
    HA_TRY(check_shape(shape));
    HA_TRY(check_window(m_max, n_sink, n_local));
    HA_TRY(check_opts(opts));
    if (bytes == nullptr) return fail(HA_ERR_INVALID_ARG, "bytes is NULL");
    const bool dense = m_max >= shape->n_cap;
    const int64_t rows_cap = dense ? shape->n_cap : rows_cap_of(shape->n_cap, m_max, n_sink, n_local);
    const Layout sparse = workspace_layout(*shape, rows_cap, nbins_of(opts), code_words_of(opts), dense);
    HA_TRY(check_segments(sparse));
    *bytes = sparse.total;
    return HA_OK;
}

ha_status hash_attn_selection_plan(const ha_shape* shape, int32_t code_words, int32_t* fused, int32_t* ranges,
                                   int32_t* range, int32_t* chunk) {
    HA_TRY(check_shape(shape));
    if (code_words != 1 && code_words != 2 && code_words != 4 && code_words != 8 && code_words != 16)
        return fail(HA_ERR_UNSUPPORTED, "code_words must be 1, 2, 4, 8 or 16 (got %d)", code_words);
    const bool f = fused_selection(virtual_shape(*shape, kv_split(*shape, code_words)), code_words);
    if (fused) *fused = f ? 1 : 0;
    if (ranges) *ranges = f ? fused_ranges(shape->n_cap) : 0;
    if (range) *range = f ? 8192 : 0;
    if (chunk) *chunk = choose_chunk((int64_t)shape->batch * shape->h_kv, shape->n_cap);
    return HA_OK;
}

ha_status hash_attn_decode_path(const ha_shape* shape, int32_t m, const int32_t* m_per_seq,
                                const ha_select_opts* opts, int32_t with_selection, int32_t* path) {
    HA_TRY(check_shape(shape));
    HA_TRY(check_opts(opts));
    if (m < 0) return fail(HA_ERR_INVALID_ARG, "m must be >= 0 (got %d)", m);
    if (path == nullptr) return fail(HA_ERR_INVALID_ARG, "path is NULL");
    int kdiv = 1;
    *path = decode_path(*shape, m, m_per_seq, opts, with_selection != 0, &kdiv);
    return HA_OK;
}

ha_status hash_attn_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
    if (workspace == nullptr) return fail(HA_ERR_WORKSPACE, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(HA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    const cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HA_OK : cuda_fail(e, "cudaMemsetAsync");
}

int32_t hash_attn_select_capacity(int32_t n_cap, int32_t m, int32_t n_sink, int32_t n_local) {
    if (n_cap < 0 || m < 0 || n_sink < 0 || n_local < 0) return 0;
    return (int32_t)rows_cap_of(n_cap, m, n_sink, n_local);
}

ha_status hash_attn_decode(const ha_shape* shape, const void* q, const uint32_t* q_sig, const uint32_t* k_sig,
                           const void* K, const void* V, const int32_t* seq_lens, const int32_t* m_per_seq,
                           int32_t m, int32_t n_sink, int32_t n_local, float* out, float* lse, int32_t* sel_idx,
                           int32_t* sel_cnt, void* workspace, size_t ws_bytes, void* stream) {
    return decode_impl(shape, q, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local, nullptr, out, lse,
                       sel_idx, sel_cnt, workspace, ws_bytes, stream, nullptr);
}

ha_status hash_attn_decode_ex(const ha_shape* shape, const void* q, const uint32_t* q_sig, const uint32_t* k_sig,
                              const void* K, const void* V, const int32_t* seq_lens, const int32_t* m_per_seq,
                              int32_t m, int32_t n_sink, int32_t n_local, const ha_select_opts* opts, float* out,
                              float* lse, int32_t* sel_idx, int32_t* sel_cnt, void* workspace, size_t ws_bytes,
                              void* stream) {
    return decode_impl(shape, q, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local, opts, out, lse,
                       sel_idx, sel_cnt, workspace, ws_bytes, stream, nullptr);
}

ha_status hash_attn_decode_timed(const ha_shape* shape, const void* q, const uint32_t* q_sig,
                                 const uint32_t* k_sig, const void* K, const void* V, const int32_t* seq_lens,
                                 const int32_t* m_per_seq, int32_t m, int32_t n_sink, int32_t n_local, float* out,
                                 float* lse, int32_t* sel_idx, int32_t* sel_cnt, void* workspace, size_t ws_bytes,
                                 void* stream, void* const* events) {
    if (events == nullptr) return fail(HA_ERR_INVALID_ARG, "events is NULL");
    for (int i = 0; i < 4; ++i)
        if (events[i] == nullptr) return fail(HA_ERR_INVALID_ARG, "events[%d] is NULL", i);
    return decode_impl(shape, q, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local, nullptr, out, lse,
                       sel_idx, sel_cnt, workspace, ws_bytes, stream, events);
}

ha_status hash_attn_score(const ha_shape* shape, const uint32_t* q_sig, const uint32_t* k_sig,
                          const int32_t* seq_lens, uint8_t* dist, uint32_t* hist, void* workspace,
                          size_t ws_bytes, void* stream) {
    HA_TRY(check_shape(shape));
    HA_TRY(check_codes(shape, q_sig, k_sig));
    if (seq_lens == nullptr) return fail(HA_ERR_INVALID_ARG, "seq_lens is NULL");
    if (dist == nullptr && hist == nullptr) return fail(HA_ERR_INVALID_ARG, "dist and hist are both NULL");
    const Layout lay = make_layout(*shape, 0, true);
    HA_TRY(check_segments(lay));
    HA_TRY(check_ws(lay, workspace, ws_bytes));
    const Views v = views(lay, workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ScoreParams sp = score_params(shape, lay, v, q_sig, k_sig, seq_lens, nullptr, 0, false);
    sp.counters = nullptr;
    sp.dist = dist;
    HA_LAUNCH(launch_score(sp, shape->batch * shape->h_kv, st), "SCORE launch");
    if (hist != nullptr) {
        HistParams hp{};
        hp.seq_lens = seq_lens;
        hp.Hq = shape->h_q;
        hp.n_cap = shape->n_cap;
        hp.chunk = lay.chunk;
        hp.nchunks = lay.nchunks;
        hp.chunk_hist = v.chunk_hist;
        hp.hist = hist;
        HA_LAUNCH(launch_hist(hp, shape->batch * shape->h_q, st), "histogram launch");
    }
    return HA_OK;
}

ha_status hash_attn_select_ex(const ha_shape* shape, const uint32_t* q_sig, const uint32_t* k_sig,
                              const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m, int32_t n_sink,
                              int32_t n_local, const ha_select_opts* opts, int32_t* sel_idx, int32_t* sel_cnt,
                              void* workspace, size_t ws_bytes, void* stream) {
    HA_TRY(check_shape(shape));
    HA_TRY(check_window(m, n_sink, n_local));
    HA_TRY(check_opts(opts));
    const int W = code_words_of(opts);
    HA_TRY(W > 1 ? check_wide_codes(shape, q_sig, k_sig, W) : check_codes(shape, q_sig, k_sig));
    if (seq_lens == nullptr || sel_idx == nullptr || sel_cnt == nullptr)
        return fail(HA_ERR_INVALID_ARG, "seq_lens, sel_idx and sel_cnt must not be NULL");
    const int64_t rows_cap = rows_cap_of(shape->n_cap, m, n_sink, n_local);
    const Layout lay = make_layout(*shape, rows_cap, true, nbins_of(opts), W);
    HA_TRY(check_segments(lay));
    HA_TRY(check_ws(lay, workspace, ws_bytes));
    const Views v = views(lay, workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int bhkv = shape->batch * shape->h_kv;
    if (lay.fused) {
        const FusedSelParams cp = fused_params(shape, lay, workspace, v, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink,
                                               n_local, opts, sel_idx, sel_cnt, 1);
        HA_LAUNCH(launch_select_fused(cp, bhkv, st), "SCORE+TOPK launch");
        return HA_OK;
    }
    if (W > 1) {
        const WideParams wp = wide_params(shape, lay, v, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink, n_local, W);
        HA_LAUNCH(launch_score_wide(wp, bhkv, st), "SCORE launch");
        HA_LAUNCH(launch_select_wide(wp, bhkv, st, false), "TOPK launch");
    } else {
        ScoreParams sp = score_params(shape, lay, v, q_sig, k_sig, seq_lens, m_per_seq, m, true);
        SelectParams tp = select_params(shape, lay, v, q_sig, k_sig, seq_lens, n_sink, n_local);
        apply_opts(opts, n_sink, n_local, &sp, &tp);
        HA_LAUNCH(launch_score(sp, bhkv, st), "SCORE launch");
        HA_LAUNCH(launch_select(tp, bhkv, st), "TOPK launch");
    }
    CompactParams cp{};
    cp.seq_lens = seq_lens;
    cp.Hq = shape->h_q;
    cp.n_cap = shape->n_cap;
    cp.seg_cap = lay.seg_cap;
    cp.nseg = lay.nseg;
    cp.cap = (int)rows_cap;
    cp.seg_cnt = v.seg_cnt;
    cp.seg_idx = v.seg_idx;
    cp.sel_idx = sel_idx;
    cp.sel_cnt = sel_cnt;
    cp.err = v.err;
    HA_LAUNCH(launch_compact(cp, shape->batch * shape->h_q, st), "compaction launch");
    return HA_OK;
}

ha_status hash_attn_select(const ha_shape* shape, const uint32_t* q_sig, const uint32_t* k_sig,
                           const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m, int32_t n_sink,
                           int32_t n_local, int32_t* sel_idx, int32_t* sel_cnt, void* workspace, size_t ws_bytes,
                           void* stream) {
    return hash_attn_select_ex(shape, q_sig, k_sig, seq_lens, m_per_seq, m, n_sink, n_local, nullptr, sel_idx,
                               sel_cnt, workspace, ws_bytes, stream);
}

ha_status hash_attn_gather_att(const ha_shape* shape, const void* q, const void* K, const void* V,
                               const int32_t* seq_lens, const int32_t* idx, int32_t idx_cap, const int32_t* cnt,
                               float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
    HA_TRY(check_shape(shape));
    if (q == nullptr || seq_lens == nullptr || out == nullptr || lse == nullptr || cnt == nullptr)
        return fail(HA_ERR_INVALID_ARG, "q, seq_lens, cnt, out and lse must not be NULL");
    if (idx_cap < 0 || idx_cap > shape->n_cap)
        return fail(HA_ERR_INVALID_ARG, "idx_cap must be in [0, n_cap] (got %d)", idx_cap);
    if (idx == nullptr && idx_cap > 0) return fail(HA_ERR_INVALID_ARG, "idx is NULL");
    HA_TRY(check_kv(shape, K, V));
    const Layout lay = make_layout(*shape, idx_cap, false);
    HA_TRY(check_ws(lay, workspace, ws_bytes));
    const Views v = views(lay, workspace);
    GatherParams gp = gather_params(shape, lay, v, q, K, V, seq_lens, out, lse);
    gp.mode = kList;
    gp.list_idx = idx;
    gp.list_cnt = cnt;
    gp.list_cap = idx_cap;
    HA_LAUNCH(launch_gather(gp, shape->d, shape->kv_dtype == HA_BF16, static_cast<cudaStream_t>(stream)),
              "GATHER-ATT launch");
    return HA_OK;
}

ha_status hash_attn_merge(const float* out_a, const float* lse_a, const float* out_b, const float* lse_b,
                          float* out, float* lse, int32_t rows, int32_t d, void* stream) {
    if (rows < 0 || d < 1) return fail(HA_ERR_INVALID_ARG, "rows must be >= 0 and d >= 1");
    if (rows == 0) return HA_OK;
    if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse)
        return fail(HA_ERR_INVALID_ARG, "merge pointers must not be NULL");
    MergeParams p{out_a, lse_a, out_b, lse_b, out, lse, rows, d};
    HA_LAUNCH(launch_merge(p, static_cast<cudaStream_t>(stream)), "merge launch");
    return HA_OK;
}

ha_status hash_attn_merge_n(const float* outs, int64_t out_seg_stride, const float* lses, int64_t lse_seg_stride,
                            int32_t nseg, float* out, float* lse, int32_t rows, int32_t d, void* stream) {
    if (nseg < 1 || rows < 0 || d < 1) return fail(HA_ERR_INVALID_ARG, "nseg must be >= 1, rows >= 0 and d >= 1");
    if (rows == 0) return HA_OK;
    if (!outs || !lses || !out || !lse) return fail(HA_ERR_INVALID_ARG, "merge pointers must not be NULL");
    if (nseg > 1 && (out_seg_stride < (int64_t)rows * d || lse_seg_stride < rows))
        return fail(HA_ERR_INVALID_ARG, "segment strides overlap (out %lld < %lld or lse %lld < %d)",
                    (long long)out_seg_stride, (long long)rows * d, (long long)lse_seg_stride, rows);
    MergeNParams p{outs, out_seg_stride, lses, lse_seg_stride, nseg, out, lse, rows, d};
    HA_LAUNCH(launch_merge_n(p, static_cast<cudaStream_t>(stream)), "merge launch");
    return HA_OK;
}

ha_status hash_attn_encode_queries(const ha_shape* shape, const void* q, const float* W, uint32_t* q_sig,
                                   void* stream) {
    HA_TRY(check_shape(shape));
    if (q == nullptr || W == nullptr || q_sig == nullptr)
        return fail(HA_ERR_INVALID_ARG, "q, W and q_sig must not be NULL");
    EncodeParams p = query_encode_params(shape, q, q_sig);
    p.W = W;
    HA_LAUNCH(launch_encode(p, static_cast<cudaStream_t>(stream)), "query encode launch");
    return HA_OK;
}

ha_status hash_attn_encode_keys(const ha_shape* shape, const void* K, const float* W, const int32_t* pos,
                                uint32_t* k_sig, uint32_t* dev_flags, void* stream) {
    HA_TRY(check_shape(shape));
    if (K == nullptr || W == nullptr || pos == nullptr || k_sig == nullptr)
        return fail(HA_ERR_INVALID_ARG, "K, W, pos and k_sig must not be NULL");
    EncodeParams p = key_encode_params(shape, K, pos, k_sig, dev_flags);
    p.W = W;
    HA_LAUNCH(launch_encode(p, static_cast<cudaStream_t>(stream)), "key encode launch");
    return HA_OK;
}

ha_status hash_attn_encode_queries_mlp(const ha_shape* shape, const void* q, const ha_mlp* mlp, uint32_t* q_sig,
                                       void* stream) {
    HA_TRY(check_shape(shape));
    if (q == nullptr || mlp == nullptr || q_sig == nullptr)
        return fail(HA_ERR_INVALID_ARG, "q, mlp and q_sig must not be NULL");
    HA_TRY(check_mlp(mlp));
    EncodeParams p = query_encode_params(shape, q, q_sig);
    set_mlp(&p, mlp);
    HA_LAUNCH(launch_encode_mlp(p, static_cast<cudaStream_t>(stream)), "query MLP encode launch");
    return HA_OK;
}

ha_status hash_attn_encode_keys_mlp(const ha_shape* shape, const void* K, const ha_mlp* mlp, const int32_t* pos,
                                    uint32_t* k_sig, uint32_t* dev_flags, void* stream) {
    HA_TRY(check_shape(shape));
    if (K == nullptr || mlp == nullptr || pos == nullptr || k_sig == nullptr)
        return fail(HA_ERR_INVALID_ARG, "K, mlp, pos and k_sig must not be NULL");
    HA_TRY(check_mlp(mlp));
    EncodeParams p = key_encode_params(shape, K, pos, k_sig, dev_flags);
    set_mlp(&p, mlp);
    HA_LAUNCH(launch_encode_mlp(p, static_cast<cudaStream_t>(stream)), "key MLP encode launch");
    return HA_OK;
}

ha_status hash_attn_host_staging_size(const ha_shape* shape, size_t* bytes) {
    HA_TRY(check_shape(shape));
    if (bytes == nullptr) return fail(HA_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = staging_layout(shape).total;
    return HA_OK;
}

ha_status hash_attn_decode_host(const ha_shape* shape, const void* q_host, const uint32_t* q_sig_host,
                                const int32_t* seq_lens_host, const int32_t* m_per_seq_host, const uint32_t* k_sig,
                                const void* K, const void* V, int32_t m, int32_t n_sink, int32_t n_local,
                                float* out_host, float* lse_host, void* staging, size_t staging_bytes,
                                void* workspace, size_t ws_bytes, void* stream) {
    HA_TRY(check_shape(shape));
    if (q_host == nullptr || seq_lens_host == nullptr || out_host == nullptr || lse_host == nullptr)
        return fail(HA_ERR_INVALID_ARG, "q_host, seq_lens_host, out_host and lse_host must not be NULL");
    const Staging L = staging_layout(shape);
    if (staging == nullptr || (reinterpret_cast<uintptr_t>(staging) & 255u) != 0 || staging_bytes < L.total)
        return fail(HA_ERR_WORKSPACE, "staging must be 256-byte aligned and hold %zu bytes", L.total);
    ha_shape s = *shape;  // the staged q is contiguous
    s.q_sh = shape->d;
    s.q_sb = (int64_t)shape->h_q * shape->d;
    char* sb = static_cast<char*>(staging);
    void* q_d = sb + L.q;
    uint32_t* sig_d = q_sig_host != nullptr ? reinterpret_cast<uint32_t*>(sb + L.q_sig) : nullptr;
    int32_t* seq_d = reinterpret_cast<int32_t*>(sb + L.seq);
    int32_t* mps_d = m_per_seq_host != nullptr ? reinterpret_cast<int32_t*>(sb + L.mps) : nullptr;
    float* out_d = reinterpret_cast<float*>(sb + L.out);
    float* lse_d = reinterpret_cast<float*>(sb + L.lse);
    // every check of the decode runs before the first copy is enqueued
    HA_TRY(decode_impl(&s, q_d, sig_d, k_sig, K, V, seq_d, mps_d, m, n_sink, n_local, nullptr, out_d, lse_d,
                       nullptr, nullptr, workspace, ws_bytes, stream, nullptr, nullptr, true));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    struct Copy {
        void* dst;
        const void* src;
        size_t bytes;
        cudaMemcpyKind kind;
    };
    const Copy in[4] = {{q_d, q_host, L.q_bytes, cudaMemcpyHostToDevice},
                        {sig_d, q_sig_host, L.sig_bytes, cudaMemcpyHostToDevice},
                        {seq_d, seq_lens_host, L.seq_bytes, cudaMemcpyHostToDevice},
                        {mps_d, m_per_seq_host, L.seq_bytes, cudaMemcpyHostToDevice}};
    // one asynchronous copy per run of inputs that are adjacent both on the host and
    // in the staging buffer (an input following the previous one directly in both)
    const Copy* run = nullptr;
    size_t run_bytes = 0;
    auto flush = [&]() -> ha_status {
        if (run == nullptr) return HA_OK;
        const cudaError_t e = cudaMemcpyAsync(run->dst, run->src, run_bytes, cudaMemcpyHostToDevice, st);
        run = nullptr;
        return e == cudaSuccess ? HA_OK : cuda_fail(e, "input copy to the device");
    };
    for (const Copy& c : in) {
        if (c.dst == nullptr) continue;
        if (run != nullptr && static_cast<const char*>(run->src) + run_bytes == static_cast<const char*>(c.src) &&
            static_cast<char*>(run->dst) + run_bytes == static_cast<char*>(c.dst)) {
            run_bytes += c.bytes;
            continue;
        }
        HA_TRY(flush());
        run = &c;
        run_bytes = c.bytes;
    }
    HA_TRY(flush());
    HA_TRY(decode_impl(&s, q_d, sig_d, k_sig, K, V, seq_d, mps_d, m, n_sink, n_local, nullptr, out_d, lse_d,
                       nullptr, nullptr, workspace, ws_bytes, stream, nullptr));
    cudaError_t e;
    if (reinterpret_cast<char*>(out_host) + L.out_bytes == reinterpret_cast<char*>(lse_host) &&
        L.out + L.out_bytes == L.lse) {
        e = cudaMemcpyAsync(out_host, out_d, L.out_bytes + L.lse_bytes, cudaMemcpyDeviceToHost, st);
    } else {
        e = cudaMemcpyAsync(out_host, out_d, L.out_bytes, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(lse_host, lse_d, L.lse_bytes, cudaMemcpyDeviceToHost, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "result copy to the host");
    return HA_OK;
}

ha_status hash_attn_decode_mapped(const ha_shape* shape, const void* q, const ha_map* map, const int32_t* pos,
                                  uint32_t* q_sig, uint32_t* k_sig, const void* K, const void* V,
                                  const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m, int32_t n_sink,
                                  int32_t n_local, const ha_select_opts* opts, float* out, float* lse,
                                  int32_t* sel_idx, int32_t* sel_cnt, void* workspace, size_t ws_bytes,
                                  uint32_t* dev_flags, void* stream) {
    HA_TRY(check_shape(shape));
    HA_TRY(check_opts(opts));
    if (map == nullptr || (map->W == nullptr) == (map->mlp == nullptr))
        return fail(HA_ERR_INVALID_ARG, "exactly one of map->W and map->mlp must be given");
    if (map->mlp != nullptr) HA_TRY(check_mlp(map->mlp));
    if (code_words_of(opts) > 1)
        return fail(HA_ERR_UNSUPPORTED, "the map writes 32-bit codes (opts->code_words must be 0 or 1)");
    HA_TRY(check_codes(shape, q_sig, k_sig));
    if (q == nullptr || K == nullptr) return fail(HA_ERR_INVALID_ARG, "q and K must not be NULL");
    MapStep ms;
    ms.mlp = map->mlp != nullptr;
    ms.with_keys = pos != nullptr;
    ms.queries = query_encode_params(shape, q, q_sig);
    ms.keys = key_encode_params(shape, K, pos, k_sig, dev_flags);
    if (ms.mlp) {
        set_mlp(&ms.queries, map->mlp);
        set_mlp(&ms.keys, map->mlp);
    } else {
        ms.queries.W = map->W;
        ms.keys.W = map->W;
    }
    return decode_impl(shape, q, q_sig, k_sig, K, V, seq_lens, m_per_seq, m, n_sink, n_local, opts, out, lse,
                       sel_idx, sel_cnt, workspace, ws_bytes, stream, nullptr, &ms);
}

ha_status hash_attn_topk_exact_workspace_size(const ha_shape* shape, size_t* bytes) {
    HA_TRY(check_shape(shape));
    if (bytes == nullptr) return fail(HA_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = 256 + align_up((size_t)shape->batch * shape->h_q * (size_t)shape->n_cap * sizeof(float), 1024) +
             (size_t)shape->batch * shape->h_kv * 64 * (size_t)shape->d * sizeof(uint16_t);
    return HA_OK;
}

ha_status hash_attn_topk_exact(const ha_shape* shape, const void* q, const void* K, const int32_t* seq_lens,
                               int32_t m, int32_t* idx, int32_t idx_cap, int32_t* cnt, void* workspace,
                               size_t ws_bytes, void* stream) {
    return hash_attn_topk_exact_timed(shape, q, K, seq_lens, m, idx, idx_cap, cnt, workspace, ws_bytes, stream,
                                      nullptr);
}

ha_status hash_attn_topk_exact_timed(const ha_shape* shape, const void* q, const void* K, const int32_t* seq_lens,
                                     int32_t m, int32_t* idx, int32_t idx_cap, int32_t* cnt, void* workspace,
                                     size_t ws_bytes, void* stream, void* const* events) {
    HA_TRY(check_shape(shape));
    if (q == nullptr || seq_lens == nullptr || idx == nullptr || cnt == nullptr)
        return fail(HA_ERR_INVALID_ARG, "q, seq_lens, idx and cnt must not be NULL");
    HA_TRY(check_kv(shape, K, K));
    if (m < 0) return fail(HA_ERR_INVALID_ARG, "m must be >= 0 (got %d)", m);
    const int32_t need = m < shape->n_cap ? m : shape->n_cap;
    if (idx_cap < need || idx_cap > shape->n_cap)
        return fail(HA_ERR_INVALID_ARG, "idx_cap must be in [min(m, n_cap), n_cap] (got %d)", idx_cap);
    size_t nbytes = 0;
    HA_TRY(hash_attn_topk_exact_workspace_size(shape, &nbytes));
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < nbytes)
        return fail(HA_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", nbytes);
    ExactParams p{};
    p.q = q;
    p.q_sb = shape->q_sb;
    p.q_sh = shape->q_sh;
    p.q_bf16 = shape->q_dtype == HA_BF16;
    p.K = static_cast<const char*>(K);
    p.k_sb = shape->k_sb;
    p.k_sh = shape->k_sh;
    p.k_sn = shape->k_sn;
    p.seq_lens = seq_lens;
    p.B = shape->batch;
    p.Hq = shape->h_q;
    p.Hkv = shape->h_kv;
    p.G = shape->h_q / shape->h_kv;
    p.n_cap = shape->n_cap;
    p.m = m;
    p.err = static_cast<uint32_t*>(workspace);
    p.scores = reinterpret_cast<float*>(static_cast<char*>(workspace) + 256);
    p.qt = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + 256 +
                                       align_up((size_t)shape->batch * shape->h_q * (size_t)shape->n_cap * sizeof(float), 1024));
    p.idx = idx;
    p.idx_cap = idx_cap;
    p.cnt = cnt;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (events != nullptr)
        for (int i = 0; i < 3; ++i)
            if (events[i] == nullptr) return fail(HA_ERR_INVALID_ARG, "events[%d] is NULL", i);
    // every call starts with a clean error word (the rest of the workspace is scratch)
    const cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
    HA_TRY(record(events, 0, st));
    HA_LAUNCH(launch_exact_scores(p, shape->d, shape->kv_dtype == HA_BF16, st), "exact score launch");
    HA_TRY(record(events, 1, st));
    HA_LAUNCH(launch_exact_topm(p, st), "exact top-m launch");
    HA_TRY(record(events, 2, st));
    return HA_OK;
}

ha_status hash_attn_recall(const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_cap, const int32_t* ref_idx,
                           const int32_t* ref_cnt, int32_t ref_cap, int32_t heads, float* recall, void* stream) {
    if (heads < 0 || sel_cap < 0 || ref_cap < 0) return fail(HA_ERR_INVALID_ARG, "heads and caps must be >= 0");
    if (heads == 0) return HA_OK;
    if (!sel_cnt || !ref_cnt || !recall || (!sel_idx && sel_cap > 0) || (!ref_idx && ref_cap > 0))
        return fail(HA_ERR_INVALID_ARG, "recall pointers must not be NULL");
    RecallParams p{sel_idx, sel_cnt, sel_cap, ref_idx, ref_cnt, ref_cap, heads, recall};
    HA_LAUNCH(launch_recall(p, static_cast<cudaStream_t>(stream)), "recall launch");
    return HA_OK;
}

ha_status hash_attn_device_status(void* workspace, void* stream, uint32_t* flags) {
    if (workspace == nullptr) return fail(HA_ERR_WORKSPACE, "workspace is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
    if (word != 0) {
        e = cudaMemsetAsync(workspace, 0, sizeof(word), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
    }
    if (flags) *flags = word;
    if (word == 0) return HA_OK;
    if (word & HA_DEVERR_TIMEOUT) return fail(HA_ERR_TIMEOUT, "device error word 0x%x (wait timed out)", word);
    return fail(HA_ERR_DEVICE, "device error word 0x%x", word);
}

const char* hash_attn_status_string(ha_status status) {
    switch (status) {
        case HA_OK: return "ok";
        case HA_ERR_INVALID_ARG: return "invalid argument";
        case HA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case HA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case HA_ERR_CUDA: return "CUDA error";
        case HA_ERR_DEVICE: return "device-side check failed";
        case HA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

const char* hash_attn_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"

// ---------------------------------------------------------------- allocation-free GATHER-ATT
//
// Scratch for hash_attn_gather_att_noalloc: a fixed device array of the library
// module. Host code must not hand the array's name to a kernel (on the host it
// only stands in for the symbol); the device address is looked up per device.

namespace ha {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[HA_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 128;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoallocMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current). The array needs no clearing at set-up: a
// module's __device__ variables start zeroed when the module loads, and every
// call clears what it relies on in stream order.
ha_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kNoallocMaxDevices)
        return fail(HA_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kNoallocMaxDevices);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return HA_OK;
}

}  // namespace
}  // namespace ha

extern "C" ha_status hash_attn_gather_att_noalloc(const ha_shape* shape, const void* q, const void* K,
                                                  const void* V, const int32_t* seq_lens, const int32_t* idx,
                                                  int32_t idx_cap, const int32_t* cnt, float* out, float* lse,
                                                  uint32_t* dev_flags, void* stream) {
    HA_TRY(check_shape(shape));
    if (q == nullptr || seq_lens == nullptr || out == nullptr || lse == nullptr || cnt == nullptr)
        return fail(HA_ERR_INVALID_ARG, "q, seq_lens, cnt, out and lse must not be NULL");
    if (idx_cap < 0 || idx_cap > shape->n_cap)
        return fail(HA_ERR_INVALID_ARG, "idx_cap must be in [0, n_cap] (got %d)", idx_cap);
    if (idx == nullptr && idx_cap > 0) return fail(HA_ERR_INVALID_ARG, "idx is NULL");
    HA_TRY(check_kv(shape, K, V));
    const Layout lay = make_layout(*shape, idx_cap, false);
    if (lay.total > HA_NOALLOC_SCRATCH_BYTES)
        return fail(HA_ERR_WORKSPACE,
                    "this shape needs %zu bytes of scratch; the built-in scratch holds %u bytes "
                    "(use hash_attn_gather_att with a caller workspace)",
                    lay.total, (unsigned)HA_NOALLOC_SCRATCH_BYTES);
    void* ws = nullptr;
    HA_TRY(noalloc_scratch(&ws));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // every call clears the error word and the split-K arrival counters on the
    // caller's stream (the partials that follow them are overwritten before they
    // are read), so nothing left by an earlier call can leak into this one
    cudaError_t e = cudaMemsetAsync(ws, 0, lay.off_part, st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the error word and counters");
    const Views v = views(lay, ws);
    GatherParams gp = gather_params(shape, lay, v, q, K, V, seq_lens, out, lse);
    gp.mode = kList;
    gp.list_idx = idx;
    gp.list_cnt = cnt;
    gp.list_cap = idx_cap;
    HA_LAUNCH(launch_gather(gp, shape->d, shape->kv_dtype == HA_BF16, st), "GATHER-ATT launch");
    if (dev_flags != nullptr) {
        e = cudaMemcpyAsync(dev_flags, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "copying the error word");
    }
    return HA_OK;
}
