// Internal declarations shared by the library's translation units: workspace
// layout, kernel parameter blocks, launch helpers and small device primitives
// (mbarrier waits with a time limit, bulk global->shared copies).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "hashattn.h"

namespace ha {

// ------------------------------------------------------------------ constants

constexpr int kScoreThreads = 256;        // SCORE / TOPK block size
constexpr int kMaxHeadsPerPass = 4;       // query heads of one KV head handled per code pass
constexpr int kTargetCtas = 2 * 152;      // two CTAs per SM of a GB300 (152 SMs)
constexpr int kTileRows = 32;             // GATHER-ATT rows per pipeline stage
constexpr int kGatherThreads = 128;       // 4 warps, each with its own copy pipeline
constexpr int kSegPerChunk = kScoreThreads / 32;  // TOPK writes one segment per warp
constexpr int kMaxSegments = 4096;        // segments per head (bounds GATHER-ATT's prefix table)
constexpr int64_t kMaxCap = int64_t(1) << 24;  // largest n_cap accepted
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per pipeline wait
constexpr int kSMs = 152;                 // SMs of a GB300
constexpr int kFusedRange = 8192;         // tokens per range of the fused selection (one CTA each)

// ------------------------------------------------------------------ workspace
//
// [0, 256)                 error word (uint32) + padding
// zero between calls (self-resetting), at offsets fixed by the shape:
// counters   uint32[heads]  split-K arrival counters of GATHER-ATT
// score_cnt  uint32[batch*h_kv]          SCORE arrival counters
// tot, ready                             fused selection totals and ready flags
// scratch (its layout depends on the budget, the options and the path):
// chunk_hist uint32[heads][nchunks][33]  SCORE histogram of every chunk
// seg_cnt    int32 [heads][nseg]         selected tokens of every segment (one
//                                          per warp sub-chunk of seg_cap tokens)
// seg_idx    int32 [heads][nseg*seg_cap] selected token indices, segment s's
//                                          entries at [s*seg_cap, s*seg_cap + seg_cnt)
// part       float [heads][splits][2 + d] split-K partials (max, sum, o[d])
// meta_t     int32 [heads]                threshold bin t of every head
// meta_qt    int2  [heads][nchunks]       per chunk: (tie quota left, ties in chunk)
struct Layout {
    int heads = 0;
    bool fused = false;      // fused selection: flat lists instead of segments
    int nranges = 0;         // fused: ranges of 8192 tokens per (batch entry, KV head)
    int chunk = 0;           // tokens per SCORE/TOPK chunk (0: no selection regions)
    int nchunks = 0;
    int seg_cap = 0;         // tokens per TOPK segment (chunk / kSegPerChunk)
    int nseg = 0;            // segments per head
    int rows_cap = 0;        // most rows one head attends to
    int splits = 1;          // GATHER-ATT CTAs per head
    int rows_per_split = 0;  // multiple of kTileRows
    int nbins = HA_NBINS;    // distance bins per chunk histogram (b + 1 for b-bit codes)
    size_t off_err = 0, off_counter = 0, off_hist = 0, off_segcnt = 0, off_seg = 0, off_part = 0;
    size_t off_scnt = 0, off_meta_t = 0, off_meta_qt = 0;
    size_t off_list = 0, off_lcnt = 0;  // fused: flat lists [heads][rows_cap] and their counts [heads]
    size_t off_dist = 0;                // fused: packed distances [batch * h_kv][d_sp]
    size_t off_rh = 0;                  // fused: per range, 3 x 4 prefix-summed histograms of 36 words
    size_t off_meta_r = 0;              // fused: per (pair, range, head) int4 {first position, ties taken, ties, count}
    size_t off_meta_tt = 0;             // fused: per (pair, head) int2 {t, total}
    size_t off_tot = 0;                 // fused: per (pair, head) 36-word distance histogram (zero at rest)
    size_t off_ready = 0;               // fused: per pair, shares-complete flag (zero at rest)
    int64_t d_sp = 0;                   // fused: words per row of the distance buffer
    size_t total = 0;
};

// Chunk of tokens per SCORE/TOPK CTA for a shape: kScoreThreads * TPT for the
// largest TPT in {32, 16, 8, 4} that still gives kTargetCtas CTAs, else TPT = 4.
int choose_chunk(int64_t batch_hkv, int64_t n_cap);
// Split-K policy for GATHER-ATT.
void choose_splits(int64_t heads, int64_t rows_cap, int* splits, int* rows_per_split);
// SCORE and TOPK with one popcount per (token, query head) (k_sel_scan +
// k_sel_emit) take 32-bit codes with at most 4 query heads per KV head; other
// shapes take the two-kernel path that recomputes the distances.
bool fused_selection(const ha_shape& s, int code_words);
// Ranges of 8192 tokens (one CTA each) per (batch entry, KV head) of the fused path.
int fused_ranges(int n_cap);
// Full layout; with_selection=false leaves out the selection regions. With a
// fused plan the selection regions are the flat lists; otherwise the chunk
// histograms, segments and threshold metadata of the two-kernel path.
// dense_parts: room for the partials of the dense path on the group kernel.
Layout make_layout(const ha_shape& s, int64_t rows_cap, bool with_selection, int nbins = HA_NBINS,
                   int code_words = 1, bool dense_parts = false);

// ------------------------------------------------------------------ parameters

struct ScoreParams {
    const uint32_t* q_sig;   // [B, Hq]
    const uint32_t* k_sig;
    int64_t ks_sb, ks_sh;
    const int32_t* seq_lens;
    int B, Hq, Hkv, G, n_cap;
    int chunk, nchunks;
    uint32_t* chunk_hist;    // [heads][nchunks][33]
    uint32_t* counters;      // reset to zero for the heads of this KV head (may be null)
    uint8_t* dist;           // optional [B, Hq, n_cap]
    uint32_t* err;
    // selection thresholds (null: histograms only): the last CTA of a
    // (batch entry, KV head) derives t and every chunk's tie quota
    const int32_t* m_per_seq;
    const int32_t* m_per_head;   // [B * Hq] or null: budgets per query head (override m_per_seq)
    int m;
    int excl;                // 1: the top-m is taken over the tokens outside the windows
    int n_sink, n_local;
    uint32_t* score_cnt;     // [B * Hkv]
    int32_t* meta_t;         // [heads]
    int2* meta_qt;           // [heads][nchunks]
};

struct SelectParams {
    const uint32_t* q_sig;
    const uint32_t* k_sig;
    int64_t ks_sb, ks_sh;
    const int32_t* seq_lens;
    int n_sink, n_local;
    int B, Hq, Hkv, G, n_cap;
    int chunk, nchunks;
    const int32_t* meta_t;   // [heads]
    const int2* meta_qt;     // [heads][nchunks]
    int excl;                // window tokens are never ties (exclusive windows)
    int32_t* seg_cnt;        // [heads][nseg]
    int32_t* seg_idx;        // [heads][nseg * seg_cap]
    uint32_t* err;
};

// Fused SCORE+TOPK (k_sel_scan, k_sel_emit): one CTA per range of 8192 tokens of
// a (batch entry, KV head) in each kernel.
struct FusedSelParams {
    const uint32_t* q_sig;   // [B * Hq]
    const uint32_t* k_sig;
    int64_t ks_sb, ks_sh;
    const int32_t* seq_lens;
    const int32_t* m_per_seq;    // [B] or null
    const int32_t* m_per_head;   // [B * Hq] or null (overrides m_per_seq)
    int m, n_sink, n_local, excl;
    int B, Hq, Hkv, G, n_cap;
    uint32_t kv_mul;         // query-head groups per KV head k: group g reads KV head kv_head(g, kv_mul)
    int nranges;             // ranges per (batch entry, KV head)
    uint32_t* dist;          // [B * Hkv][d_sp] packed distances (head e in byte e), token order
    int64_t d_sp;
    uint32_t* rh;            // [B * Hkv][nranges][3][4][36] prefix-summed histograms
    uint32_t* arrive;        // [B * Hkv] arrival counters of k_sel_scan (self-resetting)
    uint32_t* tot;           // [B * Hkv][4][36] per-sequence distance histograms (summed, then cleared)
    int4* meta_r;            // [B * Hkv][nranges][4]
    int2* meta_t;            // [B * Hkv][4]
    uint32_t* ready;         // [B * Hkv] or null: set to `epoch` once a pair's shares are
                             // written (k_group_att waits for that value and resets it)
    uint32_t epoch;          // nonzero tag of the call (a flag left by an earlier call differs)
    int32_t* list;           // [B * Hq][cap] selected tokens, ascending
    int cap;
    int32_t* cnt;            // [B * Hq]
    int pad;                 // 1: list[cnt .. cap) = -1
    uint32_t* err;
};

struct CompactParams {
    const int32_t* seq_lens;
    int Hq, n_cap, seg_cap, nseg, cap;
    const int32_t* seg_cnt;
    const int32_t* seg_idx;
    int32_t* sel_idx;        // [heads][cap]
    int32_t* sel_cnt;        // [heads]
    uint32_t* err;
};

struct HistParams {
    const int32_t* seq_lens;
    int Hq, n_cap, chunk, nchunks;
    const uint32_t* chunk_hist;
    uint32_t* hist;          // [heads][33]
};

enum IndexMode : int { kIdentity = 0, kSegmented = 1, kList = 2 };

struct GatherParams {
    const void* q;
    int64_t q_sb, q_sh;
    int q_bf16;
    const char* K;
    const char* V;
    int64_t k_sb, k_sh, k_sn, v_sb, v_sh, v_sn;  // elements
    const int32_t* seq_lens;
    int B, Hq, Hkv, G, n_cap;
    uint32_t kv_mul;         // query-head groups per KV head k: group g reads KV head kv_head(g, kv_mul)
    int mode;
    // kSegmented
    const int32_t* seg_cnt;
    const int32_t* seg_idx;
    int seg_cap, nseg;
    // kList
    const int32_t* list_idx;
    const int32_t* list_cnt;
    int list_cap;
    int splits, rows_per_split;
    float* part;
    uint32_t* counters;
    uint32_t* err;
    float* out;
    float* lse;
    float qscale;            // log2(e) / sqrt(d)
};

// k_group_att: the selection masks of a GQA group and GATHER-ATT over the union
// of its query heads' rows. `sel` carries the scan's metadata (its lists are
// not used), `att` the query, cache, outputs and the partials [heads][nranges][d + 2]
// (the arrival counters are indexed by (batch entry, KV head)).
struct GroupAttParams {
    FusedSelParams sel;
    GatherParams att;
    int nsplit;              // CTAs per range, each taking a contiguous part of the union's chunks
};

struct MergeParams {
    const float* out_a; const float* lse_a;
    const float* out_b; const float* lse_b;
    float* out; float* lse;
    int rows, d;
};

// Sign-projection codes of query vectors (keys == 0: codes[b * Hq + h] from
// x[b, h] under W[h / G]) or of appended keys (keys == 1: codes[b, g, pos[b]]
// from x[b, g, pos[b]] under W[g]; element strides x_sb/x_sh/x_sn, code strides
// c_sb/c_sh).
struct EncodeParams {
    const void* x;
    int x_bf16;
    int64_t x_sb, x_sh, x_sn;
    const float* W;          // [Hkv][32][d]
    uint32_t* codes;
    int64_t c_sb, c_sh;
    const int32_t* pos;      // keys only
    uint32_t* flags;         // optional (keys): HA_DEVERR_INDEX for a position outside [0, n_cap)
    int B, Hq, Hkv, G, d, n_cap, keys;
    // MLP map (k_encode_mlp): per KV head W1 [hidden][d], W2 [hidden][hidden], W3 [32][hidden]
    const float *W1, *b1, *W2, *b2, *W3, *b3;
    int hidden;
};

// SCORE/TOPK for codes of W > 1 words (b = 32 W bits, NB = b + 1 bins); the
// output segments are those of the 32-bit path.
struct WideParams {
    const uint32_t* q_sig;   // [B * Hq][W]
    const uint32_t* k_sig;   // word w of token i: b * ks_sb + g * ks_sh + i * W + w
    int64_t ks_sb, ks_sh;
    const int32_t* seq_lens;
    int B, Hq, Hkv, G, n_cap, W, NB;
    int chunk, nchunks;
    uint32_t* chunk_hist;    // [heads][nchunks][NB]
    uint32_t* counters;
    uint32_t* err;
    const int32_t* m_per_seq;
    int m, n_sink, n_local;
    uint32_t* score_cnt;
    int32_t* meta_t;
    int2* meta_qt;
    int32_t* seg_cnt;
    int32_t* seg_idx;
};

// Exact top-m by dot score (the comparator of the hashed selection).
struct ExactParams {
    const void* q;
    int64_t q_sb, q_sh;
    int q_bf16;
    const char* K;
    int64_t k_sb, k_sh, k_sn;  // elements
    const int32_t* seq_lens;
    int B, Hq, Hkv, G, n_cap, m;
    float* scores;             // [B * Hq][n_cap] (workspace)
    int32_t* idx;              // [B * Hq][idx_cap]
    int idx_cap;
    int32_t* cnt;              // [B * Hq]
    uint32_t* err;
    uint16_t* qt;              // [B * Hkv][64][d] bf16 query tiles of the tensor-core kernel (workspace)
    int bitmap_words;          // top-m: words of each token bitmap in shared memory (0: no fast path)
};

struct RecallParams {
    const int32_t* sel_idx; const int32_t* sel_cnt; int sel_cap;
    const int32_t* ref_idx; const int32_t* ref_cnt; int ref_cap;
    int heads;
    float* recall;
};

struct MergeNParams {
    const float* outs; int64_t out_seg_stride;
    const float* lses; int64_t lse_seg_stride;
    int nseg;
    float* out; float* lse;
    int rows, d;
};

// Launch with (pdl = true) or without programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Launchers (each returns cudaGetLastError() of its launch).
cudaError_t launch_score(const ScoreParams& p, int batch_hkv, cudaStream_t st);
cudaError_t launch_select(const SelectParams& p, int batch_hkv, cudaStream_t st, bool pdl = false);
cudaError_t launch_select_fused(const FusedSelParams& p, int batch_hkv, cudaStream_t st);
// k_sel_scan alone (the threshold metadata, no lists); write_dist = false leaves
// out the packed distances (their consumer recomputes them from the codes);
// pdl = true lets its counting overlap the previous kernel in the stream.
cudaError_t launch_sel_scan(const FusedSelParams& p, int batch_hkv, cudaStream_t st, bool write_dist, bool pdl);
cudaError_t launch_compact(const CompactParams& p, int heads, cudaStream_t st);
cudaError_t launch_hist(const HistParams& p, int heads, cudaStream_t st);
cudaError_t launch_gather(const GatherParams& p, int d, int kv_bf16, cudaStream_t st, bool pdl = false);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t st);
// bf16 query and K/V, d in {64, 128}, at most 4 query heads per KV head.
bool group_att_supported(int d, int kv_bf16, int q_bf16, int G);
// CTAs per range of k_group_att for (batch entry, KV head) pairs x ranges.
int group_splits(int64_t pair_ranges);
cudaError_t launch_group_att(const GroupAttParams& p, int d, int batch_hkv, cudaStream_t st, bool pdl);
// The dense path on the same kernel: every token of the sequence for every head
// of the group, ranges of 8192 tokens cut into group_dense_splits spans (p.sel
// needs only the shape fields, seq_lens, nranges and err; p.sel.ready null).
int group_dense_splits(int64_t batch_hkv, int n_cap);
cudaError_t launch_group_dense(const GroupAttParams& p, int d, int batch_hkv, cudaStream_t st, bool pdl);
cudaError_t launch_merge_n(const MergeNParams& p, cudaStream_t st);
cudaError_t launch_encode(const EncodeParams& p, cudaStream_t st);
cudaError_t launch_encode_mlp(const EncodeParams& p, cudaStream_t st);
// The exact comparator: every score (tensor cores or CUDA cores), then the top-m.
cudaError_t launch_exact_scores(const ExactParams& p, int d, int kv_bf16, cudaStream_t st);
cudaError_t launch_exact_topm(const ExactParams& p, cudaStream_t st);
// Tensor-core scores (bf16 K, 3 G <= 64); *used = false leaves the scores to
// the CUDA-core kernel (a layout TMA cannot describe).
cudaError_t launch_scores_tc(const ExactParams& p, int d, cudaStream_t st, bool* used);
cudaError_t launch_recall(const RecallParams& p, cudaStream_t st);
cudaError_t launch_score_wide(const WideParams& p, int batch_hkv, cudaStream_t st);
cudaError_t launch_select_wide(const WideParams& p, int batch_hkv, cudaStream_t st, bool pdl);

// Query-head groups per KV head: group g of k per KV head reads KV head g / k. The
// kernels divide by a multiply-high with kv_magic(k) = ceil(2^32 / k), exact for
// every g below 2^28 (the error of the reciprocal is below k <= 16 parts in 2^32);
// 0 stands for k = 1.
inline uint32_t kv_magic(int k) {
    return k <= 1 ? 0u : (uint32_t)((0x100000000ull + (uint64_t)k - 1u) / (uint64_t)k);
}

// ------------------------------------------------------------------ device helpers

#ifdef __CUDACC__

// The KV head of query-head group g (kv_mul = kv_magic(groups per KV head)).
__device__ __forceinline__ int kv_head(int g, uint32_t kv_mul) {
    return kv_mul != 0u ? (int)__umulhi((uint32_t)g, kv_mul) : g;
}

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t f) {
    if (err) atomicOr(err, f);
}

// Valid length of batch entry b, or 0 (flagged) when outside [0, n_cap].
__device__ __forceinline__ int checked_len(const int32_t* seq_lens, int b, int n_cap, uint32_t* err,
                                           bool report) {
    int n = seq_lens[b];
    if (n < 0 || n > n_cap) {
        if (report) flag_error(err, HA_DEVERR_SEQLEN);
        return 0;
    }
    return n;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity; gives up after
// kWaitLimitNs (returns false) or as soon as *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort) return false;
            if (global_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 only (LDGSTS).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Make `bar` track completion of every cp.async this thread has issued so far:
// its pending count rises by one now and falls by one when they have landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor drains; it must wait here
// before touching the predecessor's outputs. launch_dependents lets the next
// such kernel start early (it changes only when it may start, not what it sees).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

#endif  // __CUDACC__

}  // namespace ha
