/*
 * hashattn.h -- C ABI of the GB300 (sm_103a) sparse-decode library.
 *
 * One decode step of HashAttention sparse attention, per (batch entry b, query
 * head h), with g = h / (h_q / h_kv) the KV head h reads:
 *
 *   SCORE       dist_i = popcount(q_sig[b,h] XOR k_sig[b,g,i]),  i < n = seq_lens[b]
 *               (HashAttention: Semantic Sparsity for Faster Inference, Eq. (2):
 *                SCORE = -dist, so the best tokens have the smallest distance)
 *   TOPK        T = the min(m, n) tokens of smallest dist, ties to the smaller
 *               index; I = T u [0, min(S, n)) u [max(0, n - Lw), n), ascending
 *               (same page, Sec. 4 "three stages" and Sec. 4.4 fixed windows)
 *   GATHER-ATT  z_i = <q, K_i> / sqrt(d) over i in I, read in place (page size 1);
 *               out = sum_i e^{z_i} V_i / sum_j e^{z_j},  lse = log sum_j e^{z_j}
 *               (same page, Sec. 4 estimator; lse is the log attention mass of
 *                Nectar: Neural Estimation of Cached-Token Attention via
 *                Regression, Sec. 3 Eq. (3.1))
 *   merge       partial results over disjoint token sets combine exactly through
 *               their log-normalisers (Nectar, Eqs. (3.4)-(3.5))
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers unless stated; the caller owns every
 *    buffer. The library allocates no device memory and keeps no global state
 *    other than a thread-local last-error string, the fixed scratch array of
 *    hash_attn_gather_att_noalloc and a process-wide call count (the tag a
 *    decode call's selection writes into its workspace's ready flags, so that a
 *    kernel of the next call, which may start before this one's have finished,
 *    never takes this call's flags for its own).
 *  - A workspace sized for the largest use serves calls of any smaller budget,
 *    any window, option or path on its shape in turn (one stream at a time):
 *    what must be zero between calls sits at offsets fixed by the shape.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). All work is enqueued on it; no call synchronises except
 *    hash_attn_device_status and hash_attn_workspace_init's caller-visible copy.
 *  - Argument errors are found on the host and returned BEFORE anything is
 *    enqueued. Errors that only the device can see (a seq_len outside
 *    [0, n_cap], a per-sequence budget above the bound, an index outside
 *    [0, seq_len)) set a flag in the workspace's error word; the affected
 *    (b, h) results are defined (empty set: out = 0, lse = -inf, or the bad
 *    index is skipped) and the flag is read with hash_attn_device_status.
 *  - Kernel-launch failures return HA_ERR_CUDA. hash_attn_last_error() returns a
 *    human-readable detail of the last failure on the calling thread.
 *  - Layouts are given as element strides (not bytes). The innermost (d / token)
 *    dimension of every tensor is contiguous.
 */
#ifndef HASHATTN_H
#define HASHATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HA_OK = 0,
    HA_ERR_INVALID_ARG = -1,  /* null pointer, bad size, stride or alignment   */
    HA_ERR_UNSUPPORTED = -2,  /* d not in {64, 128}, dtype not supported        */
    HA_ERR_WORKSPACE = -3,    /* workspace null, unaligned or too small         */
    HA_ERR_CUDA = -4,         /* a CUDA runtime call or kernel launch failed    */
    HA_ERR_DEVICE = -5,       /* a device-side check failed (see the error word) */
    HA_ERR_TIMEOUT = -6       /* a bounded device wait ran out                  */
} ha_status;

typedef enum { HA_F32 = 0, HA_BF16 = 1 } ha_dtype;

/* Device error-word flags (OR-ed together, read by hash_attn_device_status). */
#define HA_DEVERR_SEQLEN   0x1u  /* seq_lens[b] < 0 or > n_cap: b treated as empty */
#define HA_DEVERR_BUDGET   0x2u  /* m_per_seq[b] < 0 or > the bound m: clamped     */
#define HA_DEVERR_INDEX    0x4u  /* a given index outside [0, seq_len): skipped     */
#define HA_DEVERR_COUNT    0x8u  /* a given count outside [0, idx_cap]: clamped     */
#define HA_DEVERR_TIMEOUT  0x10u /* a bounded pipeline wait gave up                 */
#define HA_DEVERR_STATE    0x20u /* workspace counters were not in their reset state */

/* Number of Hamming-distance bins of a 32-bit code (distances 0..32). */
#define HA_NBINS 33

/*
 * Problem shape and strides (in elements).
 *   q      [batch, h_q, d]              q[b,h,:]     at q     + b*q_sb  + h*q_sh
 *   K, V   [batch, h_kv, n_cap, d]      K[b,g,i,:]   at K     + b*k_sb  + g*k_sh + i*k_sn
 *   k_sig  [batch, h_kv, n_cap] uint32  k_sig[b,g,i] at k_sig + b*ks_sb + g*ks_sh + i
 * k_sb, v_sb and ks_sb may be 0: every batch entry then reads the same cache
 * (one shared document). q_sig is [batch, h_q] contiguous; seq_lens [batch].
 * Requirements: batch, h_q, h_kv >= 1; h_q % h_kv == 0; d in {64, 128};
 * n_cap >= 1; K/V rows start on 16-byte boundaries (pointer and k_sn/k_sh/k_sb,
 * v_* strides times the element size multiples of 16); k_sig 16-byte aligned
 * with ks_sh and ks_sb multiples of 4.
 */
typedef struct {
    int32_t batch, h_q, h_kv, d, n_cap;
    int32_t q_dtype, kv_dtype;              /* ha_dtype values */
    int64_t q_sb, q_sh;
    int64_t k_sb, k_sh, k_sn;
    int64_t v_sb, v_sh, v_sn;
    int64_t ks_sb, ks_sh;
} ha_shape;

/*
 * Bytes of workspace that hash_attn_decode / _select / _score / _gather_att need
 * for this shape and a budget bound m_max with windows n_sink / n_local
 * (m_max >= n_cap selects the dense layout). Written to *bytes.
 * Errors: HA_ERR_INVALID_ARG / HA_ERR_UNSUPPORTED for a bad shape or negative
 * m_max / n_sink / n_local.
 */
ha_status hash_attn_workspace_size(const ha_shape* shape, int32_t m_max, int32_t n_sink,
                                   int32_t n_local, size_t* bytes);

/*
 * Zero a workspace (enqueued on `stream`). A workspace must be zeroed once
 * before its first use; every call leaves its counters back at zero. After a
 * call that raised HA_DEVERR_TIMEOUT or HA_DEVERR_STATE, zero it again.
 * The workspace pointer must be 256-byte aligned.
 */
ha_status hash_attn_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of the device staging buffer hash_attn_decode_host needs for this shape
 * (the step's q, q codes, sequence lengths, budgets, out and lse).
 */
ha_status hash_attn_host_staging_size(const ha_shape* shape, size_t* bytes);

/*
 * hash_attn_decode with the step's inputs and results in HOST memory (pinned
 * memory makes the copies asynchronous): the inputs are copied into `staging`,
 * the path runs, the results are copied back, all enqueued on `stream`; the
 * results are in out_host / lse_host once the stream has reached them. The
 * cache (k_sig, K, V) and the workspace stay on the device. Copies: one per
 * input, except that inputs which follow each other directly in host memory
 * in the staging order (q, q_sig, seq_lens, m_per_seq; each staged at the next
 * 16-byte boundary) move in one copy, and so do out and lse when lse_host
 * follows out_host directly and out's size is a multiple of 16 bytes.
 *   q_host        contiguous [batch, h_q, d] of shape->q_dtype (shape's q strides
 *                 are ignored: the staged copy is contiguous)
 *   q_sig_host    [batch, h_q] uint32 (may be NULL only for the dense path)
 *   seq_lens_host [batch] int32; m_per_seq_host [batch] int32 or NULL
 *   out_host      [batch, h_q, d] float32, lse_host [batch, h_q] float32
 *   staging       device, >= hash_attn_host_staging_size bytes, 256-byte aligned
 *   the rest as hash_attn_decode (no selected-index output).
 * Errors: every check of hash_attn_decode, and the staging size, before the
 * first copy is enqueued; HA_ERR_CUDA if a copy or launch fails.
 */
ha_status hash_attn_decode_host(const ha_shape* shape, const void* q_host, const uint32_t* q_sig_host,
                                const int32_t* seq_lens_host, const int32_t* m_per_seq_host, const uint32_t* k_sig,
                                const void* K, const void* V, int32_t m, int32_t n_sink, int32_t n_local,
                                float* out_host, float* lse_host, void* staging, size_t staging_bytes,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Capacity of the per-head selected-index list for (n_cap, m, n_sink, n_local):
 * min(n_cap, m + n_sink + n_local) (HashAttention Sec. 4.4: the budget plus the
 * fixed positions bounds the number of reads). n_cap when m >= n_cap.
 */
int32_t hash_attn_select_capacity(int32_t n_cap, int32_t m, int32_t n_sink, int32_t n_local);

/*
 * The whole path: SCORE -> TOPK -> GATHER-ATT (split-K) -> merge.
 *   q          [batch, h_q, d] of shape->q_dtype
 *   q_sig      [batch, h_q] uint32 query codes
 *   k_sig      key codes (see ha_shape)
 *   K, V       cache rows of shape->kv_dtype (see ha_shape)
 *   seq_lens   [batch] int32, valid tokens per entry, 0 <= seq_lens[b] <= n_cap
 *   m_per_seq  [batch] int32 budgets, or NULL for the scalar m. When given, m is
 *              the bound every entry obeys (larger entries are clamped to m and
 *              flagged HA_DEVERR_BUDGET).
 *   m, n_sink, n_local  budget and window sizes (>= 0).
 *              With m >= n_cap and m_per_seq NULL the dense path runs (I is every
 *              token), SCORE/TOPK are skipped, and q_sig / k_sig may be NULL.
 *   out        [batch, h_q, d] float32, lse [batch, h_q] float32 (natural log;
 *              an empty I gives out = 0 and lse = -inf)
 *   sel_idx    optional [batch, h_q, cap] int32, cap = hash_attn_select_capacity,
 *              receives I ascending, padded with -1; sel_cnt optional [batch, h_q]
 *              int32 receives |I|. Both NULL to skip. Ignored by the dense path.
 *   workspace  >= hash_attn_workspace_size(shape, m, n_sink, n_local) bytes,
 *              256-byte aligned, zeroed once before first use.
 * Kernels: with 32-bit codes, a bf16 query, bf16 K/V, d in {64, 128} and sel_idx
 * NULL, two kernels run (more than 4 query heads per KV head are split into
 * groups of at most 4, each run as a KV head of its own that reads the same
 * codes and rows): the selection scan
 * (SCORE and every range's share of TOPK), then one kernel per GQA group that
 * builds each head's selection mask from the codes and attends over the union
 * of the group's rows (each row read once per group; K/V must then be finite,
 * since a row of one head's set is multiplied by weight 0 into the others').
 * The scan may start while the previous kernel in the stream drains: it waits
 * for it before writing workspace state. Otherwise the selection writes per-head
 * lists (or sel_idx) and GATHER-ATT runs per query head. The dense path runs one
 * kernel: per GQA group on the same shapes (each row read once per group; its
 * copies may start while the previous kernel drains, its results are written
 * after it), else per query head.
 * Errors: HA_ERR_INVALID_ARG, HA_ERR_UNSUPPORTED, HA_ERR_WORKSPACE before
 * launch; HA_ERR_CUDA on a failed launch.
 */
ha_status hash_attn_decode(const ha_shape* shape, const void* q, const uint32_t* q_sig,
                           const uint32_t* k_sig, const void* K, const void* V,
                           const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m,
                           int32_t n_sink, int32_t n_local, float* out, float* lse,
                           int32_t* sel_idx, int32_t* sel_cnt, void* workspace,
                           size_t ws_bytes, void* stream);

/*
 * hash_attn_decode with CUDA events recorded between its stages (for the cost
 * model T = T_scan + T_TOPK + T_att of HashAttention Sec. 4.4). `events` points
 * to 4 cudaEvent_t (as void*): recorded before SCORE, before TOPK, before
 * GATHER-ATT and after the last kernel. The dense path records all four around
 * its single kernel. Same arguments and errors as hash_attn_decode.
 */
ha_status hash_attn_decode_timed(const ha_shape* shape, const void* q, const uint32_t* q_sig,
                                 const uint32_t* k_sig, const void* K, const void* V,
                                 const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m,
                                 int32_t n_sink, int32_t n_local, float* out, float* lse,
                                 int32_t* sel_idx, int32_t* sel_cnt, void* workspace,
                                 size_t ws_bytes, void* stream, void* const* events);

/*
 * Selection variants (HashAttention Sec. 4.4 budget accounting; adaptive
 * budgets). Zero-initialise and set what is needed:
 *   m_per_head         device int32 [batch, h_q] budget of every query head (each
 *                      in [0, m]; outside values are clamped and flagged
 *                      HA_DEVERR_BUDGET), overriding m_per_seq; NULL: none.
 *   exclusive_windows  0: the top-m is taken over all n tokens and joined with
 *                      the windows (|I| <= m + windows). 1: the top-m is taken
 *                      over the tokens outside the windows, so
 *                      |I| = min(n, m + |windows|) exactly.
 *   code_words         W, the 32-bit words of every code: 0 or 1 (32-bit codes,
 *                      the layout of ha_shape), 2, 4, 8 or 16 (b = 32 W bits,
 *                      HashAttention Sec. 5 varies the signature length). Then
 *                      q_sig is [batch, h_q, W] words, word w of token i's code
 *                      is k_sig[b * ks_sb + g * ks_sh + i * W + w] (ks_* in
 *                      words, rows 16-byte aligned, ks_sh >= n_cap * W), and the
 *                      distance is summed over the words (b + 1 values). Codes
 *                      wider than 32 bits take the default budget rules
 *                      (m_per_head and exclusive_windows unset), and the
 *                      workspace must come from hash_attn_workspace_size_ex.
 *   reserved           must be zero.
 */
typedef struct {
    const int32_t* m_per_head;
    int32_t exclusive_windows;
    int32_t code_words;
    int32_t reserved[2];
} ha_select_opts;

/* hash_attn_workspace_size for the given selection options (opts may be NULL). */
ha_status hash_attn_workspace_size_ex(const ha_shape* shape, int32_t m_max, int32_t n_sink, int32_t n_local,
                                      const ha_select_opts* opts, size_t* bytes);

/*
 * hash_attn_decode with selection options (opts may be NULL: the defaults of
 * hash_attn_decode). The workspace size and the sel_idx capacity are those of
 * hash_attn_decode for the same m, n_sink, n_local.
 */
ha_status hash_attn_decode_ex(const ha_shape* shape, const void* q, const uint32_t* q_sig, const uint32_t* k_sig,
                              const void* K, const void* V, const int32_t* seq_lens, const int32_t* m_per_seq,
                              int32_t m, int32_t n_sink, int32_t n_local, const ha_select_opts* opts, float* out,
                              float* lse, int32_t* sel_idx, int32_t* sel_cnt, void* workspace, size_t ws_bytes,
                              void* stream);

/*
 * SCORE alone (HashAttention Eq. (2)).
 *   dist  optional [batch, h_q, n_cap] uint8: dist[b,h,i] for i < seq_lens[b]
 *         (entries at i >= seq_lens[b] are not written)
 *   hist  optional [batch, h_q, 33] uint32: number of tokens at each distance
 * At least one of dist / hist must be non-NULL. Errors as hash_attn_decode.
 */
ha_status hash_attn_score(const ha_shape* shape, const uint32_t* q_sig, const uint32_t* k_sig,
                          const int32_t* seq_lens, uint8_t* dist, uint32_t* hist,
                          void* workspace, size_t ws_bytes, void* stream);

/*
 * SCORE + TOPK (the selected set I of hash_attn_decode, same tie rule and
 * windows), written to sel_idx [batch, h_q, cap] (ascending, -1 padded) and
 * sel_cnt [batch, h_q]; cap = hash_attn_select_capacity(n_cap, m, n_sink, n_local).
 * m >= n_cap is allowed here (every token is then selected).
 */
ha_status hash_attn_select(const ha_shape* shape, const uint32_t* q_sig, const uint32_t* k_sig,
                           const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m,
                           int32_t n_sink, int32_t n_local, int32_t* sel_idx, int32_t* sel_cnt,
                           void* workspace, size_t ws_bytes, void* stream);

/* hash_attn_select with selection options (see ha_select_opts; NULL = defaults). */
ha_status hash_attn_select_ex(const ha_shape* shape, const uint32_t* q_sig, const uint32_t* k_sig,
                              const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m, int32_t n_sink,
                              int32_t n_local, const ha_select_opts* opts, int32_t* sel_idx, int32_t* sel_cnt,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * The selection plan the library takes for a shape (host-only: no device call,
 * no allocation). It depends only on the shape and the code width, so it also
 * fixes the layout that hash_attn_workspace_size(_ex) sizes.
 *   code_words  words per code (1 = the 32-bit codes of HashAttention Eq. (2))
 *   fused       1: the decode computes each distance once (32-bit codes; a KV
 *               head with more than 4 query heads runs as groups of at most 4):
 *               a scan kernel writes per-range histograms, then the group kernel
 *               (or, with selection outputs, an emit kernel) builds the masks;
 *               0: the two-kernel path that recomputes the distances in TOPK
 *   ranges      CTAs of 8192 tokens per (batch entry, KV head group) of the
 *               fused kernels (0 if not fused)
 *   range       8192 (tokens per fused CTA), 0 if not fused
 *   chunk       tokens per CTA of the two-kernel SCORE/TOPK (used by
 *               hash_attn_score, and by hash_attn_select for more than 4 query
 *               heads per KV head, whatever `fused` says)
 * Any output pointer may be NULL. HA_ERR_INVALID_ARG / HA_ERR_UNSUPPORTED as
 * hash_attn_workspace_size for a bad shape or code width.
 */
ha_status hash_attn_selection_plan(const ha_shape* shape, int32_t code_words, int32_t* fused,
                                   int32_t* ranges, int32_t* range, int32_t* chunk);

/*
 * The kernels hash_attn_decode_ex (and hash_attn_decode, hash_attn_decode_host)
 * runs for this shape, budget and options; nothing is launched and no pointer is
 * read. HashAttention Sec. 4 defines what every path computes; they differ only
 * in how:
 *   HA_PATH_DENSE_GROUP  m >= n_cap with no smaller budget: every token, one CTA
 *                        per (batch entry, KV head group, span of a range)
 *   HA_PATH_DENSE_HEADS  the same on the per-head GATHER-ATT, for what the
 *                        group kernel does not take (an fp32 query or cache,
 *                        d other than 64 or 128)
 *   HA_PATH_GROUP        the SCORE/TOPK scan, then one kernel per (batch entry,
 *                        KV head group, range) over the union of the group's rows
 *   HA_PATH_FUSED_LISTS  selection outputs requested: one SCORE/TOPK kernel
 *                        writing the lists, then the per-head GATHER-ATT
 *   HA_PATH_TWO_KERNEL   code_words > 1: SCORE, TOPK and the per-head GATHER-ATT
 * with_selection: nonzero when sel_idx / sel_cnt will be given. m_per_seq only
 * matters for being NULL or not. Errors as hash_attn_workspace_size for a bad
 * shape or options; HA_ERR_INVALID_ARG for m < 0 or a NULL path.
 */
enum {
    HA_PATH_DENSE_GROUP = 1,
    HA_PATH_DENSE_HEADS = 2,
    HA_PATH_GROUP = 3,
    HA_PATH_FUSED_LISTS = 4,
    HA_PATH_TWO_KERNEL = 5
};
ha_status hash_attn_decode_path(const ha_shape* shape, int32_t m, const int32_t* m_per_seq,
                                const ha_select_opts* opts, int32_t with_selection, int32_t* path);

/*
 * GATHER-ATT + merge over caller-given index lists (page size 1, read in place):
 *   idx  [batch, h_q, idx_cap] int32 token indices (any order, no duplicates
 *        expected; each must lie in [0, seq_lens[b]) or it is skipped and
 *        HA_DEVERR_INDEX is flagged), cnt [batch, h_q] int32 valid entries.
 * idx_cap <= hash_attn_select_capacity(n_cap, m_max, n_sink, n_local) of the
 * workspace's sizing. Outputs as hash_attn_decode.
 */
ha_status hash_attn_gather_att(const ha_shape* shape, const void* q, const void* K,
                               const void* V, const int32_t* seq_lens, const int32_t* idx,
                               int32_t idx_cap, const int32_t* cnt, float* out, float* lse,
                               void* workspace, size_t ws_bytes, void* stream);

/*
 * GATHER-ATT + merge over caller-given index lists, like hash_attn_gather_att,
 * but with no workspace argument and no device allocation anywhere: its scratch
 * (error word, split counters, split-K partials) is a fixed array compiled into
 * the library, HA_NOALLOC_SCRATCH_BYTES long, that every GPU which loads the
 * library keeps until the process exits. The paper has no counterpart; this is
 * for callers that are not allowed to allocate device memory, for instance a
 * plugin whose host application owns every device allocation through its own
 * pool, or a latency-critical path where cudaMalloc's implicit synchronisation
 * with the device would stall other work.
 *   dev_flags  optional device pointer to one uint32 that receives this call's
 *              HA_DEVERR_* bits (0 = clean) in stream order; NULL to skip.
 * Shapes whose scratch would exceed HA_NOALLOC_SCRATCH_BYTES are rejected with
 * HA_ERR_WORKSPACE before anything is enqueued (the scratch holds
 * 256 + 4 * batch * h_q plus 4 * batch * h_q * splits * (d + 2) bytes, rounded).
 * The first call on a device (with that device current) looks up the array's
 * device address once; the array itself starts zeroed when the library loads.
 * Every call first clears the error word and the split counters with one
 * cudaMemsetAsync on `stream`, so a call never depends on what an earlier call
 * left behind. All calls share the one array, which keeps the last call's
 * contents: calls that overlap on the GPU (other streams, other host threads)
 * race and must not be issued. Other arguments, layouts and errors as
 * hash_attn_gather_att.
 */
#define HA_NOALLOC_SCRATCH_BYTES (16u << 20)
ha_status hash_attn_gather_att_noalloc(const ha_shape* shape, const void* q, const void* K,
                                       const void* V, const int32_t* seq_lens, const int32_t* idx,
                                       int32_t idx_cap, const int32_t* cnt, float* out, float* lse,
                                       uint32_t* dev_flags, void* stream);

/*
 * Exact merge of two partial attentions over disjoint token sets, row by row
 * (Nectar Eq. (3.4)): L = log(e^{lse_a} + e^{lse_b}),
 * out = e^{lse_a - L} out_a + e^{lse_b - L} out_b. Rows with both lse = -inf
 * give out = 0, lse = -inf. out/lse may alias out_a/lse_a or out_b/lse_b.
 *   out_a, out_b, out [rows, d] float32; lse_a, lse_b, lse [rows] float32.
 */
ha_status hash_attn_merge(const float* out_a, const float* lse_a, const float* out_b,
                          const float* lse_b, float* out, float* lse, int32_t rows, int32_t d,
                          void* stream);

/*
 * Codes of the decode step's queries by sign projection (HashAttention Sec. 4.1:
 * the signature is ReLU(sign(.)) of a projection, so bit j is 1 iff projection j
 * is positive; a given 32 x d projection per KV head stands in for the learned
 * map): q_sig[b, h] = code of q[b, h, :] under W[h / G].
 *   q      per shape (q_dtype, q_sb, q_sh), device
 *   W      float32 [h_kv, 32, d] contiguous, device
 *   q_sig  uint32 [batch, h_q] contiguous, device (written)
 * Projections accumulate in float32 (four interleaved partial sums over the
 * dims, a fixed order, so results are reproducible).
 * Errors: HA_ERR_INVALID_ARG / HA_ERR_UNSUPPORTED (shape, NULL pointers) before
 * anything is enqueued.
 */
ha_status hash_attn_encode_queries(const ha_shape* shape, const void* q, const float* W, uint32_t* q_sig,
                                   void* stream);

/*
 * Append the newly cached tokens' key codes: for every batch entry b and KV head
 * g with 0 <= pos[b] < n_cap, k_sig[b, g, pos[b]] = code of K[b, g, pos[b], :]
 * under W[g] (same rule as hash_attn_encode_queries). Nothing else of k_sig is
 * touched; an entry with pos[b] outside [0, n_cap) is skipped and, when
 * dev_flags is given, HA_DEVERR_INDEX is OR-ed into *dev_flags (device uint32).
 *   K      per shape (kv_dtype, k_sb, k_sh, k_sn), device
 *   W      float32 [h_kv, 32, d] contiguous, device
 *   pos    int32 [batch], device
 *   k_sig  per shape (ks_sb, ks_sh), device
 * Errors: HA_ERR_INVALID_ARG / HA_ERR_UNSUPPORTED before anything is enqueued.
 */
ha_status hash_attn_encode_keys(const ha_shape* shape, const void* K, const float* W, const int32_t* pos,
                                uint32_t* k_sig, uint32_t* dev_flags, void* stream);

/*
 * The signature map as an MLP (HashAttention Sec. 5 runs the map as
 * d -> 128 -> 128 -> 32; the widths are given, the rest is the plainest
 * reading): per KV head g, F(x) = W3 relu(W2 relu(W1 x + b1) + b2) + b3 and
 * bit j of the code is 1 iff F_j(x) > 0. All float32, contiguous, device:
 *   W1 [h_kv, hidden, d], b1 [h_kv, hidden], W2 [h_kv, hidden, hidden],
 *   b2 [h_kv, hidden], W3 [h_kv, 32, hidden], b3 [h_kv, 32];
 *   hidden is 32, 64 or 128; W1, W2 and W3 are 16-byte aligned; reserved is 0.
 * Layers accumulate in float32 over their inputs in order.
 */
typedef struct {
    const float* W1;
    const float* b1;
    const float* W2;
    const float* b2;
    const float* W3;
    const float* b3;
    int32_t hidden;
    int32_t reserved;
} ha_mlp;

/* hash_attn_encode_queries / hash_attn_encode_keys with the MLP map (same
 * arguments otherwise). Errors: HA_ERR_INVALID_ARG / HA_ERR_UNSUPPORTED (shape,
 * NULL pointers, hidden width, alignment) before anything is enqueued. */
ha_status hash_attn_encode_queries_mlp(const ha_shape* shape, const void* q, const ha_mlp* mlp, uint32_t* q_sig,
                                       void* stream);
ha_status hash_attn_encode_keys_mlp(const ha_shape* shape, const void* K, const ha_mlp* mlp, const int32_t* pos,
                                    uint32_t* k_sig, uint32_t* dev_flags, void* stream);

/*
 * One decode step with the signature map run ahead of SCORE (HashAttention's
 * cost model: T = T_map + T_scan + T_TOPK + T_att). First the code of every
 * sequence's appended token, k_sig[b, g, pos[b]] (pos == NULL: no token is
 * appended; positions outside [0, n_cap) are skipped and flagged in dev_flags
 * as for hash_attn_encode_keys), then the query codes q_sig[b, h], both by the
 * map, then the path of hash_attn_decode_ex reading them.
 *   map     exactly one of W (sign projection float32 [h_kv, 32, d], as for
 *           hash_attn_encode_queries) and mlp non-NULL
 *   q_sig   uint32 [batch, h_q] contiguous, device (written)
 *   k_sig   key codes per shape (read; the appended tokens' codes written)
 *   the rest as hash_attn_decode_ex; the map writes 32-bit codes, so
 *           opts->code_words must be 0 or 1.
 * Errors: as hash_attn_decode_ex, plus HA_ERR_INVALID_ARG / HA_ERR_UNSUPPORTED
 * for the map, all before anything is enqueued.
 */
typedef struct {
    const float* W;
    const ha_mlp* mlp;
} ha_map;

ha_status hash_attn_decode_mapped(const ha_shape* shape, const void* q, const ha_map* map, const int32_t* pos,
                                  uint32_t* q_sig, uint32_t* k_sig, const void* K, const void* V,
                                  const int32_t* seq_lens, const int32_t* m_per_seq, int32_t m, int32_t n_sink,
                                  int32_t n_local, const ha_select_opts* opts, float* out, float* lse,
                                  int32_t* sel_idx, int32_t* sel_cnt, void* workspace, size_t ws_bytes,
                                  uint32_t* dev_flags, void* stream);

/*
 * The exact comparator of the hashed selection (HashAttention Sec. 5 measures
 * against the top-k by attention score): for every (b, h), the k = min(m, n)
 * tokens with the largest z_i = <q[b, h], K[b, h / G, i]> (float32, i < n =
 * seq_lens[b]; ties go to the smaller index), written ascending to
 * idx[b, h, 0..k) and padded with -1 to idx_cap; cnt[b, h] = k.
 *   q, K     per shape (K rows 16-byte aligned, as for hash_attn_decode)
 *   idx      int32 [batch, h_q, idx_cap], min(m, n_cap) <= idx_cap <= n_cap
 *   cnt      int32 [batch, h_q]
 *   workspace >= hash_attn_topk_exact_workspace_size bytes, 256-byte aligned
 *            (no zeroing needed: every call clears its first word, the device
 *            error word read by hash_attn_device_status; the scores z of all
 *            heads follow at byte offset 256 as float32 [batch, h_q, n_cap]
 *            (entries i < seq_lens[b] written), then scratch query tiles)
 * bf16 keys with h_q / h_kv <= 21 are scored on the tensor cores (an fp32 q as
 * three bf16 parts that sum to it exactly, float32 accumulation); other shapes on
 * the CUDA cores; both give float32 scores.
 * Errors: HA_ERR_INVALID_ARG / HA_ERR_UNSUPPORTED / HA_ERR_WORKSPACE before
 * anything is enqueued; bad seq_lens are flagged in the error word.
 */
ha_status hash_attn_topk_exact_workspace_size(const ha_shape* shape, size_t* bytes);
ha_status hash_attn_topk_exact(const ha_shape* shape, const void* q, const void* K, const int32_t* seq_lens,
                               int32_t m, int32_t* idx, int32_t idx_cap, int32_t* cnt, void* workspace,
                               size_t ws_bytes, void* stream);

/*
 * hash_attn_topk_exact with three CUDA events (cudaEvent_t as void*, all
 * non-NULL, created by the caller) recorded on `stream` before the scores,
 * between the scores and the top-m, and after the top-m.
 * Errors: those of hash_attn_topk_exact, and HA_ERR_INVALID_ARG for a NULL
 * event, all before anything is enqueued.
 */
ha_status hash_attn_topk_exact_timed(const ha_shape* shape, const void* q, const void* K, const int32_t* seq_lens,
                                     int32_t m, int32_t* idx, int32_t idx_cap, int32_t* cnt, void* workspace,
                                     size_t ws_bytes, void* stream, void* const* events);

/*
 * Recall of one selection against a reference, per head:
 * recall[h] = |sel_h & ref_h| / |ref_h| (1 for an empty reference), with sel_h =
 * sel_idx[h, 0..sel_cnt[h]) and ref_h = ref_idx[h, 0..ref_cnt[h]) ascending
 * lists (counts clamped to [0, cap]); e.g. hashed selection vs exact top-k.
 *   sel_idx [heads, sel_cap], ref_idx [heads, ref_cap] int32; recall float32 [heads].
 * Errors: HA_ERR_INVALID_ARG before anything is enqueued; heads == 0 does nothing.
 */
ha_status hash_attn_recall(const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_cap, const int32_t* ref_idx,
                           const int32_t* ref_cnt, int32_t ref_cap, int32_t heads, float* recall, void* stream);

/*
 * Exact merge of nseg partial attentions over disjoint token sets, row by row
 * (Nectar Sec. 3: each segment enters the softmax as one virtual logit lse_s
 * with value out_s; Eq. (3.4) applied to every segment):
 * L = log sum_s e^{lse_s}, out = sum_s e^{lse_s - L} out_s. Segments with
 * lse = -inf contribute nothing; rows where all are -inf give out = 0,
 * lse = -inf. Composes a sparse document segment, a dense local segment and
 * generated-token segments in one call.
 *   outs  float32, segment s row r dim k at outs[s * out_seg_stride + r * d + k]
 *   lses  float32, segment s row r at lses[s * lse_seg_stride + r]
 *   out [rows, d], lse [rows] float32 (device). out may alias the rows of one
 *   segment (each element is read before it is written); lse likewise.
 *   nseg >= 1; out_seg_stride >= rows * d and lse_seg_stride >= rows.
 * Errors: HA_ERR_INVALID_ARG (null pointers, nseg < 1, rows < 0, d < 1,
 * strides that overlap segments) before anything is enqueued; rows == 0 does
 * nothing.
 */
ha_status hash_attn_merge_n(const float* outs, int64_t out_seg_stride, const float* lses,
                            int64_t lse_seg_stride, int32_t nseg, float* out, float* lse, int32_t rows,
                            int32_t d, void* stream);

/*
 * Synchronise `stream`, read and clear the workspace's device error word.
 * Returns HA_OK, HA_ERR_TIMEOUT (timeout flag set) or HA_ERR_DEVICE (any other
 * flag); *flags (optional) receives the raw HA_DEVERR_* bits.
 */
ha_status hash_attn_device_status(void* workspace, void* stream, uint32_t* flags);

/* Static description of a status code. */
const char* hash_attn_status_string(ha_status status);

/* Detail of the last failure on the calling thread ("" if none). */
const char* hash_attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* HASHATTN_H */
