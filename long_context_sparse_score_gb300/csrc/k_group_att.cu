// TOPK's masks and GATHER-ATT for a GQA group, over the union of its query
// heads' selected rows, with the contractions on tensor cores.
//
// HashAttention: Semantic Sparsity for Faster Inference, Sec. 4: each query head
// attends over its own selected set I (its min(m, n) nearest codes by Eq. (2),
// ties to the smaller index, plus the first n_sink and last n_local tokens,
// Sec. 4.4); o = sum_{i in I} e^{z_i} v_i / sum_{j in I} e^{z_j}. Nectar: Neural
// Estimation of Cached-Token Attention via Regression, Eqs. (3.4)-(3.5): partial
// results over disjoint token ranges merge exactly through their log-normalisers.
//
// k_group_att: one CTA (4 warps, three per SM) per (batch entry, KV head, range
// of 8,192 tokens), run after k_sel_scan, which has fixed every head's threshold
// bin t and each range's share of the ties. A CTA starts as soon as the scan's
// last CTA of its (batch entry, KV head) has set the pair's ready flag to the
// call's tag (a nonzero number no earlier call used).
//  1. Masks. Each thread recomputes the distances of two 32-token lane blocks
//     from the codes (one popcount per token and head; the codes' last read) and
//     builds every head's mask with one byte-wise compare pass against a per-head
//     threshold word (t - 1, or t for a head that takes its whole bin t here; a
//     second pass at t only in a head's boundary range, whose ties are ranked in
//     token order), adds the windows, and checks each head's count against the
//     scan's. The union of the heads' masks becomes a list in token order, one word
//     per row (offset in the range | head bits << 16): its first entries in shared
//     memory, the rest in the workspace.
//  2. Attention. The union is cut into chunks of 16 rows; warp w takes chunks
//     w, w + 4, ... and runs its own two-stage ring of 16-byte asynchronous copies
//     (a K row and its V row per chunk row, each read once for the whole group,
//     with an L2 evict-first policy). Per chunk, S = K Q^T (16 rows x 8 head
//     columns, heads beyond the group zero) and O^T += V^T P^T are mma.sync
//     m16n8k16 products with bf16 operands and fp32 accumulation: the products of
//     bf16 values are exact, P is passed as two bf16 parts (p = hi + lo, relative
//     error below 2^-16) so P.V keeps fp32 accuracy. A row outside a head's own set
//     gets score -inf for that head: each head attends over exactly its own rows.
//     The softmax is online in base 2 per (warp, head).
//  3. The warps combine in shared memory into the range's partial (max, sum, o)
//     per head; the last CTA of a (batch entry, KV head) to arrive merges the
//     ranges of its heads (an arrival counter decides; nothing waits), with each
//     head's maximum and part weights found once, in shared memory.
// When the grid would not give every SM a CTA, two CTAs share a range, each with
// a contiguous half of its chunks (both build the masks), and each CTA has eight
// warps with three-stage rings (one CTA per SM; the list's first 5,248 entries
// in shared memory for d = 128, all of them for d = 64).
// K/V must be finite: a row selected by one head of the group is also multiplied
// (by weight zero) into the other heads' P.V.
// The dense path (I = every token; HashAttention Sec. 4 with m >= n) runs the
// same kernel without step 1: a range's tokens are its rows, all heads' bits
// set, cut into spans of chunks (group_dense_splits CTAs per range), and no scan
// precedes it.
#include "ha_internal.cuh"
#include "sel_common.cuh"

#include <math_constants.h>

namespace ha {
namespace {

constexpr int kLB = kFusedRange / 32;    // lane blocks of 32 tokens per range
constexpr int kCR = 16;                  // union rows per warp chunk

// NW warps per CTA: 4 (three CTAs per SM) or 8 (one CTA per SM, for grids that
// give no SM a second CTA: half the serial mask work and chunks per warp)
template <int D, int ST, int NW>
struct GCfg {
    static constexpr int GW = NW;                      // warps
    static constexpr int GT = 32 * NW;                 // threads
    static constexpr int IT = kLB / GT;                // lane blocks per thread
    static_assert(kLB % GT == 0, "whole lane blocks per thread");
    static constexpr int RB = 2 * D;                   // bytes of a bf16 row
    static constexpr int PITCH = RB + 16;              // 8 rows of an ldmatrix land on distinct banks
    static constexpr int NCH = RB / 16;                // 16-byte chunks per row
    static constexpr int RPI = 32 / (2 * NCH);         // chunk rows per copy instruction of the warp
    static constexpr int STAGE = 2 * kCR * PITCH;      // K rows, then V rows
    static constexpr int RING = GW * ST * STAGE;
    static constexpr int KS = D / 16;                  // k-steps of K Q^T, m-tiles of V^T P^T
    static constexpr int MINB = (NW > 4) ? 1 : ((ST >= 3) ? 2 : 3);  // CTAs per SM
    static constexpr int OFF_HB = RING;                // int [GW][ST][kCR] head bits of the ring's rows
    static constexpr int OFF_LST = OFF_HB + GW * ST * kCR * 4;  // uint32 [LCAP] the list's first entries
    // what the shared memory of an SM leaves a CTA beside MINB - 1 others (228 KB,
    // 1 KB reserved per CTA, the static arrays), in 16-entry chunks
    static constexpr int SMEM_CTA = (228 * 1024) / MINB - 1024 - 1024;
    static constexpr int LCAP_FIT = ((SMEM_CTA - OFF_LST) / 4) / kCR * kCR;
    static constexpr int LCAP = LCAP_FIT < kFusedRange ? LCAP_FIT : kFusedRange;
    static constexpr int BYTES = OFF_LST + LCAP * 4;
    static_assert(LCAP >= kCR, "room for a list chunk in shared memory");
    // combine area (reuses the ring): o [GW][4][D], m [GW][4], l [GW][4]
    static_assert((GW * 4 * D + 2 * GW * 4) * 4 <= RING, "combine fits in the ring");
    static_assert(RPI * 2 * NCH == 32, "whole rows per copy instruction");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// c += A B for one m16n8k16 tile (A row-major 16 x 16, B column-major 16 x 8, bf16; c fp32).
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8 x 8 matrix of 16-bit elements held one element pair per lane.
__device__ __forceinline__ uint32_t movt(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// The bf16 parts of (a, b): hi = round(x), lo = round(x - hi).
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(a, b);
    lo = pack_bf16(a - bf16lo(hi), b - bf16hi(hi));
}

// 16-byte copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void cp_async16_pol(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// DENSE: every token of the range is a row of every head of the group (no codes,
// no scan, no masks); the rows of a range are cut into contiguous spans of chunks.
template <int D, int ST, bool DENSE, int NW>
__global__ void __launch_bounds__(32 * NW, GCfg<D, ST, NW>::MINB) k_group_att(const GroupAttParams gp) {
    using C = GCfg<D, ST, NW>;
    constexpr int kGT = C::GT, kGW = C::GW, kIt = C::IT;
    const FusedSelParams& p = gp.sel;
    const GatherParams& a = gp.att;
    extern __shared__ __align__(128) unsigned char smem[];
    int* s_hb = reinterpret_cast<int*>(smem + C::OFF_HB);
    uint32_t* s_lst = reinterpret_cast<uint32_t*>(smem + C::OFF_LST);
    __shared__ int s_wt[kIt][4][kGW];   // ties per (iteration, head, warp)
    __shared__ int s_wc[kIt][4][kGW];   // selected tokens per (iteration, head, warp)
    __shared__ int s_wu[kIt][kGW];      // union rows per (iteration, warp)
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // CTA order: batch entry fastest, so that the CTAs of one (KV head, range) of a
    // cache shared by the batch run together and share its rows in L2
    const int S = gp.nsplit;
    int lin = blockIdx.x;
    const int b = lin % p.B;
    lin /= p.B;
    const int split = lin % S;
    lin /= S;
    const int range = lin % p.nranges;
    const int g = lin / p.nranges;
    const int pair = b * p.Hkv + g;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, range == 0 && g == 0 && split == 0 && tid == 0);
    // ranges past the sequence's end hold no rows: their CTAs leave at once, and
    // the pair's parts are those of the live ranges (range 0 always runs)
    const int live = max(1, (n + kFusedRange - 1) / kFusedRange);
    if (range >= live) return;
    const int lo = range * kFusedRange;
    const int head0 = b * p.Hq + g * p.G;
    const int nh = p.G;  // at most 4 (checked on the host)
    const int wlo = min(p.n_sink, n);
    const int wmid = max(max(0, n - p.n_local), wlo);

    // ---- inputs (read before waiting for the scan): query codes and the query as
    // the B operand of S = K Q^T: lane holds head lane / 4, dims 2 (lane % 4) + {0, 1}
    // (b0) and 8 + 2 (lane % 4) + {0, 1} (b1) of every 16-dim k-step
    uint32_t qs[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) qs[e] = (!DENSE && e < nh) ? p.q_sig[head0 + e] : 0u;
    uint32_t qb[C::KS][2];
    {
        const int hq = lane >> 2, qq = lane & 3;
        const uint16_t* q16 =
            reinterpret_cast<const uint16_t*>(a.q) + (int64_t)b * a.q_sb + (int64_t)(g * p.G + min(hq, nh - 1)) * a.q_sh;
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
            const int d0 = ks * 16 + 2 * qq;
            qb[ks][0] = (hq < nh) ? ((uint32_t)q16[d0] | ((uint32_t)q16[d0 + 1] << 16)) : 0u;
            qb[ks][1] = (hq < nh) ? ((uint32_t)q16[d0 + 8] | ((uint32_t)q16[d0 + 9] << 16)) : 0u;
        }
    }
    pdl_launch_dependents();
    // The packed distances of lane block `it` of this thread (head e in byte e): the
    // codes and the query codes alone. With eight warps (small grids, where the
    // wait is on the critical path) the first block's come before the wait; with
    // four, the registers are kept for the attention loop.
    const uint32_t* crow = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)kv_head(g, p.kv_mul) * p.ks_sh;
    auto distances = [&](int it, uint32_t (&Dw)[32]) {
        const int lb = lo + (it * kGT + tid) * 32;
        const uint32_t valid = low_bits(n - lb);
        if (valid == 0u) return;
        if (valid == 0xffffffffu) {
            // lb + 32 <= n <= n_cap and lb is a multiple of 32: whole 16-byte loads in the row
            // the codes' last read: streaming (evict first)
            const uint4* src = reinterpret_cast<const uint4*>(crow + lb);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 v = __ldcs(src + j);
                Dw[4 * j + 0] = v.x;
                Dw[4 * j + 1] = v.y;
                Dw[4 * j + 2] = v.z;
                Dw[4 * j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) Dw[j] = ((valid >> j) & 1u) ? crow[lb + j] : 0u;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t c = Dw[j];
            uint32_t w = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nh) w |= (uint32_t)__popc(qs[e] ^ c) << (8 * e);
            Dw[j] = w;
        }
    };
    constexpr bool kEarly = !DENSE && NW > 4;
    uint32_t D0[32];
    if constexpr (kEarly) distances(0, D0);
    // The scan's thresholds and shares of this pair: its last CTA sets ready[pair]
    // to this call's tag after writing them, so the pairs that are done start while
    // the scan drains. This grid may start while the previous call's group kernel
    // still runs (each kernel lets the next one start early), whose pairs' flags
    // hold that call's tag until its last CTAs reset them: only this call's tag
    // counts. Every scan CTA is resident before this grid starts (programmatic
    // launch), so the flag comes; the wait is bounded all the same.
    __shared__ int s_go;
    if (DENSE) {
        // nothing to wait for before the copies: the inputs are the caller's, and the
        // partials and counters are written after the wait below
    } else if (p.ready != nullptr) {
        if (tid == 0) {
            int ok = 0;
            const unsigned long long t0 = global_ns();
            for (uint32_t it = 0;; ++it) {
                uint32_t v;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.ready + pair) : "memory");
                if (v == p.epoch) {
                    ok = 1;
                    break;
                }
                if ((it & 15u) == 15u && global_ns() - t0 > kWaitLimitNs) break;
                __nanosleep(200);
            }
            if (!ok) flag_error(p.err, HA_DEVERR_TIMEOUT);
            s_go = ok;
        }
        __syncthreads();
        if (!s_go) {
            pdl_wait();
            return;
        }
    } else {
        pdl_wait();
    }

    // ---- 1. masks
    uint32_t msk[kIt][4], uni[kIt];
    int uex[kIt], expect[4];
    int U = 0;
    if constexpr (DENSE) {
        U = max(0, min(n - lo, kFusedRange));  // the range's tokens, in order
    } else {
    int T[4], Tsel[4], qv[4], mode[4];
    bool any2 = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        T[e] = 0;
        qv[e] = 0;
        expect[e] = 0;
        mode[e] = 0;
        if (e < nh && lo < n) {
            const int2 mt = __ldcg(p.meta_t + pair * 4 + e);
            const int4 m4 = __ldcg(p.meta_r + ((int64_t)pair * p.nranges + range) * 4 + e);
            T[e] = mt.x;
            qv[e] = m4.y;
            expect[e] = m4.w;
            mode[e] = (m4.y <= 0) ? 0 : (m4.y >= m4.z ? 1 : 2);
        }
        Tsel[e] = (mode[e] == 1) ? T[e] : T[e] - 1;  // all of bin t, or only below it
        any2 = any2 || mode[e] == 2;
    }
    uint32_t eqm[kIt][4], validv[kIt], winv[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int lb = lo + (it * kGT + tid) * 32;  // this thread's lane block
        const uint32_t valid = low_bits(n - lb);
        const uint32_t win = low_bits(wlo - lb) | ~low_bits(wmid - lb);
        uint32_t m1[4] = {0u, 0u, 0u, 0u}, le[4] = {0u, 0u, 0u, 0u};
        if (valid != 0u) {
            uint32_t Dw[32];
            if (kEarly && it == 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) Dw[j] = D0[j];
            } else {
                distances(it, Dw);
            }
            le_masks(Dw, thresh_word(Tsel, nh), m1);
            if (any2) le_masks(Dw, thresh_word(T, nh), le);  // the ties of a boundary range
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            msk[it][e] = m1[e];
            uint32_t eq = le[e] & ~m1[e] & valid;
            if (p.excl) eq &= ~win;
            eqm[it][e] = (mode[e] == 2) ? eq : 0u;
        }
        validv[it] = valid;
        winv[it] = win;
    }
    if (any2) {
        // a head's boundary range: its first qv ties in token order (lane blocks in
        // the order it * kGT + tid)
#pragma unroll
        for (int it = 0; it < kIt; ++it)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t c = warp_sum_u((uint32_t)__popc(eqm[it][e]));
                if (lane == 0) s_wt[it][e][warp] = (int)c;
            }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < kIt; ++it)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (mode[e] == 2) {
                    int before = 0;
                    for (int i2 = 0; i2 < kIt; ++i2)
                        for (int w2 = 0; w2 < kGW; ++w2)
                            if (i2 < it || (i2 == it && w2 < warp)) before += s_wt[i2][e][w2];
                    int tot;
                    const int ex = warp_excl_scan(__popc(eqm[it][e]), &tot);
                    msk[it][e] |= first_bits(eqm[it][e], qv[e] - before - ex);
                }
            }
    }
    // ---- the union of the heads' masks: its rows go to a list in token order,
    // entry = offset in the range | head bits << 16
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        uint32_t u = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t m = (e < nh) ? ((msk[it][e] | winv[it]) & validv[it]) : 0u;
            msk[it][e] = m;
            u |= m;
            const uint32_t c = warp_sum_u((uint32_t)__popc(m));
            if (lane == 0) s_wc[it][e][warp] = (int)c;
        }
        uni[it] = u;
        int tot;
        uex[it] = warp_excl_scan(__popc(u), &tot);
        if (lane == 0) s_wu[it][warp] = tot;
    }
    __syncthreads();
    // The list's first LCAP entries live in shared memory, the rest in the distance
    // buffer's row of this (batch entry, KV head), at the range's offset: the range
    // holds at least as many tokens as list entries, and
    // range * 8192 + (tokens of the range) <= n <= n_cap <= d_sp.
    // Split `split` of S takes chunks [c0, c1) of the range's union and writes only
    // their entries (the splits of a range write disjoint parts of the list).
    for (int i2 = 0; i2 < kIt; ++i2)
        for (int w2 = 0; w2 < kGW; ++w2) U += s_wu[i2][w2];
    }
    uint32_t* lst = p.dist + (int64_t)pair * p.d_sp + (int64_t)range * kFusedRange;
    const int nch = (U + kCR - 1) / kCR;
    const int c0 = (int)((int64_t)split * nch / S), c1 = (int)((int64_t)(split + 1) * nch / S);
    if constexpr (!DENSE) {
    const int p0 = c0 * kCR, p1 = min(U, c1 * kCR);
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        int pos = uex[it];
        for (int i2 = 0; i2 < kIt; ++i2)
            for (int w2 = 0; w2 < kGW; ++w2)
                if (i2 < it || (i2 == it && w2 < warp)) pos += s_wu[i2][w2];
        const int off0 = (it * kGT + tid) * 32;
        uint32_t u = uni[it];
        if (pos >= p1 || pos + __popc(u) <= p0) continue;  // none of this lane block's entries
        while (u != 0u) {
            const int bit = __ffs(u) - 1;
            u &= u - 1u;
            if (pos >= p0 && pos < p1) {
                uint32_t hb = 0u;
#pragma unroll
                for (int e = 0; e < 4; ++e) hb |= ((msk[it][e] >> bit) & 1u) << e;
                const uint32_t v = (uint32_t)(off0 + bit) | (hb << 16);
                if (pos < C::LCAP)
                    s_lst[pos] = v;
                else
                    lst[pos] = v;
            }
            ++pos;
        }
    }
    if (split == 0 && tid < nh) {
        int mine = 0;
        for (int i2 = 0; i2 < kIt; ++i2)
            for (int w2 = 0; w2 < kGW; ++w2) mine += s_wc[i2][tid][w2];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e == tid && mine != expect[e]) flag_error(p.err, HA_DEVERR_STATE);  // masks disagree with the scan
    }
    __syncthreads();  // the list is written (block-scope visibility)
    }

    // ---- 2. attention over the union, per warp
    const int ncw = (c1 - c0 > warp) ? (c1 - c0 - warp + kGW - 1) / kGW : 0;
    unsigned char* ring = smem + warp * ST * C::STAGE;
    int* whb = s_hb + warp * ST * kCR;
    // this lane's share of every copy: chunk `ch` of the K or V row `sub` of each
    // group of RPI chunk rows (coalesced: consecutive lanes read consecutive 16 bytes)
    const int sub = lane / (2 * C::NCH);
    const int rem = lane - sub * (2 * C::NCH);
    const int isv = rem >= C::NCH ? 1 : 0;
    const int ch = rem - isv * C::NCH;
    const int gk = kv_head(g, a.kv_mul);  // the KV head of this query-head group
    const char* cbase = (isv ? a.V + ((int64_t)b * a.v_sb + (int64_t)gk * a.v_sh) * 2
                             : a.K + ((int64_t)b * a.k_sb + (int64_t)gk * a.k_sh) * 2) + ch * 16;
    const int cstep = (int)(isv ? a.v_sn * 2 : a.k_sn * 2);  // < 2^31 (checked on the host)
    const uint32_t cdst = (uint32_t)((isv * kCR + sub) * C::PITCH + ch * 16);
    // K/V rows are read once per group: evict first, so that the codes (read again
    // by later CTAs) and the selection's small buffers keep their L2 lines
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));

    // list entries of chunk k of this warp (lanes 0-15); past the union: the range's
    // first token with no head bits (its rows are read and then masked out)
    auto entry = [&](int k) -> uint32_t {
        const int pos = (c0 + warp + k * kGW) * kCR + lane;
        if (lane >= kCR || k >= ncw || pos >= U) return 0u;
        if constexpr (DENSE) return (uint32_t)pos | (((1u << nh) - 1u) << 16);
        return pos < C::LCAP ? s_lst[pos] : lst[pos];
    };
    auto issue = [&](int k, uint32_t ent) {
        const int slot = k % ST;
        // a row outside the sequence only if the workspace was disturbed: never read
        // it (the range's first row instead, with no head bits)
        if (lo + (int)(ent & 0xffffu) >= n) {
            flag_error(p.err, HA_DEVERR_STATE);
            ent = 0u;
        }
        if (lane < kCR) whb[slot * kCR + lane] = (int)(ent >> 16);
        const int tok = lo + (int)(ent & 0xffffu);
        const uint32_t sbase = smem_addr(ring + slot * C::STAGE) + cdst;
#pragma unroll
        for (int j = 0; j < kCR / C::RPI; ++j) {
            const int tr = __shfl_sync(0xffffffffu, tok, j * C::RPI + sub);
            cp_async16_pol(sbase + j * C::RPI * C::PITCH, cbase + (int64_t)tr * cstep, pol);
        }
    };

    // O^T accumulators: m-tile mt holds dims mt * 16 + lane / 4 (+ 8) for heads
    // 2 (lane % 4) and 2 (lane % 4) + 1 (heads >= nh stay zero)
    float o[C::KS][4];
#pragma unroll
    for (int mt = 0; mt < C::KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float mr0 = -CUDART_INF_F, mr1 = -CUDART_INF_F, lr0 = 0.f, lr1 = 0.f;
    const int e0 = 2 * (lane & 3), e1 = e0 + 1;
    const int mi = lane >> 3, r8 = lane & 7;
    // ldmatrix row addresses: K as the A operand (matrices: rows 0-7 / 8-15 x dims 0-7,
    // then dims 8-15), V transposed as the A operand (rows 0-7 x dims 0-7 / 8-15, then
    // rows 8-15)
    const uint32_t koff = (uint32_t)((r8 + (mi & 1) * 8) * C::PITCH + (mi >> 1) * 16);
    const uint32_t voff = (uint32_t)((r8 + (mi >> 1) * 8) * C::PITCH + (mi & 1) * 16);

    uint32_t ent = entry(0);
#pragma unroll
    for (int k = 0; k < ST - 1; ++k) {
        if (k < ncw) {
            const uint32_t nxt = entry(k + 1);
            issue(k, ent);
            ent = nxt;
        }
        commit_group();
    }
    for (int k = 0; k < ncw; ++k) {
        if (k + ST - 1 < ncw) {
            const uint32_t nxt = entry(k + ST);
            issue(k + ST - 1, ent);
            ent = nxt;
        }
        commit_group();
        wait_group<ST - 1>();
        __syncwarp();
        const int slot = k % ST;
        const uint32_t kbase = smem_addr(ring + slot * C::STAGE);
        const uint32_t vbase = kbase + kCR * C::PITCH;

        // S = K Q^T: c0/c1 row lane/4 heads e0/e1, c2/c3 row lane/4 + 8
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kbase + koff + ks * 32, a0, a1, a2, a3);
            if (ks & 1)
                mma16816(s1, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            else
                mma16816(s0, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        }
        const int hbA = whb[slot * kCR + (lane >> 2)];
        const int hbB = whb[slot * kCR + (lane >> 2) + 8];
        const float x0 = ((hbA >> e0) & 1) ? (s0[0] + s1[0]) * a.qscale : -CUDART_INF_F;
        const float x1 = ((hbA >> e1) & 1) ? (s0[1] + s1[1]) * a.qscale : -CUDART_INF_F;
        const float x2 = ((hbB >> e0) & 1) ? (s0[2] + s1[2]) * a.qscale : -CUDART_INF_F;
        const float x3 = ((hbB >> e1) & 1) ? (s0[3] + s1[3]) * a.qscale : -CUDART_INF_F;
        float t0 = fmaxf(x0, x2), t1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
            t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
        }
        const float mn0 = fmaxf(mr0, t0), mn1 = fmaxf(mr1, t1);
        if (__any_sync(0xffffffffu, mn0 != mr0 || mn1 != mr1)) {
            // a running maximum rose: rescale (no row yet keeps every term at 0)
            const float al0 = exp2f(mr0 - ((mn0 == -CUDART_INF_F) ? 0.f : mn0));
            const float al1 = exp2f(mr1 - ((mn1 == -CUDART_INF_F) ? 0.f : mn1));
            lr0 *= al0;
            lr1 *= al1;
#pragma unroll
            for (int mt = 0; mt < C::KS; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            mr0 = mn0;
            mr1 = mn1;
        }
        const float mb0 = (mr0 == -CUDART_INF_F) ? 0.f : mr0;
        const float mb1 = (mr1 == -CUDART_INF_F) ? 0.f : mr1;
        const float p0 = exp2f(x0 - mb0), p2 = exp2f(x2 - mb0);
        const float p1 = exp2f(x1 - mb1), p3 = exp2f(x3 - mb1);
        lr0 += p0 + p2;
        lr1 += p1 + p3;
        // P^T as the B operand: the lane's (row, head pair) entries are one element
        // pair of the 8 x 8 blocks rows 0-7 / 8-15 x heads 0-7; their transposes are
        // the fragments b0 / b1 (head lane / 4, rows 2 (lane % 4) + {0, 1} (+ 8))
        uint32_t hA, lA, hB, lB;
        split_bf16(p0, p1, hA, lA);
        split_bf16(p2, p3, hB, lB);
        const uint32_t bh0 = movt(hA), bh1 = movt(hB), bl0 = movt(lA), bl1 = movt(lB);
#pragma unroll
        for (int mt = 0; mt < C::KS; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vbase + voff + mt * 32, a0, a1, a2, a3);
            mma16816(o[mt], a0, a1, a2, a3, bh0, bh1);
            mma16816(o[mt], a0, a1, a2, a3, bl0, bl1);
        }
        __syncwarp();  // the stage is read before it is refilled
    }
    wait_group<0>();
    // the whole scan grid has completed long before: this orders the next kernel
    // in the stream after it (dense: the previous kernel in the stream is done with
    // the partials and counters before this CTA writes them)
    pdl_wait();

    // ---- 3. combine the warps, then the ranges
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        lr0 += __shfl_xor_sync(0xffffffffu, lr0, off);
        lr1 += __shfl_xor_sync(0xffffffffu, lr1, off);
    }
    __syncthreads();  // every warp is done with its ring
    float* cw = reinterpret_cast<float*>(smem);   // [kGW][4][D]
    float* cm = cw + kGW * 4 * D;                 // [kGW][4]
    float* cl = cm + kGW * 4;                     // [kGW][4]
    if ((lane & 3) < 2) {
#pragma unroll
        for (int mt = 0; mt < C::KS; ++mt) {
            const int dA = mt * 16 + (lane >> 2), dB = dA + 8;
            cw[(warp * 4 + e0) * D + dA] = o[mt][0];
            cw[(warp * 4 + e1) * D + dA] = o[mt][1];
            cw[(warp * 4 + e0) * D + dB] = o[mt][2];
            cw[(warp * 4 + e1) * D + dB] = o[mt][3];
        }
        if (lane < 2) {
            cm[warp * 4 + e0] = mr0;
            cm[warp * 4 + e1] = mr1;
            cl[warp * 4 + e0] = lr0;
            cl[warp * 4 + e1] = lr1;
        }
    }
    __syncthreads();
    constexpr float kLn2 = 0.69314718055994530942f;
    const int nparts = p.nranges * S;  // partials per head (the stride of a head's parts)
    const int nlive = live * S;        // the parts this pair's live ranges write
    for (int x = tid; x < nh * D; x += kGT) {
        const int e = x / D, dd = x - e * D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kGW; ++w) M = fmaxf(M, cm[w * 4 + e]);
        float Ls = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kGW; ++w) {
                const float mw = cm[w * 4 + e];
                if (mw != -CUDART_INF_F) {
                    const float sc = exp2f(mw - M);
                    Ls += cl[w * 4 + e] * sc;
                    O += cw[(w * 4 + e) * D + dd] * sc;
                }
            }
        }
        const int64_t head = head0 + e;
        if (nlive == 1) {
            a.out[head * D + dd] = (Ls > 0.f) ? O / Ls : 0.f;
            if (dd == 0) a.lse[head] = (Ls > 0.f) ? (M + log2f(Ls)) * kLn2 : -CUDART_INF_F;
        } else {
            float* pt = a.part + (head * nparts + range * S + split) * (D + 2);
            pt[2 + dd] = O;
            if (dd == 0) {
                pt[0] = M;
                pt[1] = Ls;
            }
        }
    }
    if (nlive == 1) {
        if (tid == 0 && p.ready != nullptr) p.ready[pair] = 0u;
        return;
    }

    __syncthreads();  // every partial store of this CTA precedes thread 0's fence
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&a.counters[pair], 1u);
        if (prev >= (unsigned)nlive) flag_error(p.err, HA_DEVERR_STATE);
        s_last = (prev == (unsigned)(nlive - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Merge the pair's parts per head (Nectar Eq. (3.4)). One warp per head finds
    // the head's maximum over all parts, then, for blocks of up to kMB parts, each
    // part's weight 2^(m_r - M) once (in the ring's shared memory, free again), and
    // every (head, dim) reads only the block's outputs: loads that depend on no
    // branch, all in flight together.
    constexpr int kMB = 64;                                // parts per block
    constexpr int kItems = (4 * D + kGT - 1) / kGT;        // (head, dim) outputs per thread
    static_assert((4 * kMB + 8) * 4 <= C::RING, "a block's weights fit the ring");
    float* s_w = reinterpret_cast<float*>(smem);           // [4][kMB] weights
    float* s_ml = s_w + 4 * kMB;                           // M [4], L [4]
    if (warp < nh) {
        const float* ph = a.part + (int64_t)(head0 + warp) * nparts * (D + 2);
        float M = -CUDART_INF_F;
        for (int r = lane; r < nlive; r += 32) M = fmaxf(M, __ldcg(ph + (int64_t)r * (D + 2)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        if (lane == 0) s_ml[warp] = M;
    }
    float O[kItems];
#pragma unroll
    for (int i = 0; i < kItems; ++i) O[i] = 0.f;
    float Ls = 0.f;  // per lane of the head's warp
    for (int r0 = 0; r0 < nlive; r0 += kMB) {
        const int rn = min(kMB, nlive - r0);
        __syncthreads();  // the maxima are written; the previous block's weights are read
        if (warp < nh) {
            const float M = s_ml[warp];
            const float* ph = a.part + ((int64_t)(head0 + warp) * nparts + r0) * (D + 2);
            for (int r = lane; r < rn; r += 32) {
                const float mr = __ldcg(ph + (int64_t)r * (D + 2)), lr = __ldcg(ph + (int64_t)r * (D + 2) + 1);
                const float w = (mr != -CUDART_INF_F) ? exp2f(mr - M) : 0.f;  // an empty part adds nothing
                s_w[warp * kMB + r] = w;
                Ls += (w != 0.f) ? w * lr : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            const int x = tid + i * kGT;
            if (x < nh * D) {
                const int e = x / D, dd = x - e * D;
                const float* po = a.part + ((int64_t)(head0 + e) * nparts + r0) * (D + 2) + 2 + dd;
                const float* we = s_w + e * kMB;
                float acc = 0.f;
#pragma unroll 8
                for (int r = 0; r < rn; ++r) {
                    const float w = we[r], o = __ldcg(po + (int64_t)r * (D + 2));
                    acc += (w != 0.f) ? w * o : 0.f;
                }
                O[i] += acc;
            }
        }
    }
    if (warp < nh) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
        if (lane == 0) s_ml[4 + warp] = Ls;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const int x = tid + i * kGT;
        if (x < nh * D) {
            const int e = x / D, dd = x - e * D;
            const int64_t head = head0 + e;
            const float M = s_ml[e], L = s_ml[4 + e];
            a.out[head * D + dd] = (L > 0.f) ? O[i] / L : 0.f;
            if (dd == 0) a.lse[head] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
        }
    }
    if (tid == 0) {
        a.counters[pair] = 0u;
        if (p.ready != nullptr) p.ready[pair] = 0u;
    }
}

template <int D, int ST, bool DENSE, int NW>
cudaError_t launch_group_t(const GroupAttParams& p, int batch_hkv, cudaStream_t st, bool pdl) {
    using C = GCfg<D, ST, NW>;
    cudaError_t e =
        cudaFuncSetAttribute(k_group_att<D, ST, DENSE, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)batch_hkv * (unsigned)p.sel.nranges * (unsigned)p.nsplit;
    return launch_ex(k_group_att<D, ST, DENSE, NW>, dim3(grid), dim3(C::GT), (size_t)C::BYTES, st, pdl, p);
}

}  // namespace

int group_splits(int64_t pair_ranges) {
    // every split repeats the range's mask phase: two only when the grid would
    // not give each SM a CTA
    return pair_ranges < kSMs ? 2 : 1;
}

bool group_att_supported(int d, int kv_bf16, int q_bf16, int G) {
    return kv_bf16 && q_bf16 && (d == 64 || d == 128) && G >= 1 && G <= 4;
}

cudaError_t launch_group_att(const GroupAttParams& p, int d, int batch_hkv, cudaStream_t st, bool pdl) {
    if (p.nsplit < 1) return cudaErrorInvalidValue;
    // eight warps per CTA when the grid leaves SMs without a CTA
    const bool wide = (int64_t)batch_hkv * p.sel.nranges * p.nsplit < kSMs;
    if (d == 128) return wide ? launch_group_t<128, 3, false, 8>(p, batch_hkv, st, pdl)
                              : launch_group_t<128, 2, false, 4>(p, batch_hkv, st, pdl);
    if (d == 64) return wide ? launch_group_t<64, 3, false, 8>(p, batch_hkv, st, pdl)
                             : launch_group_t<64, 2, false, 4>(p, batch_hkv, st, pdl);
    return cudaErrorInvalidValue;
}

int group_dense_splits(int64_t batch_hkv, int n_cap) {
    // spans of about 2,048 rows; fewer per range when a head would get more than
    // 64 partials, more while the grid would not give each SM two CTAs
    const int64_t nr = fused_ranges(n_cap);
    const int r = std::min(n_cap, kFusedRange);
    int s = std::max(1, r / 2048);
    while (s > 1 && nr * s > 64) s /= 2;
    while (s < 16 && batch_hkv * nr * s < 2 * kSMs && r / (2 * s) >= 256) s *= 2;
    return s;
}

cudaError_t launch_group_dense(const GroupAttParams& p, int d, int batch_hkv, cudaStream_t st, bool pdl) {
    if (p.nsplit < 1 || p.sel.ready != nullptr) return cudaErrorInvalidValue;
    if (d == 128) return launch_group_t<128, 2, true, 4>(p, batch_hkv, st, pdl);
    if (d == 64) return launch_group_t<64, 2, true, 4>(p, batch_hkv, st, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace ha
