// SCORE and TOPK with one popcount per (token, query head): two kernels.
//
// HashAttention: Semantic Sparsity for Faster Inference, Eq. (2): a cached
// token's score is the negated Hamming distance between its 32-bit key code and
// the query code; Sec. 4 keeps the min(m, n) best tokens (ties to the smaller
// index), Sec. 4.4 adds the first n_sink and the last n_local tokens. One read
// of a KV head's codes serves all its query heads (Nectar Sec. 3, GQA sharing).
//
// The n tokens of one (batch entry b, KV head g) are split into ranges of
// R = 8192 (one CTA of 256 threads each in both kernels).
//   k_sel_scan  reads every code of its range once (16-byte loads, four rounds in
//               flight per thread) and computes the distances to the (up to
//               four) query heads once; it writes them as one packed word per
//               token (head e in byte e) to a buffer that stays in L2, counts them
//               into a 33-bin histogram per head (shared-memory columns indexed by
//               lane) and publishes exclusive prefix sums of that histogram and of
//               the sink and local window parts of its range. The last CTA of a
//               (batch entry, KV head) to finish then derives, per head, the
//               threshold bin t (smallest t whose cumulative count reaches k) and,
//               for every range, how many tied tokens (distance t) it takes (none,
//               all, or the first q in token order) and how many tokens it
//               selects, hence where its part of the ascending list starts.
//   k_sel_emit  gives each lane 32 consecutive tokens: it reads their packed
//               distances (one 128-byte line, eight 16-byte loads), builds its
//               selection mask for all heads at once with byte-wise compares (no
//               further popcounts), ORs in the windows as bit ranges, ranks the
//               boundary range's ties across warps and lanes, writes its tokens
//               into the flat lists and drops the line from L2 without writing it
//               back to memory.
#include "ha_internal.cuh"
#include "sel_common.cuh"

namespace ha {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelRange = kFusedRange;      // tokens per CTA (32 per thread)
static_assert(kSelRange == 32 * kSelThreads, "one 32-token lane block per thread");
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kCum = HA_NBINS + 3;           // entries of a published prefix-sum array (0 .. 33 used)

// Budget of head h (per-head budgets override per-sequence ones, which override m;
// out-of-range budgets are clamped and flagged).
__device__ __forceinline__ int head_budget(const FusedSelParams& p, int b, int64_t h, bool report) {
    int mb = p.m;
    if (p.m_per_seq != nullptr) {
        mb = p.m_per_seq[b];
        if (mb < 0 || mb > p.m) {
            if (report) flag_error(p.err, HA_DEVERR_BUDGET);
            mb = min(max(mb, 0), p.m);
        }
    }
    if (p.m_per_head != nullptr) {
        mb = p.m_per_head[h];
        if (mb < 0 || mb > p.m) {
            if (report) flag_error(p.err, HA_DEVERR_BUDGET);
            mb = min(max(mb, 0), p.m);
        }
    }
    return mb;
}

// WD: write the packed distances for k_sel_emit; without them the window parts
// are recounted from the codes and the codes are read with the default cache
// policy (a later kernel reads them again). NHT: query heads per KV head known
// at compile time (4), or 0 for the runtime value p.G (1 to 4).
template <bool WD, int NHT>
__global__ void __launch_bounds__(kSelThreads, WD ? 5 : 8) k_sel_scan(const FusedSelParams p) {
    constexpr int NT = kSelThreads, R = kSelRange;
    constexpr int NR = R / (4 * NT);   // rounds of 4 tokens per thread
    constexpr int U = 4;               // rounds of codes in flight per thread
    __shared__ __align__(16) uint32_t hist[HA_NBINS][2][32];  // lane columns; heads 2k, 2k+1 in 16-bit fields
    __shared__ uint32_t s_h[3][4][HA_NBINS + 3];    // per head: all tokens, sink part, local part
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // CTA order: batch entry fastest, then range, then KV head, so that the pairs of
    // one KV head complete together (and a cache shared by the batch is read once)
    const int b = blockIdx.x % p.B, range = (blockIdx.x / p.B) % p.nranges, g = blockIdx.x / (p.B * p.nranges);
    const int pair = b * p.Hkv + g;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, range == 0 && g == 0 && tid == 0);
    // ranges past the sequence's end hold no tokens: they leave at once, and the
    // pair's last CTA counts only the live ones (range 0 always runs)
    if (range > 0 && range * R >= n) return;
    const int lo = min(n, range * R);
    const int hi = min(n, lo + R);
    const int head0 = b * p.Hq + g * p.G;
    const int nh = NHT > 0 ? NHT : p.G;  // at most 4 (checked on the host)
    const int wlo = min(p.n_sink, n);                   // sink window [0, wlo)
    const int wmid = max(max(0, n - p.n_local), wlo);   // local window [wmid, n)
    uint32_t* drow = p.dist + (int64_t)pair * p.d_sp;

    uint32_t qs[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) qs[e] = (e < nh) ? p.q_sig[head0 + e] : 0u;
    for (int x = tid; x < HA_NBINS * 2 * 32; x += NT) (&hist[0][0][0])[x] = 0u;
    for (int x = tid; x < 3 * 4 * (HA_NBINS + 3); x += NT) (&s_h[0][0][0])[x] = 0u;
    pdl_launch_dependents();
    __syncthreads();

    {
        const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)kv_head(g, p.kv_mul) * p.ks_sh;
        const uint32_t col = smem_addr(&hist[0][0][lane]);
        uint4 v[U];
        auto load = [&](int k) {
            const int i = lo + k * 4 * NT + 4 * tid;
            uint4 c;
            if (i + 4 <= hi) {
                // with the distances written, the codes are read once: evict first
                c = WD ? __ldcs(reinterpret_cast<const uint4*>(row + i)) : *reinterpret_cast<const uint4*>(row + i);
            } else {
                c.x = (i < hi) ? row[i] : 0u;
                c.y = (i + 1 < hi) ? row[i + 1] : 0u;
                c.z = (i + 2 < hi) ? row[i + 2] : 0u;
                c.w = (i + 3 < hi) ? row[i + 3] : 0u;
            }
            return c;
        };
        // one token: its distances to the heads into the histogram columns, packed
        auto count = [&](uint32_t code) {
            uint32_t w = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (NHT > 0 ? e < NHT : e < nh) {
                    const uint32_t d = (uint32_t)__popc(qs[e] ^ code);
                    red_add_shared(col + (d * 2 + (e >> 1)) * 128u, 1u << (16 * (e & 1)));
                    w |= d << (8 * e);
                }
            }
            return w;
        };
        auto compute = [&](const uint4 c4, int k) {
            const int i = lo + k * 4 * NT + 4 * tid;
            uint32_t pk[4] = {0u, 0u, 0u, 0u};
            if (i + 4 <= hi) {  // four whole tokens: no per-token checks
                pk[0] = count(c4.x);
                pk[1] = count(c4.y);
                pk[2] = count(c4.z);
                pk[3] = count(c4.w);
            } else if (i < hi) {
                const uint32_t code[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (i + j < hi) pk[j] = count(code[j]);
            } else {
                return;
            }
            // i is a multiple of 4 below n <= n_cap <= d_sp: the four words stay in the row
            if constexpr (WD) *reinterpret_cast<uint4*>(drow + i) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        };
#pragma unroll
        for (int k = 0; k < NR + U; ++k) {
            if (k >= U) compute(v[(k - U) % U], k - U);
            if (k < NR) v[k % U] = load(k);
        }
    }
    __syncthreads();  // the range's distances are written and visible to this CTA
    {
        // every (bin, head pair) row of 32 lane columns: 4 threads x 8 columns, then
        // 2 shuffles (bins 0-31); bin 32 by warp 0, 16 lanes x 2 columns per pair.
        // The 16-bit fields hold at most 8192 counts: no carries between heads.
        const int r = tid >> 2, q = tid & 3;
        const uint4* rp = reinterpret_cast<const uint4*>(&hist[0][0][0] + r * 32 + q * 8);
        const uint4 x0 = rp[0], x1 = rp[1];
        uint32_t v = (x0.x + x0.y) + (x0.z + x0.w) + (x1.x + x1.y) + (x1.z + x1.w);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (q == 0) {
            s_h[0][2 * (r & 1)][r >> 1] = v & 0xffffu;
            s_h[0][2 * (r & 1) + 1][r >> 1] = v >> 16;
        }
        if (warp == 0) {
            const int pr = lane >> 4;
            const uint2 y = *reinterpret_cast<const uint2*>(&hist[HA_NBINS - 1][pr][(lane & 15) * 2]);
            uint32_t t = y.x + y.y;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            if ((lane & 15) == 0) {
                s_h[0][2 * pr][HA_NBINS - 1] = t & 0xffffu;
                s_h[0][2 * pr + 1][HA_NBINS - 1] = t >> 16;
            }
        }
    }
    {
        // the window parts of this range: [lo, min(hi, wlo)) and [max(lo, wmid), hi)
        const int a0 = lo, a1 = min(hi, wlo), b0 = max(lo, wmid), b1 = hi;
        const int na = max(0, a1 - a0), nb = max(0, b1 - b0);
        const uint32_t* crow = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)kv_head(g, p.kv_mul) * p.ks_sh;
        for (int x = tid; x < na + nb; x += NT) {
            const int i = x < na ? a0 + x : b0 + (x - na);
            uint32_t w = 0u;
            if constexpr (WD) {
                w = drow[i];
            } else {
                const uint32_t c = crow[i];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (e < nh) w |= (uint32_t)__popc(qs[e] ^ c) << (8 * e);
            }
            const int which = (x < na) ? 1 : 2;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nh) atomicAdd(&s_h[which][e][(w >> (8 * e)) & 0xffu], 1u);
        }
    }
    // Launched with programmatic dependent launch, everything above (reads of the
    // codes, this CTA's shared memory) may overlap the previous kernel in the
    // stream; everything below writes state that the previous call's kernels may
    // still read (published sums, totals, shares), so wait for it here (every
    // kernel of the library waits for its own predecessor before it completes, so
    // this orders the calls).
    pdl_wait();
    __syncthreads();
    // exclusive prefix sums over the 33 bins, one warp per (head, histogram), published
    uint32_t* pub = p.rh + ((int64_t)pair * p.nranges + range) * (3 * 4 * kCum);
    for (int job = warp; job < 3 * nh; job += kSelWarps) {
        const int e = job % nh, which = job / nh;
        const uint32_t v = s_h[which][e][lane];
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        uint32_t* dst = pub + (which * 4 + e) * kCum;
        dst[lane] = x - v;
        if (lane == 31) {
            dst[32] = x;
            dst[33] = x + s_h[which][e][32];
        }
    }

    // this range's bins into the sequence's totals (with exclusive windows, the
    // window tokens leave the ranking)
    uint32_t* tot_g = p.tot + (int64_t)pair * 4 * kCum;
    for (int x = tid; x < nh * HA_NBINS; x += NT) {
        const int e = x / HA_NBINS, u = x % HA_NBINS;
        uint32_t v = s_h[0][e][u];
        if (p.excl) v -= s_h[1][e][u] + s_h[2][e][u];
        if (v != 0u) atomicAdd(tot_g + e * kCum + u, v);
    }

    // ---- the last CTA of this (batch entry, KV head) derives every range's share
    __syncthreads();  // every store of this CTA precedes thread 0's fence
    if (tid == 0) {
        __threadfence();
        const unsigned live = (unsigned)max(1, (n + R - 1) / R);  // the ranges that arrive
        const unsigned prev = atomicAdd(&p.arrive[pair], 1u);
        if (prev >= live) flag_error(p.err, HA_DEVERR_STATE);
        s_last = (prev == live - 1u) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Per head: the threshold bin t and the ties to take over the whole sequence,
    // then for every range r in order its share of those ties and the number of
    // tokens it selects.
    //   A = tokens of the range below t, T = its ties, P / S = the sink / local
    //   window parts of the range (below t: Pl / Sl, at t: Pt / St), q' = the
    //   range's taken ties (the first ones of the range in token order):
    //   selected = A + (|P| - Pl) + (|S| - Sl) + q' - |taken in P| - |taken in S|,
    //   |taken in P| = min(q', Pt) (P is a prefix), |taken in S| = max(0, q' - (T - St))
    //   (S is a suffix); with exclusive windows no window token is a tie:
    //   selected = (A - Pl - Sl) + q' + |P| + |S|, with T counting non-window ties.
    const int nr = (n + R - 1) / R;  // ranges holding tokens
    const uint32_t* rh = p.rh + (int64_t)pair * p.nranges * (3 * 4 * kCum);
    int4* mr = p.meta_r + (int64_t)pair * p.nranges * 4;
    if (warp < nh) {
        const int e = warp;
        const int64_t h = head0 + e;
        const int mb = head_budget(p, b, h, g == 0 && e == 0 && lane == 0 || (p.m_per_head != nullptr && lane == 0));
        const int nwin = wlo + (n - wmid);
        const int k = p.excl ? min(mb, n - nwin) : min(mb, n);
        // bin `lane` over the sequence, summed by every range's CTA (bin 32 is implied
        // by the total); cleared here for the next call once read
        const uint32_t tot = __ldcg(tot_g + e * kCum + lane);
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned reach = __ballot_sync(0xffffffffu, incl >= (uint32_t)k);
        const int t = reach ? (__ffs(reach) - 1) : 32;
        const uint32_t below = __shfl_sync(0xffffffffu, incl, (t == 0 ? 0 : t - 1) & 31);
        int left = k - (t == 0 ? 0 : (int)below);  // ties still to take, in token order
        int carry = 0;
        for (int r0 = 0; r0 < nr; r0 += 32) {
            const int r = r0 + lane;
            int A = 0, T = 0, Pl = 0, Pt = 0, NP = 0, Sl = 0, St = 0, NS = 0;
            if (r < nr) {
                const uint32_t* c = rh + (int64_t)r * (3 * 4 * kCum) + e * kCum;
                const uint32_t* cp = c + 4 * kCum;
                const uint32_t* cs = c + 8 * kCum;
                A = (int)__ldcg(c + t);
                T = (int)__ldcg(c + t + 1) - A;
                Pl = (int)__ldcg(cp + t);
                Pt = (int)__ldcg(cp + t + 1) - Pl;
                NP = (int)__ldcg(cp + HA_NBINS);
                Sl = (int)__ldcg(cs + t);
                St = (int)__ldcg(cs + t + 1) - Sl;
                NS = (int)__ldcg(cs + HA_NBINS);
            }
            if (p.excl) T -= Pt + St;
            int tsum;
            const int qr = min(max(left - warp_excl_scan(T, &tsum), 0), T);
            left -= tsum;
            int c = 0;
            if (r < nr) {
                c = p.excl ? (A - Pl - Sl) + qr + NP + NS
                           : A + (NP - Pl) + (NS - Sl) + qr - min(qr, Pt) - max(0, qr - (T - St));
            }
            int csum;
            const int base = carry + warp_excl_scan(c, &csum);
            carry += csum;
            if (r < nr) mr[(int64_t)r * 4 + e] = make_int4(base, qr, T, c);
        }
        if (lane == 0) p.meta_t[pair * 4 + e] = make_int2(t, carry);
    }
    __syncthreads();  // every warp has read the totals and written its shares
    for (int x = tid; x < 4 * kCum; x += NT) tot_g[x] = 0u;
    if (tid == 0) {
        p.arrive[pair] = 0u;
        if (p.ready != nullptr) {  // the shares of this pair are complete: this call's tag
            __threadfence();
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p.ready + pair), "r"(p.epoch) : "memory");
        }
    }
}

__global__ void __launch_bounds__(kSelThreads, 4) k_sel_emit(const FusedSelParams p) {
    constexpr int NT = kSelThreads, NW = kSelWarps, R = kSelRange;
    __shared__ int s_wt[4][NW];   // ties per warp (the head's boundary range)
    __shared__ int s_wc[4][NW];   // selected tokens per warp

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pair = blockIdx.x / p.nranges, range = blockIdx.x % p.nranges;
    const int b = pair / p.Hkv, g = pair % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, nullptr, false);
    const int lo = range * R;
    if (lo >= n && range > 0) return;  // no tokens; range 0 still writes the counts
    const int head0 = b * p.Hq + g * p.G;
    const int nh = p.G;
    const int wlo = min(p.n_sink, n);
    const int wmid = max(max(0, n - p.n_local), wlo);
    const uint32_t* drow = p.dist + (int64_t)pair * p.d_sp;
    pdl_launch_dependents();
    pdl_wait();  // the distances and the ranges' shares of k_sel_scan

    int mode[4], T[4], Tm1[4], q[4], base[4], expect[4];
    bool any2 = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        mode[e] = 0;
        T[e] = 0;
        q[e] = 0;
        base[e] = 0;
        expect[e] = 0;
        if (e < nh && lo < n) {
            const int2 mt = p.meta_t[pair * 4 + e];
            const int4 m4 = p.meta_r[((int64_t)pair * p.nranges + range) * 4 + e];
            T[e] = mt.x;
            base[e] = m4.x;
            q[e] = m4.y;
            expect[e] = m4.w;
            mode[e] = (m4.y <= 0) ? 0 : (m4.y >= m4.z ? 1 : 2);
        }
        Tm1[e] = T[e] - 1;
        any2 = any2 || mode[e] == 2;
    }
    const int lb = lo + (warp * 32 + lane) * 32;  // this lane's 32 tokens
    const uint32_t valid = low_bits(n - lb);
    const uint32_t win = low_bits(wlo - lb) | ~low_bits(wmid - lb);
    uint32_t lt[4] = {0u, 0u, 0u, 0u}, le[4] = {0u, 0u, 0u, 0u};
    if (valid != 0u) {
        uint32_t D[32];
        const uint4* src = reinterpret_cast<const uint4*>(drow + lb);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = src[j];
            D[4 * j + 0] = v.x;
            D[4 * j + 1] = v.y;
            D[4 * j + 2] = v.z;
            D[4 * j + 3] = v.w;
        }
        le_masks(D, thresh_word(Tm1, nh), lt);
        le_masks(D, thresh_word(T, nh), le);
        // the line has been read for the last time: drop it from L2 without writing it back
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(drow + lb) : "memory");
    }
    uint32_t msk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) msk[e] = (mode[e] == 1) ? le[e] : lt[e];
    if (any2) {
        // the boundary range of a head: its tied tokens, ranked in token order
        uint32_t eq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            eq[e] = 0u;
            if (mode[e] == 2) {
                eq[e] = le[e] & ~lt[e] & valid;
                if (p.excl) eq[e] &= ~win;
                const uint32_t c = warp_sum_u((uint32_t)__popc(eq[e]));
                if (lane == 0) s_wt[e][warp] = (int)c;
            }
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (mode[e] == 2) {
                int qw = q[e];
                for (int w2 = 0; w2 < warp; ++w2) qw -= s_wt[e][w2];
                int tot;
                const int ex = warp_excl_scan(__popc(eq[e]), &tot);
                msk[e] |= first_bits(eq[e], qw - ex);
            }
        }
    }
    int pos[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        msk[e] = (e < nh) ? ((msk[e] | win) & valid) : 0u;
        int tot;
        pos[e] = warp_excl_scan(__popc(msk[e]), &tot);
        if (lane == 0) s_wc[e][warp] = tot;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (tid == e && e < nh) {
            int mine = 0;
            for (int w2 = 0; w2 < NW; ++w2) mine += s_wc[e][w2];
            if (mine != expect[e]) flag_error(p.err, HA_DEVERR_STATE);  // the masks disagree with the counts
        }
    }
    const int cap = p.cap;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (e < nh) {
            int at = base[e] + pos[e];
            for (int w2 = 0; w2 < warp; ++w2) at += s_wc[e][w2];
            uint32_t m = msk[e];
            int32_t* dst = p.list + (int64_t)(head0 + e) * cap;
            if (at < 0 || at + __popc(m) > cap) {
                flag_error(p.err, HA_DEVERR_STATE);
                m = 0u;
            }
            if (__popc(m) >= 8) {
                // dense (window) blocks: independent stores instead of a serial bit walk
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if ((m >> j) & 1u) dst[at + __popc(m & ((1u << j) - 1u))] = lb + j;
            } else {
                while (m != 0u) {
                    const int j = __ffs(m) - 1;
                    m &= m - 1u;
                    dst[at++] = lb + j;
                }
            }
        }
    }
    if (range == 0) {
        for (int e = 0; e < nh; ++e) {
            const int all = p.meta_t[pair * 4 + e].y;
            const int c = min(all, cap);
            if (tid == 0) {
                p.cnt[head0 + e] = c;
                if (all > cap) flag_error(p.err, HA_DEVERR_STATE);
            }
            if (p.pad) {
                int32_t* dst = p.list + (int64_t)(head0 + e) * cap;
                for (int x = c + tid; x < cap; x += NT) dst[x] = -1;
            }
        }
    }
}

}  // namespace

int fused_ranges(int n_cap) { return (n_cap + kSelRange - 1) / kSelRange; }

cudaError_t launch_select_fused(const FusedSelParams& p, int batch_hkv, cudaStream_t st) {
    const dim3 grid((unsigned)batch_hkv * (unsigned)p.nranges);
    if (p.G == 4)
        k_sel_scan<true, 4><<<grid, kSelThreads, 0, st>>>(p);
    else
        k_sel_scan<true, 0><<<grid, kSelThreads, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_ex(k_sel_emit, grid, dim3(kSelThreads), 0, st, true, p);
}

cudaError_t launch_sel_scan(const FusedSelParams& p, int batch_hkv, cudaStream_t st, bool write_dist, bool pdl) {
    const dim3 grid((unsigned)batch_hkv * (unsigned)p.nranges);
    if (p.G == 4) {
        if (write_dist) return launch_ex(k_sel_scan<true, 4>, grid, dim3(kSelThreads), 0, st, pdl, p);
        return launch_ex(k_sel_scan<false, 4>, grid, dim3(kSelThreads), 0, st, pdl, p);
    }
    if (write_dist) return launch_ex(k_sel_scan<true, 0>, grid, dim3(kSelThreads), 0, st, pdl, p);
    return launch_ex(k_sel_scan<false, 0>, grid, dim3(kSelThreads), 0, st, pdl, p);
}

}  // namespace ha
