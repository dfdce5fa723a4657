// SCORE and TOPK kernels of the sparse-decode path.
//
// HashAttention: Semantic Sparsity for Faster Inference, Eq. (2): the score of a
// cached token is the negated Hamming distance between its 32-bit key code and
// the query code; Sec. 4 keeps the m best tokens, Sec. 4.4 adds the first
// n_sink and the most recent n_local tokens.
//
// Work decomposition. A CTA owns one chunk of kScoreThreads * TPT consecutive
// tokens of one (batch entry, KV head) and serves every query head of that KV
// head from one read of the chunk's codes (the GQA sharing of Nectar Sec. 3).
// Inside the chunk, warp w owns the sub-chunk of 32 * TPT consecutive tokens
// starting at w * 32 * TPT; in round r its lane l holds the 4 tokens
// 128 r + 4 l + {0..3} of the sub-chunk (one 16-byte load; 512 contiguous bytes
// per warp load).
//   k_score   33-bin distance histogram of every chunk (and, for the SCORE entry
//             point, the distances themselves)
//   k_select  per head: the threshold bin t (smallest t whose cumulative count
//             reaches min(m, n)) and the chunk's tie quota from the chunk
//             histograms; then each warp selects its sub-chunk in token order
//             with ballots and writes it as one ascending segment. Only the one
//             chunk per head where the quota of tied tokens runs out needs the
//             per-warp tie ranks; elsewhere a token is selected iff its distance
//             is at most t (quota left) or below t (quota spent), or it lies in
//             a window.
//   k_compact gathers the segments into the caller's [heads, cap] list
//   k_hist    sums the chunk histograms (SCORE entry point)
#include "ha_internal.cuh"

namespace ha {
namespace {

constexpr int kWarps = kScoreThreads / 32;

// Codes of this thread (see the decomposition above); tokens at or beyond n read 0.
template <int TPT>
__device__ __forceinline__ void load_codes(const uint32_t* __restrict__ row, int sbase, int n,
                                           uint32_t (&c)[TPT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < TPT / 4; ++r) {
        const int i = sbase + 128 * r + 4 * lane;
        if (i + 4 <= n) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + i));
            c[4 * r + 0] = v.x;
            c[4 * r + 1] = v.y;
            c[4 * r + 2] = v.z;
            c[4 * r + 3] = v.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) c[4 * r + e] = (i + e < n) ? __ldg(row + i + e) : 0u;
        }
    }
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void red_shared_add(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t field(uint32_t w01, uint32_t w23, int e) {
    const uint32_t w = (e < 2) ? w01 : w23;
    return (e & 1) ? (w >> 16) : (w & 0xffffu);
}

// Tokens of [a, z) at distance t from qs, counted by the whole warp (every lane
// gets the total); 8 loads in flight per lane.
__device__ __forceinline__ int count_at(const uint32_t* __restrict__ row, int a, int z, uint32_t qs, int t) {
    const int lane = threadIdx.x & 31;
    int c = 0;
    for (int i0 = a; i0 < z; i0 += 256) {
        uint32_t cd[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + 32 * u + lane;
            cd[u] = (i < z) ? __ldg(row + i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) c += (i0 + 32 * u + lane < z && __popc(qs ^ cd[u]) == t) ? 1 : 0;
    }
    return __reduce_add_sync(0xffffffffu, c);
}

// ---------------------------------------------------------------- SCORE

// VARIANTS: per-head budgets / exclusive windows compiled in (launched only when asked for).
template <int TPT, bool WRITE_DIST, bool VARIANTS>
__global__ void __launch_bounds__(kScoreThreads, 5) k_score(const ScoreParams p) {
    constexpr int C = kScoreThreads * TPT;
    constexpr int SC = 32 * TPT;
    // Histogram columns hist[bin][pair][lane], shared by the CTA's warps: lane l
    // of every warp adds into column l (no bank conflict inside an instruction),
    // heads 2*pair and 2*pair+1 in the low and high 16-bit field (a column sees at
    // most kWarps * TPT <= 256 tokens per bin).
    __shared__ uint32_t hist[HA_NBINS][2][32];
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x % p.nchunks;
    const int bg = blockIdx.x / p.nchunks;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, c == 0 && g == 0 && tid == 0);
    const int head0 = b * p.Hq + g * p.G;
    pdl_launch_dependents();
    if (c == 0 && p.counters != nullptr)
        for (int e = tid; e < p.G; e += kScoreThreads) p.counters[head0 + e] = 0u;
    const int c0 = c * C;
    if (c0 >= n) return;

    const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)g * p.ks_sh;
    const int sbase = c0 + warp * SC;
    uint32_t code[TPT];
    load_codes<TPT>(row, sbase, n, code);
    const uint32_t col = smem_addr(&hist[0][0][lane]);

    for (int hp = 0; hp < p.G; hp += kMaxHeadsPerPass) {
        const int nh = min(kMaxHeadsPerPass, p.G - hp);
        uint32_t qs[kMaxHeadsPerPass];
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) qs[e] = (e < nh) ? p.q_sig[head0 + hp + e] : 0u;
        for (int x = tid; x < HA_NBINS * 2 * 32; x += kScoreThreads) (&hist[0][0][0])[x] = 0u;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            const int i = sbase + 128 * (j >> 2) + 4 * lane + (j & 3);
            if (i < n) {
#pragma unroll
                for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                    if (e < nh) {
                        const uint32_t d = (uint32_t)__popc(qs[e] ^ code[j]);
                        red_shared_add(col + (d * 2 + (e >> 1)) * (32 * 4), 1u << (16 * (e & 1)));
                    }
                }
            }
        }
        if (WRITE_DIST) {
#pragma unroll
            for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                if (e < nh) {
                    uint8_t* drow = p.dist + (int64_t)(head0 + hp + e) * p.n_cap;
#pragma unroll
                    for (int j = 0; j < TPT; ++j) {
                        const int i = sbase + 128 * (j >> 2) + 4 * lane + (j & 3);
                        if (i < n) drow[i] = (uint8_t)__popc(qs[e] ^ code[j]);
                    }
                }
            }
        }
        __syncthreads();
        for (int u = warp; u < HA_NBINS; u += kWarps) {
            const uint32_t s01 = warp_sum(hist[u][0][lane]);  // 16-bit fields: heads (0,1)
            const uint32_t s23 = warp_sum(hist[u][1][lane]);  // and (2,3)
            if (lane < nh)
                p.chunk_hist[((int64_t)(head0 + hp + lane) * p.nchunks + c) * HA_NBINS + u] =
                    field(s01, s23, lane);
        }
        __syncthreads();
    }

    // ---- the last CTA of this (batch entry, KV head) to finish turns the chunk
    // histograms into the threshold bin t of every head and, per chunk, the
    // number of tied tokens (distance == t) still to take and the chunk's ties
    if (p.meta_t == nullptr) return;
    const int nch = (n + C - 1) / C;
    __syncthreads();  // every histogram store of this CTA precedes thread 0's fence
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&p.score_cnt[bg], 1u);
        if (prev >= (unsigned)nch) flag_error(p.err, HA_DEVERR_STATE);
        s_last = (prev == (unsigned)(nch - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    int mb = p.m;
    if (p.m_per_seq != nullptr) {
        mb = p.m_per_seq[b];
        if (mb < 0 || mb > p.m) {
            if (g == 0 && tid == 0) flag_error(p.err, HA_DEVERR_BUDGET);
            mb = min(max(mb, 0), p.m);
        }
    }
    const int wlo = min(p.n_sink, n), whi = max(0, n - p.n_local);
    const int wmid = max(whi, wlo);         // windows: [0, wlo) and [wmid, n)
    const int nwin = wlo + (n - wmid);
    for (int e = warp; e < p.G; e += kWarps) {
        const int64_t h = head0 + e;
        const uint32_t* H = p.chunk_hist + h * p.nchunks * HA_NBINS;
        const int excl = VARIANTS ? p.excl : 0;
        int mh = mb;
        if (VARIANTS && p.m_per_head != nullptr) {
            mh = p.m_per_head[h];
            if (mh < 0 || mh > p.m) {
                if (lane == 0) flag_error(p.err, HA_DEVERR_BUDGET);
                mh = min(max(mh, 0), p.m);
            }
        }
        // tokens taken by score: from all n, or (exclusive windows) from those outside the windows
        const int k = excl ? min(mh, n - nwin) : min(mh, n);
        const uint32_t qs = excl ? p.q_sig[h] : 0u;  // needed for the window tokens only
        // bins 0..31 (bin 32 is implied: the cumulative count reaches n there)
        uint32_t tot = 0;
        for (int c0b = 0; c0b < nch; c0b += 8) {
            uint32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = (c0b + u < nch) ? __ldcg(H + (c0b + u) * HA_NBINS + lane) : 0u;
#pragma unroll
            for (int u = 0; u < 8; ++u) tot += v[u];
        }
        if (excl) {
            // the window tokens leave the ranking: their distance counts come off the totals
            // (this warp's slice of the CTA's histogram storage, free after the chunk pass)
            uint32_t* wh = &hist[0][0][0] + warp * HA_NBINS;
            for (int u = lane; u < HA_NBINS; u += 32) wh[u] = 0u;
            __syncwarp();
            for (int i = lane; i < nwin; i += 32) {
                const int tok = (i < wlo) ? i : wmid + (i - wlo);
                atomicAdd(&wh[__popc(qs ^ __ldg(row + tok))], 1u);
            }
            __syncwarp();
            tot -= wh[lane];
            __syncwarp();
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned reach = __ballot_sync(0xffffffffu, incl >= (uint32_t)k);
        const int t = reach ? (__ffs(reach) - 1) : 32;
        const uint32_t below = __shfl_sync(0xffffffffu, incl, (t == 0 ? 0 : t - 1) & 31);
        const int r = k - (t == 0 ? 0 : (int)below);
        int carry = 0;  // tied tokens in the chunks before
        for (int base = 0; base < nch; base += 32) {
            const int cc = base + lane;
            int v = (cc < nch) ? (int)__ldcg(H + cc * HA_NBINS + t) : 0;
            if (excl) {
                // ties inside the windows are not ties of the ranking
                const int cb = cc * C, ce = min(n, cb + C);
                const int sa = cb, sz = min(ce, wlo), la = max(cb, wmid), lz = ce;
                unsigned pend = __ballot_sync(0xffffffffu, cc < nch && (sz > sa || lz > la));
                while (pend != 0u) {
                    const int j = __ffs(pend) - 1;
                    pend &= pend - 1u;
                    const int cnt = count_at(row, __shfl_sync(0xffffffffu, sa, j), __shfl_sync(0xffffffffu, sz, j),
                                             qs, t) +
                                    count_at(row, __shfl_sync(0xffffffffu, la, j), __shfl_sync(0xffffffffu, lz, j),
                                             qs, t);
                    if (lane == j) v -= cnt;
                }
            }
            int in = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, in, o);
                if (lane >= o) in += y;
            }
            if (cc < nch) p.meta_qt[h * p.nchunks + cc] = make_int2(r - (carry + in - v), v);
            carry += __shfl_sync(0xffffffffu, in, 31);
        }
        if (lane == 0) p.meta_t[h] = t;
    }
    if (tid == 0) p.score_cnt[bg] = 0u;
}

// ---------------------------------------------------------------- TOPK

// Codes of this lane in TOPK: TPT consecutive tokens starting at lbase (a lane's
// selected tokens are then consecutive in its segment); tokens >= n read 0.
// The warp loads its 32 * TPT codes with 512-byte coalesced loads and hands
// them to their owner lanes through a shared tile (row pitch TPT + 4 words keeps
// both the stores and the per-lane reads free of bank conflicts).
template <int TPT>
__device__ __forceinline__ void load_codes_contig(const uint32_t* __restrict__ row, int sbase, int n,
                                                  uint32_t (*tile)[TPT + 4], uint32_t (&c)[TPT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < TPT / 4; ++j) {
        const int o = 128 * j + 4 * lane;  // offset in the warp's sub-chunk
        const int i = sbase + o;
        uint4 v;
        if (i + 4 <= n) {
            v = __ldg(reinterpret_cast<const uint4*>(row + i));
        } else {
            v.x = (i < n) ? __ldg(row + i) : 0u;
            v.y = (i + 1 < n) ? __ldg(row + i + 1) : 0u;
            v.z = (i + 2 < n) ? __ldg(row + i + 2) : 0u;
            v.w = (i + 3 < n) ? __ldg(row + i + 3) : 0u;
        }
        *reinterpret_cast<uint4*>(&tile[o / TPT][o % TPT]) = v;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < TPT / 4; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(&tile[lane][4 * j]);
        c[4 * j + 0] = v.x;
        c[4 * j + 1] = v.y;
        c[4 * j + 2] = v.z;
        c[4 * j + 3] = v.w;
    }
}

// Warp-inclusive prefix sum.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// Selection mask (bit j = token lbase + j, j < tpt) of one lane for one head on
// the rare path: the lane's tokens touch a window or the end of the sequence, or
// the sub-chunk holds the point where the tie quota runs out (mode 2, where the
// whole warp calls this together to rank ties across lanes). `codes` are the
// lane's codes in the shared tile.
__device__ __noinline__ uint32_t lane_mask_slow(const uint32_t* codes, uint32_t qs, int t, int mode,
                                                int qw, int lbase, int tpt, int n, int wlo, int whi,
                                                int excl) {
    const int teff = (mode == 1) ? t : t - 1;
    uint32_t m = 0u, tie = 0u;
    for (int j = 0; j < tpt; ++j) {
        const int i = lbase + j;
        if (i >= n) break;
        const int d = __popc(qs ^ codes[j]);
        const bool inw = (i < wlo) || (i >= whi);
        const bool take = (mode == 2) ? (d < t) : (d <= teff);
        if (inw || take) m |= 1u << j;
        if (d == t && !(excl && inw)) tie |= 1u << j;  // with exclusive windows a window token is never a tie
    }
    if (mode == 2) {
        const uint32_t c = (uint32_t)__popc(tie);
        const int before = (int)(warp_incl_scan(c) - c);  // ties in the lanes before
        int left = qw - before;
        uint32_t x = tie;
        while (x != 0u && left > 0) {
            const uint32_t low = x & (0u - x);
            m |= low;
            x ^= low;
            --left;
        }
    }
    return m;
}

// Selection mask of one lane for one head.
//   mode 0: no tied token (distance == t) of the sub-chunk is taken
//   mode 1: every tied token is taken
//   mode 2: the first qw tied tokens of the sub-chunk (token order) are taken
template <int TPT>
__device__ __forceinline__ uint32_t lane_mask(const uint32_t (&code)[TPT], const uint32_t* tile_row, uint32_t qs,
                                              int t, int mode, int qw, int lbase, int n, int excl, int wlo,
                                              int whi) {
    const bool edge = (lbase < wlo) || (lbase + TPT > whi) || (lbase + TPT > n);
    if (edge || mode == 2) return lane_mask_slow(tile_row, qs, t, mode, qw, lbase, TPT, n, wlo, whi, excl);
    const int teff = (mode == 1) ? t : t - 1;
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < TPT; ++j) m |= ((int)__popc(qs ^ code[j]) <= teff ? 1u : 0u) << j;
    return m;
}

template <int TPT>
__global__ void __launch_bounds__(kScoreThreads, 4) k_select(const SelectParams p) {
    constexpr int C = kScoreThreads * TPT;
    constexpr int SC = 32 * TPT;
    __shared__ int s_wt[kMaxHeadsPerPass][kWarps];
    __shared__ __align__(16) uint32_t s_codes[kWarps][32][TPT + 4];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Chunks holding the windows take the out-of-line path and run several times
    // longer, so they come first in the grid instead of trailing it: CTA i < W
    // takes the first chunk of pair i (W = B * Hkv pairs), W <= i < 2W the last
    // chunk pair i - W uses, and the rest the remaining chunks of each pair.
    const int W = p.B * p.Hkv;
    const int i = blockIdx.x;
    int bg, c;
    if (i < W) {
        bg = i;
    } else if (p.nchunks >= 2 && i < 2 * W) {
        bg = i - W;
    } else {
        bg = (i - 2 * W) / (p.nchunks - 2);
    }
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, false);
    const int nch = (n + C - 1) / C;
    const int last = nch - 1;                  // the chunk holding the local window
    if (i < W) {
        c = 0;
    } else if (p.nchunks >= 2 && i < 2 * W) {
        c = last >= 1 ? last : p.nchunks - 1;  // a one-chunk sequence: an idle CTA
    } else {
        c = 1 + (i - 2 * W) % (p.nchunks - 2);
        if (last >= 1 && c >= last) ++c;      // skip the chunk the second group took
    }
    if (c >= nch) return;

    const int wlo = min(p.n_sink, n);          // sink window [0, wlo)
    const int whi = max(0, n - p.n_local);     // local window [whi, n)
    const int head0 = b * p.Hq + g * p.G;
    const int nseg = p.nchunks * kWarps;
    const int64_t seg_stride = (int64_t)nseg * SC;
    const int sc = c * kWarps + warp;          // this warp's segment
    const int sbase = c * C + warp * SC;

    const int lbase = sbase + lane * TPT;      // this lane's first token
    const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)g * p.ks_sh;
    uint32_t code[TPT];
    load_codes_contig<TPT>(row, sbase, n, s_codes[warp], code);
    pdl_launch_dependents();
    pdl_wait();  // SCORE's thresholds are read below

    for (int hp = 0; hp < p.G; hp += kMaxHeadsPerPass) {
        const int nh = min(kMaxHeadsPerPass, p.G - hp);
        // ---- threshold bin t and this chunk's tie quota (from SCORE), per head
        uint32_t qs[kMaxHeadsPerPass];
        int t[kMaxHeadsPerPass], mode[kMaxHeadsPerPass], qw[kMaxHeadsPerPass];
        bool boundary = false;
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            qs[e] = 0u;
            t[e] = 0;
            mode[e] = 0;
            qw[e] = 0;
            if (e < nh) {
                const int64_t h = head0 + hp + e;
                const int2 qt = p.meta_qt[h * p.nchunks + c];
                qs[e] = p.q_sig[h];
                t[e] = p.meta_t[h];
                qw[e] = qt.x;
                mode[e] = (qt.x <= 0) ? 0 : (qt.x >= qt.y ? 1 : 2);
            }
            boundary = boundary || (mode[e] == 2);
        }
        // ---- the chunk where the tie quota runs out: per-warp tie counts
        if (boundary) {
#pragma unroll
            for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                if (mode[e] == 2) {
                    uint32_t cnt = 0;
#pragma unroll
                    for (int j = 0; j < TPT; ++j)
                        cnt += (lbase + j < n && (int)__popc(qs[e] ^ code[j]) == t[e] &&
                                !(p.excl && (lbase + j < wlo || lbase + j >= whi))) ? 1u : 0u;
                    cnt = __reduce_add_sync(0xffffffffu, cnt);
                    if (lane == 0) s_wt[e][warp] = (int)cnt;
                }
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                if (mode[e] == 2) {
                    int q = qw[e];
                    for (int w2 = 0; w2 < warp; ++w2) q -= s_wt[e][w2];
                    qw[e] = q;
                    mode[e] = (q <= 0) ? 0 : (q >= s_wt[e][warp] ? 1 : 2);
                }
            }
        }
        // ---- selection masks, then one prefix sum per head pair places every
        // lane's selected tokens (consecutive in the segment)
        uint32_t msk[kMaxHeadsPerPass];
        uint32_t c01 = 0u, c23 = 0u;  // per-lane counts, 16-bit fields
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            msk[e] = (e < nh) ? lane_mask<TPT>(code, &s_codes[warp][lane][0], qs[e], t[e], mode[e], qw[e], lbase, n, p.excl,
                                                 wlo, whi)
                               : 0u;
            const uint32_t c = (uint32_t)__popc(msk[e]);
            if (e == 0) c01 |= c;
            if (e == 1) c01 |= c << 16;
            if (e == 2) c23 |= c;
            if (e == 3) c23 |= c << 16;
        }
        const uint32_t i01 = warp_incl_scan(c01);
        const uint32_t i23 = (nh > 2) ? warp_incl_scan(c23) : 0u;
        const uint32_t x01 = i01 - c01, x23 = i23 - c23;
        const uint32_t t01 = __shfl_sync(0xffffffffu, i01, 31), t23 = __shfl_sync(0xffffffffu, i23, 31);
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            if (e < nh) {
                const int64_t h = head0 + hp + e;
                int32_t* seg = p.seg_idx + h * seg_stride + (int64_t)sc * SC;
                int w = (int)field(x01, x23, e);
                uint32_t x = msk[e];
                while (x != 0u) {
                    const int j = __ffs(x) - 1;
                    x &= x - 1u;
                    seg[w++] = lbase + j;
                }
                if (lane == 0) p.seg_cnt[h * nseg + sc] = (int)field(t01, t23, e);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- compaction / histogram

// One CTA per head: the segment counts are loaded together and scanned into a
// prefix table in shared memory, then every output position finds its segment
// by binary search (all loads independent), and the tail is padded with -1.
constexpr int kCompactThreads = 256;

__global__ void __launch_bounds__(kCompactThreads) k_compact(const CompactParams p) {
    __shared__ int s_pre[kMaxSegments + 1];
    __shared__ int s_wsum[kCompactThreads / 32];
    const int head = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = head / p.Hq;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, false);
    const int nused = (n + p.seg_cap - 1) / p.seg_cap;
    const int32_t* cnt = p.seg_cnt + (int64_t)head * p.nseg;
    const int32_t* seg = p.seg_idx + (int64_t)head * p.nseg * p.seg_cap;
    int32_t* dst = p.sel_idx + (int64_t)head * p.cap;
    int carry = 0;
    for (int base = 0; base < nused; base += kCompactThreads) {
        const int i = base + tid;
        const int v = (i < nused) ? min(max(cnt[i], 0), p.seg_cap) : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int w2 = 0; w2 < kCompactThreads / 32; ++w2) {
            before += (w2 < warp) ? s_wsum[w2] : 0;
            total += s_wsum[w2];
        }
        if (i < nused) s_pre[i] = carry + before + x - v;
        carry += total;
        __syncthreads();
    }
    if (tid == 0) s_pre[nused] = carry;
    __syncthreads();
    const int total = min(carry, p.cap);  // entries beyond cap cannot occur for |I| <= cap
    constexpr int kB = 4;
    for (int t0 = 0; t0 < total; t0 += kB * kCompactThreads) {
        int tok[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int t = t0 + u * kCompactThreads + tid;
            tok[u] = -1;
            if (t < total) {
                int lo = 0, hi = nused - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_pre[mid] <= t) lo = mid; else hi = mid - 1;
                }
                tok[u] = seg[(int64_t)lo * p.seg_cap + (t - s_pre[lo])];
            }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int t = t0 + u * kCompactThreads + tid;
            if (t < total) dst[t] = tok[u];
        }
    }
    for (int t = total + tid; t < p.cap; t += kCompactThreads) dst[t] = -1;
    if (tid == 0) p.sel_cnt[head] = total;
}

__global__ void __launch_bounds__(64) k_hist(const HistParams p) {
    const int head = blockIdx.x;
    const int b = head / p.Hq;
    const int n = checked_len(p.seq_lens, b, p.n_cap, nullptr, false);
    const int nch = (n + p.chunk - 1) / p.chunk;
    const int u = threadIdx.x;
    if (u >= HA_NBINS) return;
    uint32_t s = 0;
    for (int cc = 0; cc < nch; ++cc) s += p.chunk_hist[((int64_t)head * p.nchunks + cc) * HA_NBINS + u];
    p.hist[(int64_t)head * HA_NBINS + u] = s;
}

template <bool WD, bool VAR>
cudaError_t launch_score_t(const ScoreParams& p, int batch_hkv, cudaStream_t st) {
    const dim3 grid((unsigned)batch_hkv * (unsigned)p.nchunks);
    switch (p.chunk / kScoreThreads) {
        case 4: k_score<4, WD, VAR><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 8: k_score<8, WD, VAR><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 16: k_score<16, WD, VAR><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 32: k_score<32, WD, VAR><<<grid, kScoreThreads, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(const ScoreParams& p, int batch_hkv, cudaStream_t st) {
    // the distance-writing entry point computes no thresholds, so it needs no variants
    if (p.dist != nullptr) return launch_score_t<true, false>(p, batch_hkv, st);
    if (p.excl || p.m_per_head != nullptr) return launch_score_t<false, true>(p, batch_hkv, st);
    return launch_score_t<false, false>(p, batch_hkv, st);
}

cudaError_t launch_select(const SelectParams& p, int batch_hkv, cudaStream_t st, bool pdl) {
    const dim3 grid((unsigned)batch_hkv * (unsigned)p.nchunks);
    const dim3 block(kScoreThreads);
    switch (p.chunk / kScoreThreads) {
        case 4: return launch_ex(k_select<4>, grid, block, 0, st, pdl, p);
        case 8: return launch_ex(k_select<8>, grid, block, 0, st, pdl, p);
        case 16: return launch_ex(k_select<16>, grid, block, 0, st, pdl, p);
        case 32: return launch_ex(k_select<32>, grid, block, 0, st, pdl, p);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_compact(const CompactParams& p, int heads, cudaStream_t st) {
    k_compact<<<heads, kCompactThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_hist(const HistParams& p, int heads, cudaStream_t st) {
    k_hist<<<heads, 64, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ha
