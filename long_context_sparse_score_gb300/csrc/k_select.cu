// SCORE and TOPK kernels of the sparse-decode path.
//
// HashAttention: Semantic Sparsity for Faster Inference, Eq. (2): the score of a
// cached token is the negated Hamming distance between its 32-bit key code and
// the query code; Sec. 4 keeps the m best tokens, Sec. 4.4 adds the first
// n_sink and the most recent n_local tokens.
//
// Work decomposition: a CTA owns one chunk of `chunk` consecutive tokens of one
// (batch entry, KV head) and serves every query head of that KV head from a
// single read of the chunk's codes (the GQA sharing of Nectar Sec. 3).
//   k_score   per-chunk 33-bin distance histograms (and, for the SCORE entry
//             point, the distances themselves)
//   k_select  threshold bin t and tie quota r per head from the chunk
//             histograms; then, with two block-wide prefix sums in token order,
//             the deterministic selection (distance, then index) joined with
//             the windows, written as one ascending segment per chunk
//   k_compact gathers the segments into the caller's [heads, cap] list
//   k_hist    sums the chunk histograms (SCORE entry point)
#include "ha_internal.cuh"

namespace ha {
namespace {

constexpr int kWarps = kScoreThreads / 32;

template <int TPT>
__device__ __forceinline__ void load_codes(const uint32_t* __restrict__ row, int i0, int n,
                                           uint32_t (&c)[TPT]) {
    if (i0 + TPT <= n) {
        const uint4* p = reinterpret_cast<const uint4*>(row + i0);
#pragma unroll
        for (int j = 0; j < TPT / 4; ++j) {
            const uint4 v = __ldg(p + j);
            c[4 * j + 0] = v.x;
            c[4 * j + 1] = v.y;
            c[4 * j + 2] = v.z;
            c[4 * j + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < TPT; ++j) c[j] = (i0 + j < n) ? __ldg(row + i0 + j) : 0u;
    }
}

// Codes of this thread in SCORE: groups of 4 consecutive tokens, the warp's 32
// lanes reading 512 contiguous bytes per load; token of slot j is
// c0 + (j / 4) * (4 * kScoreThreads) + 4 * threadIdx.x + j % 4.
template <int TPT>
__device__ __forceinline__ void load_codes_coalesced(const uint32_t* __restrict__ row, int c0, int n,
                                                     uint32_t (&c)[TPT]) {
#pragma unroll
    for (int j = 0; j < TPT / 4; ++j) {
        const int i = c0 + j * 4 * kScoreThreads + 4 * threadIdx.x;
        if (i + 4 <= n) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + i));
            c[4 * j + 0] = v.x;
            c[4 * j + 1] = v.y;
            c[4 * j + 2] = v.z;
            c[4 * j + 3] = v.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) c[4 * j + e] = (i + e < n) ? __ldg(row + i + e) : 0u;
        }
    }
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide exclusive prefix sum of two packed words (16-bit fields each; every
// field total stays below 2^16). `wsum` is [kWarps][2] shared scratch used by
// this scan only.
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t& ex_a, uint32_t& ex_b,
                                            uint32_t& tot_a, uint32_t& tot_b, uint32_t (*wsum)[2]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t ya = __shfl_up_sync(0xffffffffu, ia, o);
        const uint32_t yb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += ya;
            ib += yb;
        }
    }
    if (lane == 31) {
        wsum[warp][0] = ia;
        wsum[warp][1] = ib;
    }
    __syncthreads();
    uint32_t pa = 0, pb = 0, sa = 0, sb = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t va = wsum[w][0], vb = wsum[w][1];
        if (w < warp) {
            pa += va;
            pb += vb;
        }
        sa += va;
        sb += vb;
    }
    ex_a = pa + ia - a;
    ex_b = pb + ib - b;
    tot_a = sa;
    tot_b = sb;
}

__device__ __forceinline__ uint32_t field(uint32_t w01, uint32_t w23, int e) {
    const uint32_t w = (e < 2) ? w01 : w23;
    return (e & 1) ? (w >> 16) : (w & 0xffffu);
}

// ---------------------------------------------------------------- SCORE

template <int TPT>
__global__ void __launch_bounds__(kScoreThreads, 3) k_score(const ScoreParams p) {
    constexpr int C = kScoreThreads * TPT;
    // Per-thread histogram columns: hist[bin][thread], the counts of up to four
    // heads packed one byte each (a thread sees at most TPT <= 32 tokens).
    __shared__ uint32_t hist[HA_NBINS][kScoreThreads];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x % p.nchunks;
    const int bg = blockIdx.x / p.nchunks;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, c == 0 && g == 0 && tid == 0);
    const int head0 = b * p.Hq + g * p.G;
    if (c == 0 && p.counters != nullptr)
        for (int e = tid; e < p.G; e += kScoreThreads) p.counters[head0 + e] = 0u;
    const int c0 = c * C;
    if (c0 >= n) return;

    const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)g * p.ks_sh;
    uint32_t code[TPT];
    load_codes_coalesced<TPT>(row, c0, n, code);
    const int nin = n - c0;  // tokens of this chunk are valid below this offset

    for (int hp = 0; hp < p.G; hp += kMaxHeadsPerPass) {
        const int nh = min(kMaxHeadsPerPass, p.G - hp);
        uint32_t qs[kMaxHeadsPerPass];
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) qs[e] = (e < nh) ? p.q_sig[head0 + hp + e] : 0u;
#pragma unroll
        for (int u = 0; u < HA_NBINS; ++u) hist[u][tid] = 0u;
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            const int off = (j >> 2) * 4 * kScoreThreads + 4 * tid + (j & 3);
            if (off < nin) {
#pragma unroll
                for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                    if (e < nh) {
                        const int d = __popc(qs[e] ^ code[j]);
                        hist[d][tid] += 1u << (8 * e);
                    }
                }
            }
        }
        if (p.dist != nullptr) {
#pragma unroll
            for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                if (e < nh) {
                    uint8_t* drow = p.dist + (int64_t)(head0 + hp + e) * p.n_cap + c0;
#pragma unroll
                    for (int j = 0; j < TPT; ++j) {
                        const int off = (j >> 2) * 4 * kScoreThreads + 4 * tid + (j & 3);
                        if (off < nin) drow[off] = (uint8_t)__popc(qs[e] ^ code[j]);
                    }
                }
            }
        }
        __syncthreads();
        for (int u = warp; u < HA_NBINS; u += kWarps) {
            uint32_t s01 = 0, s23 = 0;  // 16-bit fields: heads (0,1) and (2,3)
#pragma unroll
            for (int k = lane; k < kScoreThreads; k += 32) {
                const uint32_t w = hist[u][k];
                s01 += (w & 0xffu) | ((w & 0xff00u) << 8);
                s23 += ((w >> 16) & 0xffu) | ((w >> 8) & 0xff0000u);
            }
            s01 = warp_sum(s01);
            s23 = warp_sum(s23);
            if (lane < nh)
                p.chunk_hist[((int64_t)(head0 + hp + lane) * p.nchunks + c) * HA_NBINS + u] =
                    field(s01, s23, lane);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- TOPK

template <int TPT>
__global__ void __launch_bounds__(kScoreThreads, 3) k_select(const SelectParams p) {
    constexpr int C = kScoreThreads * TPT;
    __shared__ int s_t[kMaxHeadsPerPass];
    __shared__ int s_quota[kMaxHeadsPerPass];
    __shared__ uint32_t s_tot[kMaxHeadsPerPass][HA_NBINS];
    __shared__ uint32_t s_pre[kMaxHeadsPerPass][HA_NBINS];
    __shared__ uint32_t s_w1[kWarps][2];
    __shared__ uint32_t s_w2[kWarps][2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x % p.nchunks;
    const int bg = blockIdx.x / p.nchunks;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, false);
    const int nch = (n + C - 1) / C;
    if (c >= nch) return;

    int mb = p.m;
    if (p.m_per_seq != nullptr) {
        mb = p.m_per_seq[b];
        if (mb < 0 || mb > p.m) {
            if (c == 0 && g == 0 && tid == 0) flag_error(p.err, HA_DEVERR_BUDGET);
            mb = min(max(mb, 0), p.m);
        }
    }
    const int k = min(mb, n);                  // tokens taken by score
    const int wlo = min(p.n_sink, n);          // sink window [0, wlo)
    const int whi = max(0, n - p.n_local);     // local window [whi, n)
    const int head0 = b * p.Hq + g * p.G;
    const int64_t seg_stride = (int64_t)p.nchunks * p.chunk;

    const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)g * p.ks_sh;
    const int i0 = c * C + tid * TPT;
    uint32_t code[TPT];
    load_codes<TPT>(row, i0, n, code);
    const int nvalid = max(0, min(TPT, n - i0));

    for (int hp = 0; hp < p.G; hp += kMaxHeadsPerPass) {
        const int nh = min(kMaxHeadsPerPass, p.G - hp);
        // ---- threshold bin t and this chunk's tie quota: the histograms of all
        // chunks (totals) and of the chunks before this one (prefix), per head
        for (int i = tid; i < kMaxHeadsPerPass * HA_NBINS; i += kScoreThreads) {
            (&s_tot[0][0])[i] = 0u;
            (&s_pre[0][0])[i] = 0u;
        }
        __syncthreads();
        {
            const int per = nch * HA_NBINS;
            const int total = nh * per;
            const uint32_t* H0 = p.chunk_hist + (int64_t)(head0 + hp) * p.nchunks * HA_NBINS;
            constexpr int kBatch = 8;
            for (int i0 = 0; i0 < total; i0 += kBatch * kScoreThreads) {
                uint32_t v[kBatch];
#pragma unroll
                for (int k2 = 0; k2 < kBatch; ++k2) {
                    const int i = i0 + k2 * kScoreThreads + tid;
                    v[k2] = 0u;
                    if (i < total) {
                        const int e = i / per;
                        v[k2] = H0[(int64_t)e * p.nchunks * HA_NBINS + (i - e * per)];
                    }
                }
#pragma unroll
                for (int k2 = 0; k2 < kBatch; ++k2) {
                    const int i = i0 + k2 * kScoreThreads + tid;
                    if (v[k2] != 0u) {
                        const int e = i / per;
                        const int rem = i - e * per;
                        const int cc = rem / HA_NBINS;
                        const int u = rem - cc * HA_NBINS;
                        atomicAdd(&s_tot[e][u], v[k2]);
                        if (cc < c) atomicAdd(&s_pre[e][u], v[k2]);
                    }
                }
            }
        }
        __syncthreads();
        if (warp < nh) {
            // bins 0..31 (bin 32 is implied: the cumulative count reaches n there)
            uint32_t incl = s_tot[warp][lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned reach = __ballot_sync(0xffffffffu, incl >= (uint32_t)k);
            const int t = reach ? (__ffs(reach) - 1) : 32;
            const uint32_t below = __shfl_sync(0xffffffffu, incl, (t == 0 ? 0 : t - 1) & 31);
            const int r = k - (t == 0 ? 0 : (int)below);
            if (lane == 0) {
                s_t[warp] = t;
                s_quota[warp] = r - (int)s_pre[warp][t];
            }
        }
        __syncthreads();
        uint32_t qs[kMaxHeadsPerPass];
        int t[kMaxHeadsPerPass], quota[kMaxHeadsPerPass];
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            qs[e] = (e < nh) ? p.q_sig[head0 + hp + e] : 0u;
            t[e] = (e < nh) ? s_t[e] : -1;
            quota[e] = (e < nh) ? s_quota[e] : 0;
        }
        // ---- pass 1: ties (distance == t) per head, prefix over the chunk
        uint32_t tie01 = 0, tie23 = 0;
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            if (j < nvalid) {
#pragma unroll
                for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                    const uint32_t hit = (__popc(qs[e] ^ code[j]) == t[e]) ? 1u : 0u;
                    if (e == 0) tie01 += hit;
                    if (e == 1) tie01 += hit << 16;
                    if (e == 2) tie23 += hit;
                    if (e == 3) tie23 += hit << 16;
                }
            }
        }
        uint32_t tb01, tb23, tt01, tt23;
        block_scan2(tie01, tie23, tb01, tb23, tt01, tt23, s_w1);
        // ---- pass 2: selection flags in token order
        int run[kMaxHeadsPerPass];
        uint32_t selmask[kMaxHeadsPerPass];
        uint32_t sel01 = 0, sel23 = 0;
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            run[e] = (int)field(tb01, tb23, e);
            selmask[e] = 0u;
        }
#pragma unroll
        for (int j = 0; j < TPT; ++j) {
            if (j < nvalid) {
                const int i = i0 + j;
                const bool inw = (i < wlo) || (i >= whi);
#pragma unroll
                for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                    const int d = __popc(qs[e] ^ code[j]);
                    const bool tie = (d == t[e]);
                    const bool s = inw || (d < t[e]) || (tie && run[e] < quota[e]);
                    run[e] += tie ? 1 : 0;
                    if (s) selmask[e] |= 1u << j;
                }
            }
        }
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            if (e >= nh) selmask[e] = 0u;
            const uint32_t cnt = (uint32_t)__popc(selmask[e]);
            if (e == 0) sel01 += cnt;
            if (e == 1) sel01 += cnt << 16;
            if (e == 2) sel23 += cnt;
            if (e == 3) sel23 += cnt << 16;
        }
        uint32_t sb01, sb23, st01, st23;
        block_scan2(sel01, sel23, sb01, sb23, st01, st23, s_w2);
        // ---- pass 3: write this chunk's ascending segment per head
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            if (e < nh) {
                int32_t* seg = p.seg_idx + (int64_t)(head0 + hp + e) * seg_stride + (int64_t)c * p.chunk;
                int pos = (int)field(sb01, sb23, e);
                uint32_t msk = selmask[e];
                while (msk) {
                    const int j = __ffs(msk) - 1;
                    msk &= msk - 1;
                    seg[pos++] = i0 + j;
                }
                if (tid == 0) p.seg_cnt[(int64_t)(head0 + hp + e) * p.nchunks + c] = (int)field(st01, st23, e);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- compaction / histogram

__global__ void __launch_bounds__(256) k_compact(const CompactParams p) {
    const int head = blockIdx.x;
    const int b = head / p.Hq;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, false);
    const int nch = (n + p.chunk - 1) / p.chunk;
    const int32_t* cnt = p.seg_cnt + (int64_t)head * p.nchunks;
    const int32_t* seg = p.seg_idx + (int64_t)head * p.nchunks * p.chunk;
    int32_t* dst = p.sel_idx + (int64_t)head * p.cap;
    int base = 0;
    for (int cc = 0; cc < nch; ++cc) {
        int k = cnt[cc];
        if (base + k > p.cap) k = p.cap - base;  // cannot happen for |I| <= cap
        for (int t = threadIdx.x; t < k; t += blockDim.x) dst[base + t] = seg[(int64_t)cc * p.chunk + t];
        base += k;
    }
    for (int t = base + threadIdx.x; t < p.cap; t += blockDim.x) dst[t] = -1;
    if (threadIdx.x == 0) p.sel_cnt[head] = base;
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

}  // namespace

cudaError_t launch_score(const ScoreParams& p, int batch_hkv, cudaStream_t st) {
    const dim3 grid((unsigned)batch_hkv * (unsigned)p.nchunks);
    switch (p.chunk / kScoreThreads) {
        case 4: k_score<4><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 8: k_score<8><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 16: k_score<16><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 32: k_score<32><<<grid, kScoreThreads, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_select(const SelectParams& p, int batch_hkv, cudaStream_t st) {
    const dim3 grid((unsigned)batch_hkv * (unsigned)p.nchunks);
    switch (p.chunk / kScoreThreads) {
        case 4: k_select<4><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 8: k_select<8><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 16: k_select<16><<<grid, kScoreThreads, 0, st>>>(p); break;
        case 32: k_select<32><<<grid, kScoreThreads, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_compact(const CompactParams& p, int heads, cudaStream_t st) {
    k_compact<<<heads, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_hist(const HistParams& p, int heads, cudaStream_t st) {
    k_hist<<<heads, 64, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ha
