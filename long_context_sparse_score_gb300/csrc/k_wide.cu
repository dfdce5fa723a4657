// SCORE and TOPK for codes wider than 32 bits (W 32-bit words per token).
//
// HashAttention: Semantic Sparsity for Faster Inference, Eq. (2) with a
// signature of b = 32 W bits (Sec. 5 varies the signature length): the distance
// of a cached token is the Hamming distance summed over the W words, in
// [0, b]. The selection rule is that of the 32-bit path (the min(m, n) smallest
// distances, ties to the smaller index, joined with the windows), and the
// output is the same per-warp segments, so GATHER-ATT and the compaction are
// shared with it.
//
//   k_score_wide   CTA = 256 threads over a chunk of tokens of one (sequence,
//                  KV head); per token the W words are read once and give the
//                  distance of every query head of the pass; b + 1 bins per
//                  head in shared memory. The last CTA of a (sequence, KV head)
//                  turns the chunk histograms into t, r and every chunk's
//                  (quota left, ties) with a warp scan over the bins.
//   k_select_wide  same chunking; lane l owns tpt consecutive tokens of its
//                  warp's sub-chunk; distances are recomputed per pass (a tie
//                  count pass runs only in the chunk where the quota of tied
//                  tokens runs out), selected tokens go to the warp's segment.
// The query codes of the pass sit in shared memory; codes are read with
// 16-byte loads when W is a multiple of 4.
#include "ha_internal.cuh"

namespace ha {
namespace {

constexpr int kWideWarps = kScoreThreads / 32;

// The W code words of token i into registers (16-byte loads when W is a multiple of 4).
template <int W>
__device__ __forceinline__ void load_words(const uint32_t* __restrict__ row, int64_t i, uint32_t (&kw)[W]) {
    const uint32_t* k = row + i * W;
    if constexpr ((W & 3) == 0) {
#pragma unroll
        for (int w = 0; w < W; w += 4) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(k + w));
            kw[w] = v.x;
            kw[w + 1] = v.y;
            kw[w + 2] = v.z;
            kw[w + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int w = 0; w < W; ++w) kw[w] = __ldg(k + w);
    }
}

// Distance of the words in kw to query code qw[0..W) (shared memory).
template <int W>
__device__ __forceinline__ int words_dist(const uint32_t (&kw)[W], const uint32_t* qw) {
    int d = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) d += __popc(kw[w] ^ qw[w]);
    return d;
}

// dynamic shared memory: kMaxHeadsPerPass * (NB + W) words
template <int W>
__global__ void __launch_bounds__(kScoreThreads) k_score_wide(const WideParams p) {
    extern __shared__ uint32_t s_dyn[];
    uint32_t* s_hist = s_dyn;                               // [kMaxHeadsPerPass][NB]
    uint32_t* s_qw = s_dyn + kMaxHeadsPerPass * p.NB;       // [kMaxHeadsPerPass][W]
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
    const int c0 = c * p.chunk, c1 = min(n, c0 + p.chunk);
    if (c0 >= n) return;
    const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)g * p.ks_sh;

    for (int hp = 0; hp < p.G; hp += kMaxHeadsPerPass) {
        const int nh = min(kMaxHeadsPerPass, p.G - hp);
        for (int x = tid; x < kMaxHeadsPerPass * p.NB; x += kScoreThreads) s_hist[x] = 0u;
        for (int x = tid; x < nh * W; x += kScoreThreads)
            s_qw[x] = p.q_sig[(int64_t)(head0 + hp + x / W) * W + x % W];
        __syncthreads();
        for (int i = c0 + tid; i < c1; i += kScoreThreads) {
            uint32_t kw[W];
            load_words<W>(row, i, kw);  // one read of the token's code serves every head of the pass
            for (int e = 0; e < nh; ++e) atomicAdd(&s_hist[e * p.NB + words_dist<W>(kw, s_qw + e * W)], 1u);
        }
        __syncthreads();
        for (int x = tid; x < nh * p.NB; x += kScoreThreads) {
            const int e = x / p.NB, u = x - e * p.NB;
            p.chunk_hist[((int64_t)(head0 + hp + e) * p.nchunks + c) * p.NB + u] = s_hist[x];
        }
        __syncthreads();
    }

    // ---- the last CTA of this (sequence, KV head): thresholds and chunk quotas
    const int nch = (n + p.chunk - 1) / p.chunk;
    __syncthreads();
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
    const int k = min(mb, n);
    for (int e = warp; e < p.G; e += kWideWarps) {
        const int64_t h = head0 + e;
        const uint32_t* H = p.chunk_hist + h * p.nchunks * p.NB;
        // t: the smallest bin whose cumulative count reaches k (bins in groups of 32)
        int t = p.NB - 1, below = 0, carry = 0;
        bool found = false;
        for (int u0 = 0; u0 < p.NB && !found; u0 += 32) {
            const int u = u0 + lane;
            int tot = 0;
            for (int cc0 = 0; cc0 < nch; cc0 += 16) {  // 16 loads in flight
                int v[16];
#pragma unroll
                for (int x = 0; x < 16; ++x)
                    v[x] = (u < p.NB && cc0 + x < nch) ? (int)__ldcg(H + (int64_t)(cc0 + x) * p.NB + u) : 0;
#pragma unroll
                for (int x = 0; x < 16; ++x) tot += v[x];
            }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned reach = __ballot_sync(0xffffffffu, u < p.NB && carry + incl >= k);
            if (reach) {
                const int l = __ffs(reach) - 1;
                t = u0 + l;
                below = carry + __shfl_sync(0xffffffffu, incl - tot, l);
                found = true;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (!found) below = carry;  // cannot happen: every token lies in a bin
        const int r = k - below;
        int tcarry = 0;  // tied tokens in the chunks before
        for (int base = 0; base < nch; base += 32) {
            const int cc = base + lane;
            const int v = (cc < nch) ? (int)__ldcg(H + (int64_t)cc * p.NB + t) : 0;
            int in = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, in, o);
                if (lane >= o) in += y;
            }
            if (cc < nch) p.meta_qt[h * p.nchunks + cc] = make_int2(r - (tcarry + in - v), v);
            tcarry += __shfl_sync(0xffffffffu, in, 31);
        }
        if (lane == 0) p.meta_t[h] = t;
    }
    if (tid == 0) p.score_cnt[bg] = 0u;
}

__device__ __forceinline__ uint32_t wide_warp_incl_scan(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// dynamic shared memory: kMaxHeadsPerPass * W words (the pass's query codes)
template <int W>
__global__ void __launch_bounds__(kScoreThreads) k_select_wide(const WideParams p) {
    extern __shared__ uint32_t s_qw[];
    __shared__ int s_wt[kMaxHeadsPerPass * kWideWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x % p.nchunks;
    const int bg = blockIdx.x / p.nchunks;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, false);
    const int nch = (n + p.chunk - 1) / p.chunk;
    if (c >= nch) return;
    pdl_launch_dependents();
    pdl_wait();  // SCORE's thresholds are read below

    const int tpt = p.chunk / kScoreThreads;
    const int SC = 32 * tpt;
    const int head0 = b * p.Hq + g * p.G;
    const int nseg = p.nchunks * kWideWarps;
    const int sc = c * kWideWarps + warp;
    const int lbase = c * p.chunk + warp * SC + lane * tpt;
    const int wlo = min(p.n_sink, n), whi = max(0, n - p.n_local);
    const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)g * p.ks_sh;

    for (int hp = 0; hp < p.G; hp += kMaxHeadsPerPass) {
        const int nh = min(kMaxHeadsPerPass, p.G - hp);
        __syncthreads();  // the previous pass is done with s_qw and s_wt
        for (int x = tid; x < nh * W; x += kScoreThreads)
            s_qw[x] = p.q_sig[(int64_t)(head0 + hp + x / W) * W + x % W];
        __syncthreads();
        // thresholds and tie quotas of the pass's heads
        int t[kMaxHeadsPerPass], mode[kMaxHeadsPerPass], left[kMaxHeadsPerPass];
        int qx[kMaxHeadsPerPass];
        bool boundary = false;
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            t[e] = 0;
            mode[e] = 0;
            qx[e] = 0;
            if (e < nh) {
                const int64_t h = head0 + hp + e;
                const int2 mq = p.meta_qt[h * p.nchunks + c];
                t[e] = p.meta_t[h];
                qx[e] = mq.x;
                mode[e] = (mq.x <= 0) ? 0 : (mq.x >= mq.y ? 1 : 2);
            }
            left[e] = (mode[e] == 1) ? tpt : 0;
            boundary = boundary || (mode[e] == 2);
        }
        if (boundary) {  // uniform across the CTA: ranks of the tied tokens across warps and lanes
            int ties[kMaxHeadsPerPass] = {0, 0, 0, 0};
            for (int j = 0; j < tpt; ++j) {
                const int i = lbase + j;
                if (i >= n) break;
                uint32_t kw[W];
                load_words<W>(row, i, kw);
#pragma unroll
                for (int e = 0; e < kMaxHeadsPerPass; ++e)
                    if (mode[e] == 2) ties[e] += (words_dist<W>(kw, s_qw + e * W) == t[e]) ? 1 : 0;
            }
#pragma unroll
            for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                if (mode[e] == 2) {
                    const int wsum = __reduce_add_sync(0xffffffffu, ties[e]);
                    if (lane == 0) s_wt[e * kWideWarps + warp] = wsum;
                }
            }
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                if (mode[e] == 2) {
                    int before = (int)(wide_warp_incl_scan((uint32_t)ties[e]) - (uint32_t)ties[e]);
                    for (int w2 = 0; w2 < warp; ++w2) before += s_wt[e * kWideWarps + w2];
                    left[e] = min(max(qx[e] - before, 0), ties[e]);
                }
            }
        }
        // selection masks: one read of every token's code serves the pass's heads
        uint32_t msk[kMaxHeadsPerPass] = {0u, 0u, 0u, 0u};
        for (int j = 0; j < tpt; ++j) {
            const int i = lbase + j;
            if (i >= n) break;
            uint32_t kw[W];
            load_words<W>(row, i, kw);
            const bool inw = (i < wlo) || (i >= whi);
#pragma unroll
            for (int e = 0; e < kMaxHeadsPerPass; ++e) {
                if (e < nh) {
                    const int d = words_dist<W>(kw, s_qw + e * W);
                    bool take = d < t[e];
                    if (d == t[e] && left[e] > 0) {
                        take = true;
                        --left[e];
                    }
                    if (take || inw) msk[e] |= 1u << j;
                }
            }
        }
#pragma unroll
        for (int e = 0; e < kMaxHeadsPerPass; ++e) {
            if (e < nh) {
                const int64_t h = head0 + hp + e;
                const uint32_t cnt = (uint32_t)__popc(msk[e]);
                const uint32_t incl = wide_warp_incl_scan(cnt);
                int32_t* seg = p.seg_idx + h * (int64_t)nseg * SC + (int64_t)sc * SC;
                int w = (int)(incl - cnt);
                uint32_t x = msk[e];
                while (x != 0u) {
                    const int j = __ffs(x) - 1;
                    x &= x - 1u;
                    seg[w++] = lbase + j;
                }
                if (lane == 31) p.seg_cnt[h * nseg + sc] = (int)incl;
            }
        }
    }
}

}  // namespace

cudaError_t launch_score_wide(const WideParams& p, int batch_hkv, cudaStream_t st) {
    const size_t smem = (size_t)kMaxHeadsPerPass * (p.NB + p.W) * sizeof(uint32_t);
    const unsigned grid = (unsigned)batch_hkv * (unsigned)p.nchunks;
    switch (p.W) {
        case 2: k_score_wide<2><<<grid, kScoreThreads, smem, st>>>(p); break;
        case 4: k_score_wide<4><<<grid, kScoreThreads, smem, st>>>(p); break;
        case 8: k_score_wide<8><<<grid, kScoreThreads, smem, st>>>(p); break;
        case 16: k_score_wide<16><<<grid, kScoreThreads, smem, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_select_wide(const WideParams& p, int batch_hkv, cudaStream_t st, bool pdl) {
    const size_t smem = (size_t)kMaxHeadsPerPass * p.W * sizeof(uint32_t);
    const dim3 grid((unsigned)batch_hkv * (unsigned)p.nchunks), block(kScoreThreads);
    switch (p.W) {
        case 2: return launch_ex(k_select_wide<2>, grid, block, smem, st, pdl, p);
        case 4: return launch_ex(k_select_wide<4>, grid, block, smem, st, pdl, p);
        case 8: return launch_ex(k_select_wide<8>, grid, block, smem, st, pdl, p);
        case 16: return launch_ex(k_select_wide<16>, grid, block, smem, st, pdl, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ha
