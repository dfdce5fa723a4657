// The exact comparator of the hashed selection and its recall.
//
// HashAttention: Semantic Sparsity for Faster Inference, Sec. 5 measures the
// hashed selection against the oracle top-k by attention score. Here:
//   k_dot_scores   z[head, i] = <q[b, h], k_i> (float32) for every cached token
//                  i < n on the CUDA cores, for the keys the tensor-core kernel
//                  does not take (float32 keys, more than 21 query heads per
//                  KV head); one read of a KV head's rows serves its G query
//                  heads (4 lanes share a row, 16-byte loads, q in shared
//                  memory).
//   k_topk_exact   per head, the min(m, n) largest z (ties: smaller index),
//                  by radix select over order-preserving 32-bit keys: a
//                  threshold from a 1/16 sample admits a few thousand
//                  candidates into shared memory in one pass over the
//                  scores, the exact select runs on those, and a token bitmap
//                  gives the ascending list (-1 padded); when the estimate
//                  misses, four 8-bit passes over all scores and a compaction
//                  pass in token order.
//   k_recall       per head, |selected & reference| / |reference|: the
//                  reference list is staged in shared memory in tiles and every
//                  selected index is looked up by binary search.
#include "ha_internal.cuh"

#include <math_constants.h>

namespace ha {
namespace {

constexpr int kScoreRowsPerCta = 1024;
constexpr int kTopkThreads = 512;
constexpr int kCandCap = 10240;        // candidate tokens held in shared memory
constexpr int kSampleCap = 8192;       // sampled scores (in the candidate key array)
constexpr int kTieCap = 1024;          // tokens equal to the k-th largest key, fast path
constexpr int kBitmapTokens = 1 << 18; // fast path up to this n_cap (a bitmap of n_cap bits)
constexpr int kRecallThreads = 256;
constexpr int kRecallTile = 8192;

template <typename KT>
__device__ __forceinline__ void to_float8(const uint4 w, float* f);

template <>
__device__ __forceinline__ void to_float8<__nv_bfloat16>(const uint4 w, float* f) {
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
    f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
    f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

template <>
__device__ __forceinline__ void to_float8<float>(const uint4 w, float* f) {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
}

// grid: (token blocks of kScoreRowsPerCta, B * Hkv): CTAs launched together
// stream consecutive blocks of one KV head (the heads' K regions are a power of
// two apart, which same-offset reads across heads would concentrate on few
// memory channels); 256 threads; dynamic shared memory G * D floats.
// GQ: the group size when it is known at compile time (4: the heads' loop
// unrolls), else 0 (a run-time loop over p.G).
template <int D, typename KT, int GQ>
__global__ void __launch_bounds__(256, 4) k_dot_scores(const ExactParams p) {
    constexpr int ES = sizeof(KT);
    constexpr int NCH = D * ES / 16;  // 16-byte chunks per row
    constexpr int CPL = NCH / 4;      // chunks per lane (4 lanes per row)
    constexpr int EPC = 16 / ES;      // elements per chunk
    extern __shared__ float s_q[];    // [G][D]
    const int bg = blockIdx.y;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, blockIdx.x == 0 && g == 0 && threadIdx.x == 0);
    for (int i = threadIdx.x; i < p.G * D; i += blockDim.x) {
        const int hh = i / D, k = i - hh * D;
        const int64_t off = (int64_t)b * p.q_sb + (int64_t)(g * p.G + hh) * p.q_sh + k;
        s_q[i] = p.q_bf16 ? __uint_as_float(((uint32_t) reinterpret_cast<const uint16_t*>(p.q)[off]) << 16)
                          : reinterpret_cast<const float*>(p.q)[off];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane & 7, qt = lane >> 3;
    const char* Kb = p.K + ((int64_t)b * p.k_sb + (int64_t)g * p.k_sh) * ES;
    const int row_end = min(n, (int)(blockIdx.x + 1) * kScoreRowsPerCta);
    auto load_rows = [&](int row0, uint4 (&w)[CPL]) {
        const int row = row0 + r;
#pragma unroll
        for (int jc = 0; jc < CPL; ++jc)
            w[jc] = (row < row_end) ? __ldg(reinterpret_cast<const uint4*>(Kb + (int64_t)row * p.k_sn * ES +
                                                                          (jc * 4 + qt) * 16))
                                    : make_uint4(0u, 0u, 0u, 0u);
    };
    // each warp walks 8-row tiles; the next tile's rows load while this one is scored
    int row0 = blockIdx.x * kScoreRowsPerCta + warp * 8;
    uint4 wc[CPL];
    if (row0 < row_end) load_rows(row0, wc);
    for (; row0 < row_end; row0 += 8 * 8) {
        uint4 wn[CPL];
        if (row0 + 64 < row_end) load_rows(row0 + 64, wn);
        const int row = row0 + r;
        float f[CPL * EPC];  // this lane's elements of the row, converted once for every head
#pragma unroll
        for (int jc = 0; jc < CPL; ++jc) to_float8<KT>(wc[jc], f + jc * EPC);
        const int G = GQ ? GQ : p.G;
        auto head_score = [&](int hh) {
            const float* qh = s_q + hh * D;
            float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int jc = 0; jc < CPL; ++jc) {
#pragma unroll
                for (int e = 0; e < EPC; e += 4) {
                    const float4 q4 = *reinterpret_cast<const float4*>(qh + (jc * 4 + qt) * EPC + e);
                    a2 = __ffma2_rn(make_float2(q4.x, q4.y), make_float2(f[jc * EPC + e], f[jc * EPC + e + 1]), a2);
                    a2 = __ffma2_rn(make_float2(q4.z, q4.w), make_float2(f[jc * EPC + e + 2], f[jc * EPC + e + 3]),
                                    a2);
                }
            }
            float acc = a2.x + a2.y;
            acc += __shfl_xor_sync(0xffffffffu, acc, 8);
            acc += __shfl_xor_sync(0xffffffffu, acc, 16);
            if (qt == 0 && row < row_end)
                p.scores[((int64_t)b * p.Hq + g * G + hh) * p.n_cap + row] = acc;
        };
        if constexpr (GQ > 0) {
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) head_score(hh);
        } else {
#pragma unroll 1
            for (int hh = 0; hh < G; ++hh) head_score(hh);
        }
#pragma unroll
        for (int jc = 0; jc < CPL; ++jc) wc[jc] = wn[jc];
    }
}

// Order-preserving key of a float: larger float, larger key.
__device__ __forceinline__ uint32_t fkey(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sum of one int per thread; returns the exclusive
// value and writes the block total to *total (every thread).
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int y = (lane < nw) ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        if (lane < nw) s_warp[lane] = y;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    *total = s_warp[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before;
}

// Warp 0 of the block: given the histogram of the keys still in play (those
// whose resolved high bits equal `prefix`), find the bin of the need-th
// largest and publish the extended prefix and the count still needed in it.
__device__ __forceinline__ void pick_bin(const unsigned* s_hist, int need, uint32_t prefix, int shift,
                                         uint32_t* s_prefix, int* s_need) {
    const int lane = threadIdx.x & 31;
    unsigned c[8], sum = 0u;  // lane l holds bins 255 - 8l ... 248 - 8l
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        c[u] = s_hist[255 - 8 * lane - u];
        sum += c[u];
    }
    unsigned incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    unsigned above = incl - sum;  // keys in the bins above this lane's
    const unsigned hit = __ballot_sync(0xffffffffu, above < (unsigned)need && (unsigned)need <= incl);
    if (lane == __ffs(hit) - 1) {
        int bin = 255 - 8 * lane;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (above + c[u] >= (unsigned)need) {
                bin = 255 - 8 * lane - u;
                break;
            }
            above += c[u];
        }
        *s_prefix = prefix | ((uint32_t)bin << shift);
        *s_need = need - (int)above;
    }
}

// Radix select over keys[0, cnt) in shared memory: resolves `passes` 8-bit
// digits (from the top) of the need-th largest key. With 4 passes, prefix is
// that key and need the number of keys equal to it among the largest `need`;
// with fewer, prefix has its low bits zero and at least `need` keys are >= it.
// Lanes with equal digits are merged (match_any) before the shared atomics:
// scores cluster in few high-order bins.
__device__ void smem_radix_select(const uint32_t* keys, int cnt, int need, int passes, unsigned* s_hist,
                                  uint32_t* s_prefix, int* s_need, uint32_t& prefix_out, int& need_out) {
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t prefix = 0u, mask = 0u;
    if (tid == 0) {
        *s_prefix = 0u;
        *s_need = need;
    }
    for (int pass = 0; pass < passes; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += blockDim.x) s_hist[i] = 0u;
        __syncthreads();
        for (int i0 = 0; i0 < cnt; i0 += 8 * blockDim.x) {  // 8 keys per thread loaded before counting
            uint32_t kv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * blockDim.x + tid;
                kv[u] = (i < cnt) ? keys[i] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * blockDim.x + tid;
                const bool in = i < cnt && (kv[u] & mask) == prefix;
                const unsigned bin = in ? (kv[u] >> shift) & 0xFFu : 256u;
                const unsigned peers = __match_any_sync(0xffffffffu, bin);
                if (in && lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], (unsigned)__popc(peers));
            }
        }
        __syncthreads();
        if (tid < 32) pick_bin(s_hist, need, prefix, shift, s_prefix, s_need);
        __syncthreads();
        prefix = *s_prefix;
        need = *s_need;
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    prefix_out = prefix;
    need_out = need;
}

// Ascending output of the selected tokens of one block of up to 32 consecutive
// tokens per thread: take/tie bit u = token ib + u. Ties are taken in token
// order while fewer than `need` have been taken; out_base and ties_seen
// advance by the block's totals (uniform across the block).
__device__ __forceinline__ void emit_block(uint32_t take, uint32_t tie, int ib, int need, int* s_warp,
                                           int32_t* dst, int idx_cap, int& out_base, int& ties_seen) {
    int ties_total;
    const int tie_before = block_excl_scan(__popc(tie), s_warp, &ties_total);
    int rank = ties_seen + tie_before;  // ties of the tokens before this thread's
    for (uint32_t t = tie; t != 0u; t &= t - 1u) {
        if (rank < need) take |= t & (0u - t);
        ++rank;
    }
    ties_seen += ties_total;
    int taken_total;
    int pos = out_base + block_excl_scan(__popc(take), s_warp, &taken_total);
    for (uint32_t t = take; t != 0u; t &= t - 1u) {
        if (pos < idx_cap) dst[pos] = ib + __ffs(t) - 1;
        ++pos;
    }
    out_base += taken_total;
}

constexpr int kOffBins = 2 * kTopkThreads;   // 16-bit prefixes below the largest, one histogram pass
constexpr int kVec = 4;                      // float4 loads per thread per batch of the candidate pass

// Block-wide maximum (every thread gets it).
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* s_red) {
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t m = 0u;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) m = max(m, s_red[w]);
    __syncthreads();
    return m;
}

// The 16-bit prefix of the need-th largest of keys[0, cnt) (shared memory) from
// one histogram of off = top16 - (key >> 16) over kOffBins bins, top16 being the
// prefix of the largest key. Returns false (block-uniform) when that key lies
// kOffBins or more prefixes below the largest; else its prefix p16, its rank
// among the keys of its prefix (1-based) and their count.
__device__ bool select16_onepass(const uint32_t* keys, int cnt, int need, uint32_t top16, unsigned* s_bins,
                                 int* s_warp, int* s_res, uint32_t& p16, int& rank_in, int& bin_cnt) {
    const int tid = threadIdx.x;
    if (tid == 0) s_res[0] = -1;
    for (int i = tid; i < kOffBins; i += kTopkThreads) s_bins[i] = 0u;
    __syncthreads();
    for (int i = tid; i < cnt; i += kTopkThreads) {
        const uint32_t off = top16 - (keys[i] >> 16);
        if (off < (uint32_t)kOffBins) atomicAdd(&s_bins[off], 1u);
    }
    __syncthreads();
    const int c0 = (int)s_bins[2 * tid], c1 = (int)s_bins[2 * tid + 1];
    int total;
    const int before = block_excl_scan(c0 + c1, s_warp, &total);  // keys with larger prefixes
    if (before < need && need <= before + c0 + c1) {
        const bool first = need <= before + c0;
        s_res[0] = first ? 2 * tid : 2 * tid + 1;
        s_res[1] = need - (first ? before : before + c0);
        s_res[2] = first ? c0 : c1;
    }
    __syncthreads();
    const int bin = s_res[0];
    p16 = top16 - (uint32_t)bin;
    rank_in = s_res[1];
    bin_cnt = s_res[2];
    __syncthreads();
    return bin >= 0;
}

// Exact need-th largest of keys[0, cnt) and the number of keys equal to it among
// the largest `need`: one prefix histogram, then a rank by counting inside the
// one 16-bit prefix that holds it (its keys gathered into s_list). False
// (block-uniform) when the prefix lies out of the histogram's reach or holds more
// than kTieCap keys.
__device__ bool bin_select(const uint32_t* keys, int cnt, int need, uint32_t top16, unsigned* s_bins, int* s_warp,
                           int* s_res, uint32_t* s_list, int* s_lcount, uint32_t* s_prefix, int* s_need,
                           uint32_t& kth, int& need_out) {
    const int tid = threadIdx.x;
    uint32_t p16;
    int rank_in, bc;
    if (!select16_onepass(keys, cnt, need, top16, s_bins, s_warp, s_res, p16, rank_in, bc)) return false;
    if (bc > kTieCap) return false;
    if (tid == 0) *s_lcount = 0;
    __syncthreads();
    for (int i = tid; i < cnt; i += kTopkThreads) {
        const uint32_t key = keys[i];
        if ((key >> 16) == p16) s_list[atomicAdd(s_lcount, 1)] = key;
    }
    __syncthreads();
    for (int j = tid; j < bc; j += kTopkThreads) {
        const uint32_t x = s_list[j];
        int gt = 0, eq = 0;
        for (int l = 0; l < bc; ++l) {
            const uint32_t y = s_list[l];
            gt += (y > x) ? 1 : 0;
            eq += (y == x) ? 1 : 0;
        }
        if (gt < rank_in && rank_in <= gt + eq) {  // every such thread holds the same key
            *s_prefix = x;
            *s_need = rank_in - gt;
        }
    }
    __syncthreads();
    kth = *s_prefix;
    need_out = *s_need;
    __syncthreads();
    return true;
}

__device__ __forceinline__ float f4_comp(const float4& v, int c) {
    return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

__device__ __forceinline__ void load_f4(const float4* z4, int n4, int base, float4 (&b)[kVec]) {
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
        const int i4 = base + u * kTopkThreads + threadIdx.x;
        b[u] = (i4 < n4) ? __ldcg(z4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Append the tokens flagged in tk (bit e: value val(e), token idx(e)) to the
// candidate arrays: one slot reservation per warp (inclusive scan of the lanes'
// counts); cmax tracks the largest appended key.
template <int NB, typename ValF, typename IdxF>
__device__ __forceinline__ void append_candidates(uint32_t tk, ValF val, IdxF idx, int* s_ccount, uint32_t* s_ckey,
                                                  int* s_cidx, uint32_t& cmax) {
    const int lane = threadIdx.x & 31;
    const int c = __popc(tk);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int wbase = 0;
    if (lane == 31 && incl > 0) wbase = atomicAdd(s_ccount, incl);
    int pos = __shfl_sync(0xffffffffu, wbase, 31) + incl - c;
#pragma unroll
    for (int e = 0; e < NB; ++e) {
        if ((tk >> e) & 1u) {
            const uint32_t key = fkey(val(e));
            cmax = max(cmax, key);
            if (pos < kCandCap) {
                s_ckey[pos] = key;
                s_cidx[pos] = idx(e);
            }
            ++pos;
        }
    }
}

// One CTA (kTopkThreads) per query head: the k = min(m, n) largest scores.
//  fast path (n within the bitmap capacity): a 16-bit threshold T16 from a
//   1/16 sample (8 consecutive tokens out of every 128, so the sample costs
//   1/16 of the sectors) with the target rank raised well past k's share; one
//   pass collects every token with key >= T16 into shared memory; when their
//   count lies in [k, kCandCap] the exact k-th largest key is among them
//   (at least k keys are >= T16), so the exact radix select runs on the
//   candidates alone; the tokens above the k-th key and the smallest-index
//   tokens equal to it are marked in a token bitmap, which is written out in
//   token order.
//  Ties beyond kTieCap (degenerate inputs) take the general path.
//  otherwise: radix select over all n scores (four passes of 8 bits) and a
//   compaction pass in token order.
__global__ void __launch_bounds__(kTopkThreads) k_topk_exact(const ExactParams p) {
    extern __shared__ uint32_t s_dyn[];
    uint32_t* s_ckey = s_dyn;                              // [kCandCap] (the sample first)
    int* s_cidx = reinterpret_cast<int*>(s_dyn + kCandCap);  // [kCandCap]
    uint32_t* s_sel = s_dyn + 2 * kCandCap;                // [bitmap_words]
    int* s_tlist = reinterpret_cast<int*>(s_sel + p.bitmap_words);  // [kTieCap]
    __shared__ unsigned s_hist[256];
    __shared__ int s_warp[kTopkThreads / 32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    __shared__ int s_ccount, s_tcount, s_lcount;
    __shared__ unsigned s_bins[kOffBins];
    __shared__ uint32_t s_red[kTopkThreads / 32];
    __shared__ int s_res[3];
    const int head = blockIdx.x;
    const int b = head / p.Hq;
    const int tid = threadIdx.x, lane = tid & 31;
    const int n = checked_len(p.seq_lens, b, p.n_cap, nullptr, false);
    const int k = max(0, min(p.m, n));
    const float* z = p.scores + (int64_t)head * p.n_cap;
    int32_t* dst = p.idx + (int64_t)head * p.idx_cap;
    int out_base = 0;

    if (k > 0 && k >= n) {  // every token
        for (int i = tid; i < n; i += kTopkThreads)
            if (i < p.idx_cap) dst[i] = i;
        out_base = n;
    } else if (k > 0) {
        bool fast = p.bitmap_words > 0 && n <= 32 * p.bitmap_words;
        if (fast) {
            // ---- sample: blocks of 8 tokens, one every 8 * step tokens. The first
            // batch of the candidate pass loads with it (it needs no threshold).
            const int step = (n + kSampleCap - 9) / (kSampleCap - 8);
            const int nb = (n + 8 * step - 1) / (8 * step);
            const int ns = min(nb * 8, (nb - 1) * 8 + (n - (nb - 1) * 8 * step));
            const int n4 = ((p.n_cap & 3) == 0) ? (n >> 2) : 0;  // float4 part (16-byte aligned rows)
            const float4* z4 = reinterpret_cast<const float4*>(z);
            float4 cur[kVec];
            load_f4(z4, n4, 0, cur);
            uint32_t smax = 0u;
            {
                constexpr int kPerThread = kSampleCap / kTopkThreads;  // all loads in flight at once
                float v[kPerThread];
#pragma unroll
                for (int u = 0; u < kPerThread; ++u) {
                    const int s = tid + u * kTopkThreads;
                    v[u] = (s < ns) ? __ldcg(z + (int64_t)(s >> 3) * 8 * step + (s & 7)) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < kPerThread; ++u) {
                    const int s = tid + u * kTopkThreads;
                    if (s < ns) {
                        const uint32_t key = fkey(v[u]);
                        s_ckey[s] = key;
                        smax = max(smax, key);
                    }
                }
            }
            smax = block_max_u32(smax, s_red);
            const float share = (float)k * (float)ns / (float)n;  // k's expected rank in the sample
            const int r = min(ns, (int)ceilf(1.25f * share + 4.f * sqrtf(share) + 8.f));
            fast = (float)r * ((float)n / (float)ns) <= 0.8f * (float)kCandCap;
            if (fast) {
                uint32_t t16;
                {
                    uint32_t p16;
                    int rank_in, bc;
                    if (select16_onepass(s_ckey, ns, r, smax >> 16, s_bins, s_warp, s_res, p16, rank_in, bc)) {
                        t16 = p16 << 16;
                    } else {
                        int unused;
                        smem_radix_select(s_ckey, ns, r, 2, s_hist, &s_prefix, &s_need, t16, unused);
                    }
                }
                // ---- candidates: every token with key >= t16
                if (tid == 0) {
                    s_ccount = 0;
                    s_tcount = 0;
                }
                __syncthreads();
                uint32_t cmax = 0u;
                for (int base = 0; base < n4; base += kVec * kTopkThreads) {  // the next batch loads meanwhile
                    float4 nxt[kVec];
                    if (base + kVec * kTopkThreads < n4) load_f4(z4, n4, base + kVec * kTopkThreads, nxt);
                    uint32_t tk = 0u;  // bit 4u + c: element c of float4 base + u * kTopkThreads + tid
#pragma unroll
                    for (int u = 0; u < kVec; ++u) {
                        const bool in = base + u * kTopkThreads + tid < n4;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (in && fkey(f4_comp(cur[u], c)) >= t16) tk |= 1u << (4 * u + c);
                    }
                    append_candidates<4 * kVec>(
                        tk, [&](int e) { return f4_comp(cur[e >> 2], e & 3); },
                        [&](int e) { return 4 * (base + (e >> 2) * kTopkThreads + tid) + (e & 3); }, &s_ccount, s_ckey,
                        s_cidx, cmax);
#pragma unroll
                    for (int u = 0; u < kVec; ++u) cur[u] = nxt[u];
                }
                constexpr int kInFlight = 16;  // the tokens past the float4 part (all when rows are unaligned)
                for (int i0 = 4 * n4; i0 < n; i0 += kInFlight * kTopkThreads) {
                    float v[kInFlight];
#pragma unroll
                    for (int u = 0; u < kInFlight; ++u) {
                        const int i = i0 + u * kTopkThreads + tid;
                        v[u] = (i < n) ? __ldcg(z + i) : 0.f;
                    }
                    uint32_t tk = 0u;  // bit u: token i0 + u * kTopkThreads + tid
#pragma unroll
                    for (int u = 0; u < kInFlight; ++u)
                        if (i0 + u * kTopkThreads + tid < n && fkey(v[u]) >= t16) tk |= 1u << u;
                    append_candidates<kInFlight>(
                        tk, [&](int e) { return v[e]; }, [&](int e) { return i0 + e * kTopkThreads + tid; },
                        &s_ccount, s_ckey, s_cidx, cmax);
                }
                __syncthreads();
                cmax = block_max_u32(cmax, s_red);
                const int cc = s_ccount;
                fast = cc >= k && cc <= kCandCap;
                if (fast) {
                    // ---- exact k-th largest among the candidates, then the bitmap
                    uint32_t kth;
                    int need;
                    if (!bin_select(s_ckey, cc, k, cmax >> 16, s_bins, s_warp, s_res,
                                    reinterpret_cast<uint32_t*>(s_tlist), &s_lcount, &s_prefix, &s_need, kth, need))
                        smem_radix_select(s_ckey, cc, k, 4, s_hist, &s_prefix, &s_need, kth, need);
                    const int nw = (n + 31) >> 5;
                    for (int w = tid; w < nw; w += kTopkThreads) s_sel[w] = 0u;
                    __syncthreads();
                    for (int c = tid; c < cc; c += kTopkThreads) {
                        const uint32_t key = s_ckey[c];
                        const int i = s_cidx[c];
                        if (key > kth) {
                            atomicOr(&s_sel[i >> 5], 1u << (i & 31));
                        } else if (key == kth) {
                            const int t = atomicAdd(&s_tcount, 1);
                            if (t < kTieCap) s_tlist[t] = i;
                        }
                    }
                    __syncthreads();
                    const int tc = s_tcount;
                    fast = tc <= kTieCap;
                    if (fast) {
                        // the `need` smallest indices among the ties: rank by counting
                        for (int j = tid; j < tc; j += kTopkThreads) {
                            const int i = s_tlist[j];
                            int rank = 0;
                            if (need < tc)
                                for (int l = 0; l < tc; ++l) rank += (s_tlist[l] < i) ? 1 : 0;
                            if (rank < need) atomicOr(&s_sel[i >> 5], 1u << (i & 31));
                        }
                        __syncthreads();
                        // 8 consecutive bitmap words (256 tokens) per thread, in token order
                        for (int w0 = 0; w0 < nw; w0 += 8 * kTopkThreads) {
                            const int wb = w0 + 8 * tid;
                            uint32_t wv[8];
                            if (wb + 8 <= nw) {
                                const uint4 a = *reinterpret_cast<const uint4*>(s_sel + wb);
                                const uint4 c = *reinterpret_cast<const uint4*>(s_sel + wb + 4);
                                wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
                                wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
                            } else {
#pragma unroll
                                for (int u = 0; u < 8; ++u) wv[u] = (wb + u < nw) ? s_sel[wb + u] : 0u;
                            }
                            int mine = 0;
#pragma unroll
                            for (int u = 0; u < 8; ++u) mine += __popc(wv[u]);
                            int total;
                            int pos = out_base + block_excl_scan(mine, s_warp, &total);
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                for (uint32_t t = wv[u]; t != 0u; t &= t - 1u) {
                                    if (pos < p.idx_cap) dst[pos] = (wb + u) * 32 + __ffs(t) - 1;
                                    ++pos;
                                }
                            out_base += total;
                        }
                    }
                }
            }
        }
        if (!fast) {
            // ---- radix select over all n scores, then a compaction pass
            uint32_t prefix = 0u, mask = 0u;
            int need = k;
            if (tid == 0) {
                s_prefix = 0u;
                s_need = need;
            }
            for (int shift = 24; shift >= 0; shift -= 8) {
                for (int i = tid; i < 256; i += kTopkThreads) s_hist[i] = 0u;
                __syncthreads();
                for (int i0 = 0; i0 < n; i0 += 8 * kTopkThreads) {  // 8 loads in flight per thread
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = i0 + u * kTopkThreads + tid;
                        v[u] = (i < n) ? __ldcg(z + i) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t key = fkey(v[u]);
                        const bool in = i0 + u * kTopkThreads + tid < n && (key & mask) == prefix;
                        const unsigned bin = in ? (key >> shift) & 0xFFu : 256u;
                        const unsigned peers = __match_any_sync(0xffffffffu, bin);
                        if (in && lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], (unsigned)__popc(peers));
                    }
                }
                __syncthreads();
                if (tid < 32) pick_bin(s_hist, need, prefix, shift, &s_prefix, &s_need);
                __syncthreads();
                prefix = s_prefix;
                need = s_need;
                mask |= 0xFFu << shift;
                __syncthreads();
            }
            // each thread takes 8 consecutive tokens of a block of 8 * kTopkThreads
            constexpr int kPer = 8;
            int ties_seen = 0;
            for (int i0 = 0; i0 < n; i0 += kPer * kTopkThreads) {
                const int ib = i0 + tid * kPer;
                uint32_t take = 0u, tie = 0u;  // bit u: token ib + u
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int i = ib + u;
                    if (i < n) {
                        const uint32_t key = fkey(__ldcg(z + i));
                        if (key > prefix) take |= 1u << u;
                        if (key == prefix) tie |= 1u << u;
                    }
                }
                emit_block(take, tie, ib, need, s_warp, dst, p.idx_cap, out_base, ties_seen);
            }
        }
    }
    for (int t = k + tid; t < p.idx_cap; t += kTopkThreads) dst[t] = -1;
    if (tid == 0) {
        p.cnt[head] = k;
        if (out_base != k) flag_error(p.err, HA_DEVERR_STATE);
    }
}

// One CTA per head: recall[head] = |selected & reference| / |reference|.
__global__ void __launch_bounds__(kRecallThreads) k_recall(const RecallParams p) {
    __shared__ int s_ref[kRecallTile];
    __shared__ int s_sum[kRecallThreads / 32];
    const int head = blockIdx.x;
    const int tid = threadIdx.x;
    const int na = min(max(p.sel_cnt[head], 0), p.sel_cap);
    const int nb = min(max(p.ref_cnt[head], 0), p.ref_cap);
    const int32_t* A = p.sel_idx + (int64_t)head * p.sel_cap;
    const int32_t* Bv = p.ref_idx + (int64_t)head * p.ref_cap;
    int hits = 0;
    for (int t0 = 0; t0 < nb; t0 += kRecallTile) {
        const int tn = min(kRecallTile, nb - t0);
        __syncthreads();
        for (int i = tid; i < tn; i += kRecallThreads) s_ref[i] = Bv[t0 + i];
        __syncthreads();
        for (int i = tid; i < na; i += kRecallThreads) {
            const int x = A[i];
            int lo = 0, hi = tn - 1;
            while (lo < hi) {  // the reference list is ascending
                const int mid = (lo + hi) >> 1;
                if (s_ref[mid] < x) lo = mid + 1; else hi = mid;
            }
            hits += (s_ref[lo] == x) ? 1 : 0;
        }
    }
    int v = hits;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((tid & 31) == 0) s_sum[tid >> 5] = v;
    __syncthreads();
    if (tid == 0) {
        int total = 0;
        for (int w = 0; w < kRecallThreads / 32; ++w) total += s_sum[w];
        p.recall[head] = (nb == 0) ? 1.f : (float)total / (float)nb;
    }
}

template <int D, typename KT>
cudaError_t launch_scores_t(const ExactParams& p, cudaStream_t st) {
    const dim3 grid((unsigned)((p.n_cap + kScoreRowsPerCta - 1) / kScoreRowsPerCta), (unsigned)(p.B * p.Hkv));
    const size_t smem = (size_t)p.G * D * sizeof(float);
    if (p.G == 4) k_dot_scores<D, KT, 4><<<grid, 256, smem, st>>>(p);
    else k_dot_scores<D, KT, 0><<<grid, 256, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_exact_scores(const ExactParams& p, int d, int kv_bf16, cudaStream_t st) {
    bool tc = false;
    cudaError_t e = kv_bf16 ? launch_scores_tc(p, d, st, &tc) : cudaSuccess;
    if (e != cudaSuccess || tc) return e;
    e = cudaErrorInvalidValue;
    if (d == 128 && kv_bf16) e = launch_scores_t<128, __nv_bfloat16>(p, st);
    if (d == 64 && kv_bf16) e = launch_scores_t<64, __nv_bfloat16>(p, st);
    if (d == 128 && !kv_bf16) e = launch_scores_t<128, float>(p, st);
    if (d == 64 && !kv_bf16) e = launch_scores_t<64, float>(p, st);
    return e;
}

cudaError_t launch_exact_topm(const ExactParams& p, cudaStream_t st) {
    cudaError_t e;
    ExactParams q = p;
    q.bitmap_words = p.n_cap <= kBitmapTokens ? (p.n_cap + 31) / 32 : 0;
    const size_t smem = (size_t)(2 * kCandCap + q.bitmap_words + kTieCap) * sizeof(uint32_t);
    e = cudaFuncSetAttribute(k_topk_exact, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_topk_exact<<<p.B * p.Hq, kTopkThreads, smem, st>>>(q);
    return cudaGetLastError();
}

cudaError_t launch_recall(const RecallParams& p, cudaStream_t st) {
    if (p.heads <= 0) return cudaSuccess;
    k_recall<<<p.heads, kRecallThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ha
