// SCORE and TOPK as one kernel: a thread-block cluster per (batch entry, KV head).
//
// HashAttention: Semantic Sparsity for Faster Inference, Eq. (2): a cached
// token's score is the negated Hamming distance between its 32-bit key code and
// the query code; Sec. 4 keeps the min(m, n) best tokens (ties to the smaller
// index), Sec. 4.4 adds the first n_sink and the last n_local tokens. One read
// of a KV head's codes serves all its query heads (Nectar Sec. 3, GQA sharing).
//
// Decomposition. The CL CTAs of a cluster split the n tokens of one (batch
// entry b, KV head g) into contiguous ranges of R = 8192 LB tokens (rank r owns
// [r R, min(n, (r + 1) R))); R is chosen so that the whole grid is resident at
// once where it can be (every SM streams codes at the same time instead of in
// waves that finish together).
//   phase 1  every code of the range is read once (16-byte streaming loads, 512
//            contiguous bytes per warp instruction, four rounds in flight per
//            thread); per token the distances to the (up to four) query heads
//            are computed once, written as one packed word (head e in byte e) to
//            a buffer in token order that stays in L2, and counted into a 33-bin
//            histogram per head (shared-memory columns indexed by lane).
//   meta     after a cluster barrier every CTA reads the cluster's histograms
//            through distributed shared memory and derives, per head, the
//            threshold bin t (smallest t whose cumulative count reaches k), the
//            number of tied tokens (distance t) still to take, how many of those
//            fall to each CTA (none, all, or the first q in token order: at most
//            one CTA per head takes part of its ties) and so how many tokens each
//            CTA selects, which fixes this CTA's first output position.
//   masks    warp w owns 1024 LB consecutive tokens of the range and each lane LB
//            consecutive 32-token blocks, one 128-byte line of packed distances
//            each; a lane builds its selection masks for all heads at once with
//            byte-wise compares (no further popcounts); windows and the sequence
//            end enter as bit ranges; in the boundary CTA the tied tokens are
//            ranked across warps and lanes.
//   output   the lane writes its tokens straight into one flat ascending list per
//            query head and drops each distance line from L2 without writing it
//            back; rank 0 writes the count (and, when asked, pads the list with -1).
#include <cooperative_groups.h>

#include "ha_internal.cuh"

namespace cg = cooperative_groups;

namespace ha {
namespace {


__device__ __forceinline__ uint32_t warp_sum_u(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_excl_scan(int v, int* total) {
    const int lane = threadIdx.x & 31;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

__device__ __forceinline__ void red_add_shared(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t half_field(uint32_t w01, uint32_t w23, int e) {
    const uint32_t w = (e < 2) ? w01 : w23;
    return (e & 1) ? (w >> 16) : (w & 0xffffu);
}

constexpr int kBlockWords = 36;  // shared words per 32-token block of packed distances

// Bits [0, k) set, k clamped to [0, 32].
__device__ __forceinline__ uint32_t low_bits(int k) {
    return k <= 0 ? 0u : (k >= 32 ? 0xffffffffu : ((1u << k) - 1u));
}

// Per-head masks over a lane block of 32 tokens: bit j of m[e] is set iff byte e
// of D[j] is at most byte e of the threshold word, where TE holds 0x80 + T_e in
// byte e (T_e in [-1, 32]; distances are at most 32, so no byte borrows from its
// neighbour and bit 7 of byte e of TE - D[j] is set exactly when D_e <= T_e).
__device__ __forceinline__ void le_masks(const uint32_t (&D)[32], uint32_t TE, uint32_t (&m)[4]) {
    uint32_t X[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t x = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) x |= ((TE - D[8 * q + j]) & 0x80808080u) >> (7 - j);
        X[q] = x;  // byte e: tokens 8q .. 8q+7 of head e
    }
    // 4 x 4 byte transpose: byte q of m[e] = byte e of X[q]
    const uint32_t a = __byte_perm(X[0], X[1], 0x5140);
    const uint32_t c = __byte_perm(X[0], X[1], 0x7362);
    const uint32_t bb = __byte_perm(X[2], X[3], 0x5140);
    const uint32_t dd = __byte_perm(X[2], X[3], 0x7362);
    m[0] = __byte_perm(a, bb, 0x5410);
    m[1] = __byte_perm(a, bb, 0x7632);
    m[2] = __byte_perm(c, dd, 0x5410);
    m[3] = __byte_perm(c, dd, 0x7632);
}

// Threshold word: byte e = 0x80 + T_e for heads e < nh, 0x7F (select nothing) above.
__device__ __forceinline__ uint32_t thresh_word(const int (&T)[4], int nh) {
    uint32_t w = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) w |= (uint32_t)((e < nh) ? (0x80 + T[e]) : 0x7F) << (8 * e);
    return w;
}

// Keep the first q set bits of x (q >= 0).
__device__ __forceinline__ uint32_t first_bits(uint32_t x, int q) {
    uint32_t keep = 0u;
    while (x != 0u && q > 0) {
        const uint32_t low = x & (0u - x);
        keep |= low;
        x ^= low;
        --q;
    }
    return keep;
}

// A CTA of NT threads covers R = 32 NT LB tokens of one (batch entry, KV head):
// warp w owns [w 1024 LB, (w + 1) 1024 LB) of the range and lane l of it the LB
// consecutive 32-token blocks from w 1024 LB + 32 LB l. The packed distances of
// the range stay in shared memory, 36 words per 32-token block (the 4 spare words
// keep both the phase-1 stores and the per-lane block reads free of bank conflicts).
template <int NT, int LB>
__global__ void __launch_bounds__(NT, (NT >= 1024 || LB > 1) ? 1 : 1024 / NT) k_select_cl(const ClSelectParams p) {
    constexpr int NW = NT / 32;
    constexpr int R = 32 * NT * LB;
    constexpr int NR = R / (4 * NT);   // phase-1 rounds of 4 tokens per thread
    constexpr int U = 4;               // rounds of codes in flight per thread
    extern __shared__ __align__(16) uint32_t sD[];  // [R / 32][kBlockWords]
    __shared__ uint32_t hist[HA_NBINS][2][32];      // lane columns; heads 2k, 2k+1 in 16-bit fields
    // Per head, the histogram of this CTA's tokens and of the two window parts of
    // its range (the sink part is a prefix of the range, the local part a suffix)
    __shared__ uint32_t s_hc[4][HA_NBINS + 3];
    __shared__ uint32_t s_hp[4][HA_NBINS + 3];
    __shared__ uint32_t s_hs[4][HA_NBINS + 3];
    // Read by the whole cluster: the same three as exclusive prefix sums,
    // c[u] = tokens at distances below u, u = 0 .. 33 (c[33] = all of them)
    __shared__ uint32_t s_ca[4][HA_NBINS + 3];
    __shared__ uint32_t s_cp[4][HA_NBINS + 3];
    __shared__ uint32_t s_cs[4][HA_NBINS + 3];
    __shared__ int s_wt[4][NW];                     // ties per warp (the head's boundary CTA)
    __shared__ int s_wc[4][NW];                     // selected tokens per warp
    __shared__ int s_t[4], s_mode[4], s_q[4], s_base[4], s_all[4], s_cnt[4];

    cg::cluster_group cluster = cg::this_cluster();
    const int CL = p.CL;
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pair = blockIdx.x / CL;
    const int b = pair / p.Hkv, g = pair % p.Hkv;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, rank == 0 && g == 0 && tid == 0);
    const int lo = min(n, rank * R);
    const int hi = min(n, lo + R);
    const int head0 = b * p.Hq + g * p.G;
    const int nh = p.G;  // at most 4 (checked on the host)
    const int wlo = min(p.n_sink, n);                   // sink window [0, wlo)
    const int wmid = max(max(0, n - p.n_local), wlo);   // local window [wmid, n)

    uint32_t qs[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) qs[e] = (e < nh) ? p.q_sig[head0 + e] : 0u;
    for (int x = tid; x < HA_NBINS * 2 * 32; x += NT) (&hist[0][0][0])[x] = 0u;
    for (int x = tid; x < 4 * (HA_NBINS + 3); x += NT) {
        (&s_hp[0][0])[x] = 0u;
        (&s_hs[0][0])[x] = 0u;
    }
    pdl_launch_dependents();
    __syncthreads();

    // ---------------------------------------------------------------- phase 1
    {
        const uint32_t* row = p.k_sig + (int64_t)b * p.ks_sb + (int64_t)g * p.ks_sh;
        const uint32_t col = smem_addr(&hist[0][0][lane]);
        uint4 v[U];
        auto load = [&](int k) {
            const int i = lo + k * 4 * NT + 4 * tid;
            uint4 c;
            if (i + 4 <= hi) {
                c = __ldg(reinterpret_cast<const uint4*>(row + i));
            } else {
                c.x = (i < hi) ? __ldg(row + i) : 0u;
                c.y = (i + 1 < hi) ? __ldg(row + i + 1) : 0u;
                c.z = (i + 2 < hi) ? __ldg(row + i + 2) : 0u;
                c.w = (i + 3 < hi) ? __ldg(row + i + 3) : 0u;
            }
            return c;
        };
        auto compute = [&](const uint4 c4, int k) {
            const int i = lo + k * 4 * NT + 4 * tid;
            if (i >= hi) return;
            const uint32_t code[4] = {c4.x, c4.y, c4.z, c4.w};
            uint32_t pk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t w = 0u;
                if (i + j < hi) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (e < nh) {
                            const uint32_t d = (uint32_t)__popc(qs[e] ^ code[j]);
                            red_add_shared(col + (d * 2 + (e >> 1)) * 128u, 1u << (16 * (e & 1)));
                            w |= d << (8 * e);
                        }
                    }
                }
                pk[j] = w;
            }
            const int o = i - lo;  // 4-aligned: the four words stay in one block
            *reinterpret_cast<uint4*>(sD + (o >> 5) * kBlockWords + (o & 31)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        };
#pragma unroll
        for (int k = 0; k < NR + U; ++k) {
            if (k >= U) compute(v[(k - U) % U], k - U);
            if (k < NR) v[k % U] = load(k);
        }
    }
    __syncthreads();  // the range's distances are in shared memory
    // lane columns -> this CTA's histogram
    for (int u = warp; u < HA_NBINS; u += NW) {
        const uint32_t s01 = warp_sum_u(hist[u][0][lane]);
        const uint32_t s23 = warp_sum_u(hist[u][1][lane]);
        if (lane < 4) s_hc[lane][u] = (lane < nh) ? half_field(s01, s23, lane) : 0u;
    }
    {
        // histograms of the window parts of this range: [lo, min(hi, wlo)) and [max(lo, wmid), hi)
        const int a0 = lo, a1 = min(hi, wlo), b0 = max(lo, wmid), b1 = hi;
        const int na = max(0, a1 - a0), nb = max(0, b1 - b0);
        for (int x = tid; x < na + nb; x += NT) {
            const int o = (x < na ? a0 + x : b0 + (x - na)) - lo;
            const uint32_t w = sD[(o >> 5) * kBlockWords + (o & 31)];
            uint32_t(*hw)[HA_NBINS + 3] = (x < na) ? s_hp : s_hs;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nh) atomicAdd(&hw[e][(w >> (8 * e)) & 0xffu], 1u);
        }
    }
    __syncthreads();
    // exclusive prefix sums over the 33 bins, one warp per (head, histogram)
    for (int job = warp; job < 3 * nh; job += NW) {
        const int e = job % nh, which = job / nh;
        const uint32_t* hsrc = (which == 0) ? s_hc[e] : (which == 1 ? s_hp[e] : s_hs[e]);
        uint32_t* cdst = (which == 0) ? s_ca[e] : (which == 1 ? s_cp[e] : s_cs[e]);
        const uint32_t v = hsrc[lane];
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        cdst[lane] = x - v;
        if (lane == 31) {
            cdst[32] = x;
            cdst[33] = x + hsrc[32];
        }
    }
    cluster.sync();  // every CTA's prefix sums are complete and visible to the cluster

    // ---------------------------------------------------------------- meta
    // Per head: the threshold bin t and the ties still to take over the whole
    // sequence, then for every rank r in order its share of those ties and the
    // number of tokens it selects, which gives this CTA's first output position.
    //   A = tokens of the range below t, T = its ties, P / S = the sink / local
    //   window parts of the range (below t: Pl / Sl, at t: Pt / St), q' = the
    //   rank's taken ties (the first ones of the range in token order):
    //   selected = A + (|P| - Pl) + (|S| - Sl) + q' - |taken in P| - |taken in S|,
    //   |taken in P| = min(q', Pt) (P is a prefix), |taken in S| = max(0, q' - (T - St))
    //   (S is a suffix); with exclusive windows no window token is a tie:
    //   selected = (A - Pl - Sl) + q' + |P| + |S|, with T counting non-window ties.
    if (warp < nh) {
        const int e = warp;
        const int64_t h = head0 + e;
        int mb = p.m;
        if (p.m_per_seq != nullptr) {
            mb = p.m_per_seq[b];
            if (mb < 0 || mb > p.m) {
                if (rank == 0 && g == 0 && e == 0 && lane == 0) flag_error(p.err, HA_DEVERR_BUDGET);
                mb = min(max(mb, 0), p.m);
            }
        }
        if (p.m_per_head != nullptr) {
            mb = p.m_per_head[h];
            if (mb < 0 || mb > p.m) {
                if (rank == 0 && lane == 0) flag_error(p.err, HA_DEVERR_BUDGET);
                mb = min(max(mb, 0), p.m);
            }
        }
        const int nwin = wlo + (n - wmid);
        const int k = p.excl ? min(mb, n - nwin) : min(mb, n);
        // bin `lane` summed over the cluster, every load in flight together (bin 32
        // is implied by the total)
        uint32_t tot = 0u;
#pragma unroll
        for (int r = 0; r < kClMax; ++r) {
            if (r < CL) {
                const uint32_t* ca = cluster.map_shared_rank(&s_ca[e][0], r);
                tot += ca[lane + 1] - ca[lane];
                if (p.excl) {
                    const uint32_t* cp = cluster.map_shared_rank(&s_cp[e][0], r);
                    const uint32_t* cs = cluster.map_shared_rank(&s_cs[e][0], r);
                    tot -= (cp[lane + 1] - cp[lane]) + (cs[lane + 1] - cs[lane]);
                }
            }
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
        const int rq = k - (t == 0 ? 0 : (int)below);  // ties to take over the whole sequence, in token order
        // lane r: rank r's counts at t, its share of the ties and its selected tokens
        int A = 0, T = 0, Pl = 0, Pt = 0, NP = 0, Sl = 0, St = 0, NS = 0;
        if (lane < CL) {
            const uint32_t* ca = cluster.map_shared_rank(&s_ca[e][0], lane);
            const uint32_t* cp = cluster.map_shared_rank(&s_cp[e][0], lane);
            const uint32_t* cs = cluster.map_shared_rank(&s_cs[e][0], lane);
            A = (int)ca[t];
            T = (int)ca[t + 1] - A;
            Pl = (int)cp[t];
            Pt = (int)cp[t + 1] - Pl;
            NP = (int)cp[HA_NBINS];
            Sl = (int)cs[t];
            St = (int)cs[t + 1] - Sl;
            NS = (int)cs[HA_NBINS];
        }
        if (p.excl) T -= Pt + St;
        int tsum;
        const int qr = min(max(rq - warp_excl_scan(T, &tsum), 0), T);
        int c = 0;
        if (lane < CL) {
            c = p.excl ? (A - Pl - Sl) + qr + NP + NS
                       : A + (NP - Pl) + (NS - Sl) + qr - min(qr, Pt) - max(0, qr - (T - St));
        }
        int all;
        const int base = warp_excl_scan(c, &all);
        const int my_q = __shfl_sync(0xffffffffu, qr, rank & 31);
        const int my_T = __shfl_sync(0xffffffffu, T, rank & 31);
        const int my_base = __shfl_sync(0xffffffffu, base, rank & 31);
        const int my_cnt = __shfl_sync(0xffffffffu, c, rank & 31);
        if (lane == 0) {
            s_t[e] = t;
            s_q[e] = my_q;
            s_mode[e] = (my_q <= 0) ? 0 : (my_q >= my_T ? 1 : 2);
            s_base[e] = my_base;
            s_all[e] = all;
            s_cnt[e] = my_cnt;
        }
    }
    cluster.barrier_arrive();  // this CTA reads no other CTA's shared memory after this point
    __syncthreads();

    // ---------------------------------------------------------------- selection masks
    int mode[4], T[4], Tm1[4];
    bool any2 = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        T[e] = (e < nh) ? s_t[e] : 0;
        Tm1[e] = T[e] - 1;
        mode[e] = (e < nh) ? s_mode[e] : 0;
        any2 = any2 || mode[e] == 2;
    }
    const uint32_t TLT = thresh_word(Tm1, nh), TLE = thresh_word(T, nh);
    const int lane0 = lo + warp * 1024 * LB + lane * 32 * LB;  // this lane's first token
    // masks of block k of this lane: lt (distance < t), le (distance <= t), the
    // windows and the valid tokens; false when the block lies past the sequence
    auto block = [&](int k, uint32_t (&lt)[4], uint32_t (&le)[4], uint32_t& win, uint32_t& valid) {
        const int lb = lane0 + 32 * k;
        valid = low_bits(n - lb);
        win = low_bits(wlo - lb) | ~low_bits(wmid - lb);
        if (valid == 0u) return false;
        uint32_t D[32];
        const uint4* src = reinterpret_cast<const uint4*>(sD + ((lb - lo) >> 5) * kBlockWords);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = src[j];
            D[4 * j + 0] = v.x;
            D[4 * j + 1] = v.y;
            D[4 * j + 2] = v.z;
            D[4 * j + 3] = v.w;
        }
        le_masks(D, TLT, lt);
        le_masks(D, TLE, le);
        return true;
    };
    // tied tokens (distance t) of a block that may be taken
    auto ties = [&](int e, const uint32_t (&lt)[4], const uint32_t (&le)[4], uint32_t win, uint32_t valid) {
        uint32_t eq = le[e] & ~lt[e] & valid;
        if (p.excl) eq &= ~win;
        return eq;
    };
    int qrem[4] = {0, 0, 0, 0};  // ties this lane still takes (the head's boundary CTA)
    if (any2) {
        int tl[4] = {0, 0, 0, 0};
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            uint32_t lt[4], le[4], win, valid;
            if (!block(k, lt, le, win, valid)) continue;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (mode[e] == 2) tl[e] += __popc(ties(e, lt, le, win, valid));
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (mode[e] == 2) {
                int tot;
                qrem[e] = -warp_excl_scan(tl[e], &tot);
                if (lane == 0) s_wt[e][warp] = tot;
            }
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (mode[e] == 2) {
                int qw = s_q[e];
                for (int w2 = 0; w2 < warp; ++w2) qw -= s_wt[e][w2];
                qrem[e] += qw;
            }
        }
    }
    // the final mask of head e for a block, taking this lane's ties in token order
    auto final_mask = [&](int e, const uint32_t (&lt)[4], const uint32_t (&le)[4], uint32_t win, uint32_t valid,
                          int (&q)[4]) {
        uint32_t m = (mode[e] == 1) ? le[e] : lt[e];
        if (mode[e] == 2) {
            const uint32_t take = first_bits(ties(e, lt, le, win, valid), q[e]);
            q[e] -= __popc(take);
            m |= take;
        }
        return (m | win) & valid;
    };
    // final masks of the lane's blocks, kept for the output
    uint32_t keep[LB][4];
    int cnt[4] = {0, 0, 0, 0};
    {
        int q[4] = {qrem[0], qrem[1], qrem[2], qrem[3]};
#pragma unroll
        for (int k = 0; k < LB; ++k) {
            uint32_t lt[4], le[4], win, valid;
            const bool any = block(k, lt, le, win, valid);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                keep[k][e] = (any && e < nh) ? final_mask(e, lt, le, win, valid, q) : 0u;
                cnt[e] += __popc(keep[k][e]);
            }
        }
    }
    int pos[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int tot;
        pos[e] = warp_excl_scan(cnt[e], &tot);
        if (lane == 0) s_wc[e][warp] = tot;
    }
    __syncthreads();
    if (tid < nh) {
        int mine = 0;
        for (int w2 = 0; w2 < NW; ++w2) mine += s_wc[tid][w2];
        if (mine != s_cnt[tid]) flag_error(p.err, HA_DEVERR_STATE);  // the masks disagree with the counts
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        pos[e] += s_base[e];
        for (int w2 = 0; w2 < warp; ++w2) pos[e] += s_wc[e][w2];
    }

    // ---------------------------------------------------------------- output
    const int cap = p.cap;
#pragma unroll
    for (int k = 0; k < LB; ++k) {
        const int lb = lane0 + 32 * k;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (e < nh) {
                uint32_t m = keep[k][e];
                int32_t* dst = p.list + (int64_t)(head0 + e) * cap;
                const int at = pos[e];
                pos[e] += __popc(m);
                if (at + __popc(m) > cap) {
                    flag_error(p.err, HA_DEVERR_STATE);
                    m = 0u;
                }
                if (__popc(m) >= 8) {
                    // dense (window) blocks: independent stores instead of a serial bit walk
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if ((m >> j) & 1u) dst[at + __popc(m & ((1u << j) - 1u))] = lb + j;
                } else {
                    int a = at;
                    while (m != 0u) {
                        const int j = __ffs(m) - 1;
                        m &= m - 1u;
                        dst[a++] = lb + j;
                    }
                }
            }
        }
    }
    if (rank == 0) {
        for (int e = 0; e < nh; ++e) {
            const int all = s_all[e];
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
    cluster.barrier_wait();  // no CTA leaves while another may still read its shared memory
}

template <int NT, int LB>
cudaError_t launch_cl_t(const ClSelectParams& p, int batch_hkv, cudaStream_t st) {
    const size_t smem = cl_select_smem(32 * NT * LB);
    // function attributes belong to the current device's context: set them on every launch
    cudaError_t e = cudaFuncSetAttribute(k_select_cl<NT, LB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && p.CL > 8)
        e = cudaFuncSetAttribute(k_select_cl<NT, LB>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)batch_hkv * (unsigned)p.CL);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_select_cl<NT, LB>, p);
}

}  // namespace

size_t cl_select_smem(int rmax) { return (size_t)(rmax / 32) * kBlockWords * 4; }

cudaError_t launch_select_cl(const ClSelectParams& p, int batch_hkv, cudaStream_t st) {
    switch (p.rmax) {
        case 8192: return launch_cl_t<256, 1>(p, batch_hkv, st);
        case 16384: return launch_cl_t<512, 1>(p, batch_hkv, st);
        case 32768: return launch_cl_t<512, 2>(p, batch_hkv, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ha
