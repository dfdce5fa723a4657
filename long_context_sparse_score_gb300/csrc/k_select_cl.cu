// SCORE and TOPK as one kernel: a thread-block cluster per (batch entry, KV head).
//
// HashAttention: Semantic Sparsity for Faster Inference, Eq. (2): a cached
// token's score is the negated Hamming distance between its 32-bit key code and
// the query code; Sec. 4 keeps the min(m, n) best tokens (ties to the smaller
// index), Sec. 4.4 adds the first n_sink and the last n_local tokens. One read
// of a KV head's codes serves all its query heads (Nectar Sec. 3, GQA sharing).
//
// Decomposition. The CL CTAs of a cluster split the n tokens of one (batch
// entry b, KV head g) into contiguous ranges of R = 32 NT tokens (NT threads per
// CTA; rank r owns [r R, min(n, (r + 1) R))). A CTA keeps its intermediates on
// chip:
//   phase 1  every code of the range is read once (16-byte loads, 512 contiguous
//            bytes per warp instruction, four rounds in flight per thread); per
//            token the distances to the (up to four) query heads are computed
//            once, kept as one packed word (head e in byte e) in shared memory
//            and counted into a 33-bin histogram per head (shared-memory columns
//            indexed by lane).
//   meta     after a cluster barrier every CTA reads the cluster's histograms
//            through distributed shared memory and derives, per head, the
//            threshold bin t (smallest t whose cumulative count reaches k), the
//            number of tied tokens (distance t) still to take, and how many of
//            those fall to this CTA: none (mode 0), all (mode 1) or the first q
//            in token order (mode 2, one CTA per head at most).
//   masks    warp w owns tokens [w 1024, (w + 1) 1024) of the range and lane l
//            of it the 32 tokens of block 32 w + l; the lane builds its
//            selection mask for all heads at once with byte-wise compares of the
//            packed distances (no further popcounts); windows and the sequence
//            end enter as bit ranges; in the boundary CTA the tied tokens are
//            ranked across warps and lanes.
//   output   after a second cluster barrier each CTA knows the selected count
//            of the ranks before it, so it writes its tokens straight into one
//            flat ascending list per query head; rank 0 writes the count (and,
//            when asked, pads the list with -1).
#include <cooperative_groups.h>

#include "ha_internal.cuh"

namespace cg = cooperative_groups;

namespace ha {
namespace {

constexpr int kPadWords = 36;            // shared pitch of a 32-token lane block (32 words + 4 pad)

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

// The 32 packed distance words of this lane's block (the warp's blocks are 32 w .. 32 w + 31).
__device__ __forceinline__ void load_block(const uint32_t* sD, int warp, uint32_t (&D)[32]) {
    const int lane = threadIdx.x & 31;
    const uint4* src = reinterpret_cast<const uint4*>(sD + (warp * 32 + lane) * kPadWords);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = src[j];
        D[4 * j + 0] = v.x;
        D[4 * j + 1] = v.y;
        D[4 * j + 2] = v.z;
        D[4 * j + 3] = v.w;
    }
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

// NT threads per CTA; a CTA covers R = 32 NT tokens: warp w owns the 1024
// consecutive tokens [w 1024, (w + 1) 1024) of the range and lane l of it the 32
// tokens of block 32 w + l.
template <int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) k_select_cl(const ClSelectParams p) {
    constexpr int NW = NT / 32;
    constexpr int R = 32 * NT;
    constexpr int NR = R / (4 * NT);   // phase-1 rounds of 4 tokens per thread
    constexpr int U = 4;               // rounds of codes in flight per thread
    extern __shared__ __align__(16) uint32_t sD[];  // [R / 32][kPadWords] packed distances
    __shared__ uint32_t hist[HA_NBINS][2][32];      // lane columns; heads 2k, 2k+1 in 16-bit fields
    // Read by the whole cluster: per head, the histogram of this CTA's tokens and
    // of the two window parts of its range (the sink part is a prefix of the
    // range, the local part a suffix); entry 33 of a window histogram holds its
    // token count.
    __shared__ uint32_t s_hc[4][HA_NBINS + 3];
    __shared__ uint32_t s_hp[4][HA_NBINS + 3];
    __shared__ uint32_t s_hs[4][HA_NBINS + 3];
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
            const int o = k * 4 * NT + 4 * tid;  // offset in the range
            const int i = lo + o;
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
            *reinterpret_cast<uint4*>(sD + (o >> 5) * kPadWords + (o & 31)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        };
#pragma unroll
        for (int k = 0; k < NR + U; ++k) {
            if (k >= U) compute(v[(k - U) % U], k - U);
            if (k < NR) v[k % U] = load(k);
        }
    }
    __syncthreads();
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
            const uint32_t w = sD[(o >> 5) * kPadWords + (o & 31)];
            uint32_t(*hw)[HA_NBINS + 3] = (x < na) ? s_hp : s_hs;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nh) atomicAdd(&hw[e][(w >> (8 * e)) & 0xffu], 1u);
        }
        if (tid < nh) {
            s_hp[tid][HA_NBINS] = (uint32_t)na;
            s_hs[tid][HA_NBINS] = (uint32_t)nb;
        }
    }
    cluster.sync();  // every CTA's histograms are complete and visible to the cluster

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
        // bin `lane` of every rank, all loads in flight together (bin 32 is implied by the total)
        uint32_t hr[kClMax], np[kClMax], ns[kClMax];
#pragma unroll
        for (int r = 0; r < kClMax; ++r) {
            hr[r] = np[r] = ns[r] = 0u;
            if (r < CL) {
                hr[r] = cluster.map_shared_rank(&s_hc[e][0], r)[lane];
                np[r] = cluster.map_shared_rank(&s_hp[e][0], r)[HA_NBINS];
                ns[r] = cluster.map_shared_rank(&s_hs[e][0], r)[HA_NBINS];
            }
        }
        uint32_t tot = 0u;
        if (p.excl) {
#pragma unroll
            for (int r = 0; r < kClMax; ++r) {
                if (r < CL && np[r] + ns[r] != 0u)
                    tot -= cluster.map_shared_rank(&s_hp[e][0], r)[lane] + cluster.map_shared_rank(&s_hs[e][0], r)[lane];
            }
        }
#pragma unroll
        for (int r = 0; r < kClMax; ++r) tot += hr[r];
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
        int base = 0, all = 0, my_q = 0, my_T = 0, my_cnt = 0;
#pragma unroll
        for (int r = 0; r < kClMax; ++r) {
            if (r < CL) {
                const uint32_t* hc = cluster.map_shared_rank(&s_hc[e][0], r);
                const int A = (int)warp_sum_u(lane < t ? hr[r] : 0u);
                int T = (t < 32) ? (int)__shfl_sync(0xffffffffu, hr[r], t) : (int)hc[32];
                int Pl = 0, Pt = 0, Sl = 0, St = 0;
                if (np[r] + ns[r] != 0u) {
                    const uint32_t* hp = cluster.map_shared_rank(&s_hp[e][0], r);
                    const uint32_t* hs = cluster.map_shared_rank(&s_hs[e][0], r);
                    const uint32_t pv = hp[lane], sv = hs[lane];
                    Pl = (int)warp_sum_u(lane < t ? pv : 0u);
                    Sl = (int)warp_sum_u(lane < t ? sv : 0u);
                    Pt = (t < 32) ? (int)__shfl_sync(0xffffffffu, pv, t) : (int)hp[32];
                    St = (t < 32) ? (int)__shfl_sync(0xffffffffu, sv, t) : (int)hs[32];
                }
                if (p.excl) T -= Pt + St;
                const int qr = min(max(left, 0), T);
                left -= T;
                int c;
                if (p.excl) {
                    c = (A - Pl - Sl) + qr + (int)np[r] + (int)ns[r];
                } else {
                    c = A + ((int)np[r] - Pl) + ((int)ns[r] - Sl) + qr - min(qr, Pt) - max(0, qr - (T - St));
                }
                if (r < rank) base += c;
                if (r == rank) {
                    my_q = qr;
                    my_T = T;
                    my_cnt = c;
                }
                all += c;
            }
        }
        if (lane == 0) {
            s_t[e] = t;
            s_q[e] = my_q;
            s_mode[e] = (my_q <= 0) ? 0 : (my_q >= my_T ? 1 : 2);
            s_base[e] = base;
            s_all[e] = all;
            s_cnt[e] = my_cnt;
        }
    }
    cluster.barrier_arrive();  // this CTA reads no other CTA's shared memory after this point
    __syncthreads();

    // ---------------------------------------------------------------- selection masks
    int mode[4];
    bool any2 = false;
    int Tm1[4], T[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        T[e] = (e < nh) ? s_t[e] : 0;
        Tm1[e] = T[e] - 1;
        mode[e] = (e < nh) ? s_mode[e] : 0;
        any2 = any2 || mode[e] == 2;
    }
    const int lbase = lo + (warp * 32 + lane) * 32;  // this lane's 32 tokens
    const uint32_t win = low_bits(wlo - lbase) | ~low_bits(wmid - lbase);
    const uint32_t valid = low_bits(n - lbase);
    uint32_t msk[4];
    {
        uint32_t D[32];
        load_block(sD, warp, D);
        uint32_t lt[4], le[4];
        le_masks(D, thresh_word(Tm1, nh), lt);
        le_masks(D, thresh_word(T, nh), le);
#pragma unroll
        for (int e = 0; e < 4; ++e) msk[e] = (mode[e] == 1) ? le[e] : lt[e];
        if (any2) {
            // the boundary CTA of a head: its tied tokens, ranked in token order
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
                    int qw = s_q[e];
                    for (int w2 = 0; w2 < warp; ++w2) qw -= s_wt[e][w2];
                    int tot;
                    const int ex = warp_excl_scan(__popc(eq[e]), &tot);
                    msk[e] |= first_bits(eq[e], qw - ex);
                }
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
    if (tid < nh) {
        int mine = 0;
        for (int w2 = 0; w2 < NW; ++w2) mine += s_wc[tid][w2];
        if (mine != s_cnt[tid]) flag_error(p.err, HA_DEVERR_STATE);  // the masks disagree with the counts
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
        for (int w2 = 0; w2 < warp; ++w2) pos[e] += s_wc[e][w2];

    // ---------------------------------------------------------------- output
    const int cap = p.cap;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (e < nh) {
            uint32_t m = msk[e];
            int at = s_base[e] + pos[e];
            int32_t* dst = p.list + (int64_t)(head0 + e) * cap;
            if (at + __popc(m) > cap) {
                flag_error(p.err, HA_DEVERR_STATE);
                m = 0u;
            }
            if (__popc(m) >= 8) {
                // dense (window) lanes: independent stores instead of a serial bit walk
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if ((m >> j) & 1u) dst[at + __popc(m & ((1u << j) - 1u))] = lbase + j;
            } else {
                while (m != 0u) {
                    const int j = __ffs(m) - 1;
                    m &= m - 1u;
                    dst[at++] = lbase + j;
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

}  // namespace

size_t cl_select_smem(int rmax) { return (size_t)(rmax / 32) * kPadWords * 4; }

template <int NT>
cudaError_t launch_cl_t(const ClSelectParams& p, int batch_hkv, cudaStream_t st) {
    const size_t smem = cl_select_smem(32 * NT);
    static int s_smem_set = 0;
    if ((int)smem > s_smem_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(k_select_cl<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        s_smem_set = (int)smem;
    }
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
    return cudaLaunchKernelEx(&cfg, k_select_cl<NT>, p);
}

cudaError_t launch_select_cl(const ClSelectParams& p, int batch_hkv, cudaStream_t st) {
    switch (p.rmax) {
        case 32 * 256: return launch_cl_t<256>(p, batch_hkv, st);
        case 32 * 512: return launch_cl_t<512>(p, batch_hkv, st);
        case 32 * 1024: return launch_cl_t<1024>(p, batch_hkv, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ha
