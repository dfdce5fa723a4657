// GATHER-ATT and merge kernels of the sparse-decode path.
//
// HashAttention: Semantic Sparsity for Faster Inference, Sec. 4: attention over
// the selected set I only, o = sum_{i in I} e^{z_i} v_i / sum_{j in I} e^{z_j},
// z_i = <q, k_i>/sqrt(d); Sec. 4.4: paged attention with a page of one token, the
// selected indices used directly, no gathered copy of the KV rows.
// Nectar: Neural Estimation of Cached-Token Attention via Regression, Eq. (3.1)
// and Eqs. (3.4)-(3.5): the log-normaliser lse = log sum_j e^{z_j} is returned
// with o, and partial results over disjoint token sets merge exactly.
//
// k_gather_att: one CTA per (query head, split of I). The CTA first turns its
// range of list positions into token indices in shared memory. Then each warp
// runs its own pipeline over 8-row tiles (tiles w, w + W, w + 2W, ... of the
// CTA): it copies the K and V rows of a tile straight from the cache with
// 16-byte asynchronous copies (one warp instruction moves a 256-byte K row and
// its 256-byte V row) into a private ring of P shared-memory stages, keeping
// P - 1 tiles in flight while it computes the oldest one. Waits are on the
// warp's own copy groups only: no barrier couples warps until the final combine.
// In a tile, 4 lanes share a row: scores are fp32 (q pre-scaled by
// log2(e)/sqrt(d) and kept in shared memory, packed fp32x2 FMAs), the softmax is online in base 2 and P.V
// accumulates per lane over its rows. Splits write (max, sum, o) partials; the
// last CTA of a head to finish merges them (an arrival counter decides who is
// last; nothing waits).
#include "ha_internal.cuh"

#include <math_constants.h>

namespace ha {
namespace {

constexpr int kWarpsG = kGatherThreads / 32;

template <int D, typename KT>
struct Cfg {
    static constexpr int ES = sizeof(KT);
    static constexpr int RB = D * ES;                 // bytes of one K or V row
    static constexpr int PITCH = RB + 16;             // shared row pitch: rows land on distinct banks
    static constexpr int R = 8;                       // rows per warp tile
    static constexpr int P = 2;                       // stages per warp (more warps beat deeper rings)
    static constexpr int NCH = RB / 16;               // 16-byte chunks per row
    static constexpr int CPL = NCH / 4;               // chunks per lane (4 lanes per row)
    static constexpr int EPC = 16 / ES;               // elements per chunk
    static constexpr int DPL = CPL * EPC;             // dims per lane (= D / 4)
    static constexpr int STAGE_BYTES = 2 * R * PITCH; // K rows, then V rows
    static constexpr int WARP_BYTES = P * STAGE_BYTES;
    static constexpr int DATA_BYTES = kWarpsG * WARP_BYTES;
    static constexpr int OFF_CMB = DATA_BYTES;                            // float wm[W], wl[W], wo[W][D]
    static constexpr int OFF_TOKL = OFF_CMB + (2 * kWarpsG + kWarpsG * D) * 4;  // int tokl[rows_per_split]
};

template <typename KT>
__device__ __forceinline__ void chunk_to_float(const uint4 w, float* f);

template <>
__device__ __forceinline__ void chunk_to_float<__nv_bfloat16>(const uint4 w, float* f) {
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
    f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
    f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

template <>
__device__ __forceinline__ void chunk_to_float<float>(const uint4 w, float* f) {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
}

__device__ __forceinline__ float load_q(const void* q, int64_t off, int bf16) {
    if (bf16) {
        const uint16_t raw = reinterpret_cast<const uint16_t*>(q)[off];
        return __uint_as_float(((uint32_t)raw) << 16);
    }
    return reinterpret_cast<const float*>(q)[off];
}

// acc + q.lo * k.lo + q.hi * k.hi for two bf16 pairs: the products of bf16
// operands are exact in fp32 and each add rounds once, as in an fp32 FMA.
__device__ __forceinline__ float fma_bf16x2(uint32_t q2, uint32_t k2, float acc) {
    asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
        "mov.b32 {ql, qh}, %1;\n\t"
        "mov.b32 {kl, kh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ql, kl, %0;\n\t"
        "fma.rn.f32.bf16 %0, qh, kh, %0;\n\t}"
        : "+f"(acc)
        : "r"(q2), "r"(k2));
    return acc;
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Token of list position pp (kSegmented: the prefix table `pre` of the head's
// segments; kList: the caller's list, checked against [0, n)).
__device__ __forceinline__ int token_at(const GatherParams& p, int pp, int n, const int* pre, int nused,
                                        const int32_t* seg, const int32_t* lst) {
    if (p.mode == kIdentity) return pp;
    if (p.mode == kSegmented) {
        int lo = 0, hi = nused - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= pp) lo = mid; else hi = mid - 1;
        }
        // TOPK's own entries: outside [0, n) only if the workspace was disturbed
        const int tok = seg[(int64_t)lo * p.seg_cap + (pp - pre[lo])];
        if (tok < 0 || tok >= n) {
            flag_error(p.err, HA_DEVERR_STATE);
            return -1;
        }
        return tok;
    }
    const int tok = lst[pp];
    if (tok < 0 || tok >= n) {
        flag_error(p.err, HA_DEVERR_INDEX);
        return -1;
    }
    return tok;
}

// Five CTAs per SM for rows of up to 256 bytes (20 warps of copy pipelines);
// the 512-byte-row instantiation keeps three to avoid spills.
// QREG: bf16 query and bf16 K/V; each lane keeps the query elements of its
// dims as packed bf16 in registers and forms q.k with bf16 x bf16 -> fp32 FMAs
// straight from the K chunk (no query reads from shared memory, no K
// conversion); the score is scaled once per row.
template <int D, typename KT, bool QREG>
__global__ void __launch_bounds__(kGatherThreads, (D * sizeof(KT) <= 256) ? 5 : 3)
    k_gather_att(const GatherParams p) {
    using C = Cfg<D, KT>;
    extern __shared__ __align__(128) unsigned char smem[];
    float* wm = reinterpret_cast<float*>(smem + C::OFF_CMB);
    float* wl = wm + kWarpsG;
    float* wo = wl + kWarpsG;
    int* tokl = reinterpret_cast<int*>(smem + C::OFF_TOKL);
    int* pre = tokl + p.rows_per_split;   // [nseg + 1] (segmented lists only)
    __shared__ int s_L, s_last;
    __shared__ __align__(16) float s_q[D];   // q * log2(e) / sqrt(d), shared by the CTA's warps

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int lin = blockIdx.x;
    const int split = lin % p.splits;
    lin /= p.splits;
    const int hh = lin % p.G;
    lin /= p.G;
    const int b = lin % p.B;
    const int g = lin / p.B;
    const int head = b * p.Hq + g * p.G + hh;
    const bool report = (p.mode != kSegmented) && split == 0 && hh == 0 && g == 0 && tid == 0;
    const int n = checked_len(p.seq_lens, b, p.n_cap, p.err, report);
    const int nused = (p.mode == kSegmented) ? (n + p.seg_cap - 1) / p.seg_cap : 0;

    // ---- the query (an input: read before waiting for TOPK's output)
    const int r = lane & 7, qt = lane >> 3;
    constexpr int QW = QREG ? D / 8 : 1;   // packed bf16 pairs of this lane's D / 4 dims
    uint32_t qreg[QW];
    {
        const int64_t qoff = (int64_t)b * p.q_sb + (int64_t)(g * p.G + hh) * p.q_sh;
        if constexpr (QREG) {
            // chunk jc of the lane holds dims (jc * 4 + qt) * 8 .. + 7
            const uint16_t* qh16 = reinterpret_cast<const uint16_t*>(p.q) + qoff;
#pragma unroll
            for (int jc = 0; jc < QW / 4; ++jc)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int dim = (jc * 4 + qt) * 8 + 2 * u;
                    qreg[jc * 4 + u] = (uint32_t)qh16[dim] | ((uint32_t)qh16[dim + 1] << 16);
                }
        } else {
            for (int dd = tid; dd < D; dd += kGatherThreads) s_q[dd] = load_q(p.q, qoff + dd, p.q_bf16) * p.qscale;
        }
    }
    pdl_launch_dependents();
    pdl_wait();

    // ---- list length (and the segment prefix table), warp 0
    if (warp == 0) {
        int L = 0;
        if (p.mode == kIdentity) {
            L = n;
        } else if (p.mode == kList) {
            L = p.list_cnt[head];
            if (L < 0 || L > p.list_cap) {
                if (lane == 0) flag_error(p.err, HA_DEVERR_COUNT);
                L = min(max(L, 0), p.list_cap);
            }
        } else {
            const int32_t* cnt = p.seg_cnt + (int64_t)head * p.nseg;
            int carry = 0;
            if (lane == 0) pre[0] = 0;
            // counts in batches of 4 x 32 loads in flight, then the scans
            for (int base = 0; base < nused; base += 128) {
                int v4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int cc = base + 32 * k + lane;
                    v4[k] = (cc < nused) ? cnt[cc] : 0;
                    if (v4[k] < 0 || v4[k] > p.seg_cap) {  // a disturbed workspace: stay in the segment
                        flag_error(p.err, HA_DEVERR_STATE);
                        v4[k] = min(max(v4[k], 0), p.seg_cap);
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int cc = base + 32 * k + lane;
                    int v = v4[k];
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, v, o);
                        if (lane >= o) v += y;
                    }
                    if (cc < nused) pre[cc + 1] = carry + v;
                    carry += __shfl_sync(0xffffffffu, v, 31);
                }
            }
            L = carry;
        }
        if (lane == 0) s_L = L;
    }
    __syncthreads();

    const int L = s_L;
    const int r0 = split * p.rows_per_split;
    const int nrows = max(0, min(L, r0 + p.rows_per_split) - r0);

    // ---- this CTA's token indices (list positions [r0, r0 + nrows)) into shared memory
    {
        const int32_t* seg = (p.mode == kSegmented) ? p.seg_idx + (int64_t)head * p.nseg * p.seg_cap : nullptr;
        const int32_t* lst = (p.mode == kList) ? p.list_idx + (int64_t)head * p.list_cap : nullptr;
        constexpr int kB = 4;
        for (int i0 = 0; i0 < nrows; i0 += kB * kGatherThreads) {
            int tk[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int i = i0 + u * kGatherThreads + tid;
                tk[u] = (i < nrows) ? token_at(p, r0 + i, n, pre, nused, seg, lst) : -1;
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int i = i0 + u * kGatherThreads + tid;
                if (i < nrows) tokl[i] = tk[u];
            }
        }
    }
    __syncthreads();

    // ---- per-warp pipeline over 8-row tiles
    const int gk = kv_head(g, p.kv_mul);  // the KV head of this query-head group
    const char* Kb = p.K + ((int64_t)b * p.k_sb + (int64_t)gk * p.k_sh) * C::ES;
    const char* Vb = p.V + ((int64_t)b * p.v_sb + (int64_t)gk * p.v_sh) * C::ES;
    const int64_t kstep = p.k_sn * C::ES, vstep = p.v_sn * C::ES;
    unsigned char* wbuf = smem + warp * C::WARP_BYTES;
    const int ntiles = (nrows + C::R - 1) / C::R;
    const int ntw = (ntiles > warp) ? (ntiles - warp + kWarpsG - 1) / kWarpsG : 0;

    auto issue = [&](int k) {
        const int row0 = (warp + k * kWarpsG) * C::R;
        unsigned char* st = wbuf + (k % C::P) * C::STAGE_BYTES;
#pragma unroll
        for (int it = lane; it < C::R * 2 * C::NCH; it += 32) {
            const int row = it / (2 * C::NCH);
            const int rem = it - row * (2 * C::NCH);
            const int isv = rem >= C::NCH ? 1 : 0;
            const int ch = rem - isv * C::NCH;
            const int rr = row0 + row;
            if (rr < nrows) {
                const int tr = tokl[rr];
                if (tr >= 0) {
                    const char* src = (isv ? Vb + (int64_t)tr * vstep : Kb + (int64_t)tr * kstep) + ch * 16;
                    cp_async16(smem_addr(st + (isv * C::R + row) * C::PITCH + ch * 16), src);
                }
            }
        }
    };

    float2 ov[C::DPL / 2];
#pragma unroll
    for (int i = 0; i < C::DPL / 2; ++i) ov[i] = make_float2(0.f, 0.f);
    float mrun = -CUDART_INF_F, lrun = 0.f;

#pragma unroll
    for (int k = 0; k < C::P - 1; ++k) {
        if (k < ntw) issue(k);
        cp_async_commit();
    }
    for (int k = 0; k < ntw; ++k) {
        if (k + C::P - 1 < ntw) issue(k + C::P - 1);
        cp_async_commit();
        cp_async_wait<C::P - 1>();
        __syncwarp();
        const int rr = (warp + k * kWarpsG) * C::R + r;
        const int tok = (rr < nrows) ? tokl[rr] : -1;
        const unsigned char* kr = wbuf + (k % C::P) * C::STAGE_BYTES + r * C::PITCH;
        const unsigned char* vr = kr + C::R * C::PITCH;

        float part = 0.f;
        if (tok >= 0) {
            if constexpr (QREG) {
                float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int jc = 0; jc < C::CPL; ++jc) {
                    const uint4 w = *reinterpret_cast<const uint4*>(kr + (jc * 4 + qt) * 16);
                    a[0] = fma_bf16x2(qreg[jc * 4 + 0], w.x, a[0]);
                    a[1] = fma_bf16x2(qreg[jc * 4 + 1], w.y, a[1]);
                    a[2] = fma_bf16x2(qreg[jc * 4 + 2], w.z, a[2]);
                    a[3] = fma_bf16x2(qreg[jc * 4 + 3], w.w, a[3]);
                }
                part = (a[0] + a[1]) + (a[2] + a[3]);
            } else {
                float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int jc = 0; jc < C::CPL; ++jc) {
                    const uint4 w = *reinterpret_cast<const uint4*>(kr + (jc * 4 + qt) * 16);
                    float f[C::EPC];
                    chunk_to_float<KT>(w, f);
#pragma unroll
                    for (int e = 0; e < C::EPC; e += 4) {
                        const float4 q4 = *reinterpret_cast<const float4*>(s_q + (jc * 4 + qt) * C::EPC + e);
                        a0 = __ffma2_rn(make_float2(q4.x, q4.y), make_float2(f[e], f[e + 1]), a0);
                        a1 = __ffma2_rn(make_float2(q4.z, q4.w), make_float2(f[e + 2], f[e + 3]), a1);
                    }
                }
                part = (a0.x + a0.y) + (a1.x + a1.y);
            }
        }
        part += __shfl_xor_sync(0xffffffffu, part, 8);
        part += __shfl_xor_sync(0xffffffffu, part, 16);
        const float sc = (tok >= 0) ? (QREG ? part * p.qscale : part) : -CUDART_INF_F;
        float mx = sc;
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        const float mnew = fmaxf(mrun, mx);
        if (mnew != -CUDART_INF_F) {
            if (mnew > mrun) {
                const float alpha = exp2f(mrun - mnew);
                lrun *= alpha;
#pragma unroll
                for (int i = 0; i < C::DPL / 2; ++i) ov[i] = __fmul2_rn(ov[i], make_float2(alpha, alpha));
                mrun = mnew;
            }
            const float pr = exp2f(sc - mnew);
            float ps = pr;
            ps += __shfl_xor_sync(0xffffffffu, ps, 1);
            ps += __shfl_xor_sync(0xffffffffu, ps, 2);
            ps += __shfl_xor_sync(0xffffffffu, ps, 4);
            lrun += ps;
            if (tok >= 0) {
                const float2 pp2 = make_float2(pr, pr);
#pragma unroll
                for (int jc = 0; jc < C::CPL; ++jc) {
                    const uint4 w = *reinterpret_cast<const uint4*>(vr + (jc * 4 + qt) * 16);
                    float f[C::EPC];
                    chunk_to_float<KT>(w, f);
#pragma unroll
                    for (int e = 0; e < C::EPC; e += 2)
                        ov[(jc * C::EPC + e) / 2] =
                            __ffma2_rn(pp2, make_float2(f[e], f[e + 1]), ov[(jc * C::EPC + e) / 2]);
                }
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    // ---- per warp: reduce the 8 row-lanes of each dim group (lanes r == 0 hold the sums)
#pragma unroll
    for (int i = 0; i < C::DPL / 2; ++i) {
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            ov[i].x += __shfl_xor_sync(0xffffffffu, ov[i].x, o);
            ov[i].y += __shfl_xor_sync(0xffffffffu, ov[i].y, o);
        }
    }
    if (r == 0) {
#pragma unroll
        for (int jc = 0; jc < C::CPL; ++jc) {
            const int dim0 = (jc * 4 + qt) * C::EPC;
#pragma unroll
            for (int e = 0; e < C::EPC; e += 2) {
                wo[warp * D + dim0 + e] = ov[(jc * C::EPC + e) / 2].x;
                wo[warp * D + dim0 + e + 1] = ov[(jc * C::EPC + e) / 2].y;
            }
        }
    }
    if (lane == 0) {
        wm[warp] = mrun;
        wl[warp] = lrun;
    }
    __syncthreads();

    // ---- combine the warps: (M, Lsum, O[d]) in base-2 units
    constexpr float kLn2 = 0.69314718055994530942f;
    for (int dd = tid; dd < D; dd += kGatherThreads) {
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarpsG; ++w) M = fmaxf(M, wm[w]);
        float Ls = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kWarpsG; ++w) {
                if (wm[w] != -CUDART_INF_F) {
                    const float s = exp2f(wm[w] - M);
                    Ls += wl[w] * s;
                    O += wo[w * D + dd] * s;
                }
            }
        }
        if (p.splits == 1) {
            p.out[(int64_t)head * D + dd] = (Ls > 0.f) ? O / Ls : 0.f;
            if (dd == 0) p.lse[head] = (Ls > 0.f) ? (M + log2f(Ls)) * kLn2 : -CUDART_INF_F;
        } else {
            float* pt = p.part + ((int64_t)head * p.splits + split) * (D + 2);
            pt[2 + dd] = O;
            if (dd == 0) {
                pt[0] = M;
                pt[1] = Ls;
            }
        }
    }
    if (p.splits == 1) return;

    __syncthreads();  // every partial store of this CTA precedes thread 0's fence
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&p.counters[head], 1u);
        if (prev >= (unsigned)p.splits) flag_error(p.err, HA_DEVERR_STATE);
        s_last = (prev == (unsigned)(p.splits - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int dd = tid; dd < D; dd += kGatherThreads) {
        const float* pt = p.part + (int64_t)head * p.splits * (D + 2);
        float M = -CUDART_INF_F;
#pragma unroll 8
        for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(pt + (int64_t)s * (D + 2)));
        float Ls = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
            // loads that depend on no branch, so the splits' loads are in flight together
#pragma unroll 8
            for (int s = 0; s < p.splits; ++s) {
                const float* ps = pt + (int64_t)s * (D + 2);
                const float ms = __ldcg(ps), ls = __ldcg(ps + 1), os = __ldcg(ps + 2 + dd);
                const bool live = ms != -CUDART_INF_F;  // an empty split adds nothing
                const float sc = exp2f((live ? ms : M) - M);
                Ls += live ? ls * sc : 0.f;
                O += live ? os * sc : 0.f;
            }
        }
        p.out[(int64_t)head * D + dd] = (Ls > 0.f) ? O / Ls : 0.f;
        if (dd == 0) p.lse[head] = (Ls > 0.f) ? (M + log2f(Ls)) * kLn2 : -CUDART_INF_F;
    }
    if (tid == 0) p.counters[head] = 0u;
}

// Exact merge of two partial attentions (Nectar Eq. (3.4)); one warp per row.
__global__ void __launch_bounds__(256) k_merge(const MergeParams p) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= p.rows) return;
    const float la = p.lse_a[row], lb = p.lse_b[row];
    const float M = fmaxf(la, lb);
    const bool empty = (M == -CUDART_INF_F);
    const float wa = empty ? 0.f : expf(la - M);
    const float wb = empty ? 0.f : expf(lb - M);
    const float S = wa + wb;
    const float ca = empty ? 0.f : wa / S, cb = empty ? 0.f : wb / S;
    const int64_t base = (int64_t)row * p.d;
    for (int k = lane; k < p.d; k += 32) {
        const float oa = p.out_a[base + k], ob = p.out_b[base + k];
        p.out[base + k] = empty ? 0.f : ca * oa + cb * ob;
    }
    __syncwarp();
    if (lane == 0) p.lse[row] = empty ? -CUDART_INF_F : M + logf(S);
}

template <int D, typename KT, bool QREG>
cudaError_t launch_gather_t(const GatherParams& p, cudaStream_t st, bool pdl) {
    using C = Cfg<D, KT>;
    const size_t smem = (size_t)C::OFF_TOKL + (size_t)(p.rows_per_split + p.nseg + 1) * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(k_gather_att<D, KT, QREG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(p.B * p.Hq) * (unsigned)p.splits;
    return launch_ex(k_gather_att<D, KT, QREG>, dim3(grid), dim3(kGatherThreads), smem, st, pdl, p);
}

}  // namespace

cudaError_t launch_gather(const GatherParams& p, int d, int kv_bf16, cudaStream_t st, bool pdl) {
    if (d == 128 && kv_bf16 && p.q_bf16) return launch_gather_t<128, __nv_bfloat16, true>(p, st, pdl);
    if (d == 64 && kv_bf16 && p.q_bf16) return launch_gather_t<64, __nv_bfloat16, true>(p, st, pdl);
    if (d == 128 && kv_bf16) return launch_gather_t<128, __nv_bfloat16, false>(p, st, pdl);
    if (d == 64 && kv_bf16) return launch_gather_t<64, __nv_bfloat16, false>(p, st, pdl);
    if (d == 128 && !kv_bf16) return launch_gather_t<128, float, false>(p, st, pdl);
    if (d == 64 && !kv_bf16) return launch_gather_t<64, float, false>(p, st, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t st) {
    if (p.rows <= 0) return cudaSuccess;
    k_merge<<<(p.rows + 7) / 8, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ha
