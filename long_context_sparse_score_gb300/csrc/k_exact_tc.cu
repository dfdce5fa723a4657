// Scores of the exact comparator on the tensor cores: z[b, h, i] = <q[b, h], k_i>
// for every cached token i < n of bf16 keys.
//
// HashAttention: Semantic Sparsity for Faster Inference, Sec. 5 measures the
// hashed selection against the top-k by attention score; the scores of one KV
// head g are the product Q_g K_g^T of its G query rows with all of its cached
// rows, a dense contraction streamed once from HBM.
//
// k_qsplit       per (b, g): the query tile, NCOL rows of d bf16 values; row
//                3 hh + j holds part j of query head hh, where hi = bf16(q),
//                mid = bf16(q - hi), lo = bf16(q - hi - mid). For a float32
//                q the three parts sum to q exactly (each takes the next 8
//                significant bits), so the three partial dot products add up
//                to the float32 score up to accumulation rounding; for a bf16
//                q, mid = lo = 0.
// k_dot_scores_tc persistent, one CTA per SM, 6 warps:
//                warp 0  lane 0 streams tiles of 128 K rows and the matching
//                        query tile into a ring of shared-memory stages by TMA
//                        (128-byte swizzle, zero fill past n_cap);
//                warp 1  owns the tensor memory (two accumulators of NCOL
//                        float32 columns) and lane 0 issues the d / 16
//                        tcgen05.mma (M = 128, N = NCOL, K = 16, bf16 inputs,
//                        float32 accumulate) of every tile;
//                warps 2-5 read the accumulator rows back (tcgen05.ld, one
//                        TMEM lane quadrant each), add the three parts of every
//                        head and store 32 consecutive scores per head.
// Every wait is bounded: a wait that gives up flags HA_DEVERR_TIMEOUT, stops
// the other roles, lets the copies and products in flight land and frees the
// tensor memory before the CTA exits.
#include "ha_internal.cuh"

#include <cuda.h>

namespace ha {
namespace {

constexpr int kTcRows = 128;             // K rows per tile (the MMA's M)
constexpr int kTcThreads = 192;
constexpr int kTcSmemBudget = 220 * 1024;

template <int D, int NCOL>
struct TcCfg {
    static constexpr int kA = kTcRows * D * 2;   // bytes of a K tile
    static constexpr int kB = NCOL * D * 2;      // bytes of a query tile
    static constexpr int kStage = kA + kB;       // a multiple of 1024 (swizzle atoms stay aligned)
    static constexpr int kStages = (kTcSmemBudget / kStage) < 8 ? (kTcSmemBudget / kStage) : 8;
    static constexpr int kSpans = D / 64;        // 128-byte swizzle spans of a row
    static constexpr uint32_t kTmemCols = (2 * NCOL <= 32) ? 32u : ((2 * NCOL <= 64) ? 64u : 128u);
    static constexpr int kBarBytes = 8 * (2 * kStages + 5) + 16;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kBarBytes;
    static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment");
    static_assert(NCOL % 16 == 0 && NCOL <= 64, "N of the MMA");
};

// kind::f16 instruction descriptor: float32 accumulator, bf16 A and B, both
// K-major, N = NCOL, M = 128.
template <int NCOL>
__host__ __device__ constexpr uint32_t mma_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NCOL >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle
// layout that TMA writes: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmap_prefetch(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive float32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Wait with the time limit only (teardown: copies in flight always land).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ uint16_t bf16_bits(__nv_bfloat16 x) { return __bfloat16_as_ushort(x); }

// grid: B * Hkv; writes qt[bg][NCOL][D].
template <int NCOL>
__global__ void __launch_bounds__(256) k_qsplit(const ExactParams p, int D) {
    const int bg = blockIdx.x;
    const int b = bg / p.Hkv, g = bg - b * p.Hkv;
    uint16_t* dst = p.qt + (int64_t)bg * NCOL * D;
    for (int i = threadIdx.x; i < NCOL * D; i += blockDim.x) {
        const int j = i / D, k = i - j * D;
        const int hh = j / 3, part = j - 3 * hh;
        uint16_t out = 0;
        if (hh < p.G) {
            const int64_t off = (int64_t)b * p.q_sb + (int64_t)(g * p.G + hh) * p.q_sh + k;
            const float x = p.q_bf16 ? __uint_as_float(((uint32_t) reinterpret_cast<const uint16_t*>(p.q)[off]) << 16)
                                     : reinterpret_cast<const float*>(p.q)[off];
            const __nv_bfloat16 hi = __float2bfloat16_rn(x);
            const float r1 = x - __bfloat162float(hi);
            const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(mid);
            const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
            out = part == 0 ? bf16_bits(hi) : (part == 1 ? bf16_bits(mid) : bf16_bits(lo));
        }
        dst[i] = out;
    }
}

template <int D, int NCOL>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_dot_scores_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                    const ExactParams p, const int tiles_per_bg) {
    using C = TcCfg<D, NCOL>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t s_raw[];
    const uint32_t raw = smem_addr(s_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + (uint32_t)(S * C::kStage);
    uint8_t* gbars = s_raw + (bars - raw);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(gbars + 8 * (2 * S + 5));
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    auto full = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bars + 8u * (uint32_t)(S + s); };
    auto tfull = [&](int a) { return bars + 8u * (uint32_t)(2 * S + a); };
    auto tempty = [&](int a) { return bars + 8u * (uint32_t)(2 * S + 2 + a); };
    const uint32_t done = bars + 8u * (uint32_t)(2 * S + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), 4);
        }
        mbar_init(done, 1);
        *s_abort = 0;
        mbar_fence_init();
        tmap_prefetch(&tmK);
        tmap_prefetch(&tmQ);
    }
    if (warp == 1) tmem_alloc(smem_addr(s_tmem), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const long long T = (long long)p.B * p.Hkv * tiles_per_bg;
    // tile t -> (b, g, first row, valid length); the same rule in every role
    auto tile_of = [&](long long t, int& b, int& g, int& row0, int& n, bool report) {
        const int bg = (int)(t / tiles_per_bg);
        row0 = (int)(t - (long long)bg * tiles_per_bg) * kTcRows;
        b = bg / p.Hkv;
        g = bg - b * p.Hkv;
        n = checked_len(p.seq_lens, b, p.n_cap, p.err, report && row0 == 0 && g == 0);
        return row0 < n;
    };
    auto give_up = [&]() {
        flag_error(p.err, HA_DEVERR_TIMEOUT);
        *s_abort = 1;
    };

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (long long t = blockIdx.x; t < T; t += gridDim.x) {
                int b, g, row0, n;
                if (!tile_of(t, b, g, row0, n, false)) continue;
                const int s = it % S;
                const uint32_t ph = (uint32_t)(it / S) & 1u;
                if (!mbar_wait_bounded(empty(s), ph ^ 1u, s_abort)) {
                    give_up();
                    break;
                }
                const uint32_t a_s = base + (uint32_t)(s * C::kStage), b_s = a_s + (uint32_t)C::kA;
                mbar_arrive_expect_tx(full(s), (uint32_t)C::kStage);
#pragma unroll
                for (int h = 0; h < C::kSpans; ++h) {
                    tma_load_4d(a_s + (uint32_t)(h * kTcRows * 128), &tmK, full(s), h * 64, row0,
                                p.k_sh != 0 ? g : 0, p.k_sb != 0 ? b : 0);
                    tma_load_2d(b_s + (uint32_t)(h * NCOL * 128), &tmQ, full(s), h * 64, (b * p.Hkv + g) * NCOL);
                }
                ++it;
            }
            // before the CTA can exit: the products of the last stages have released
            // them (their arrivals land in this CTA's shared memory), or, after a
            // timeout, at least the copies into them have landed
            const bool clean = *s_abort == 0;
            for (int j = (it > S ? it - S : 0); j < it; ++j)
                mbar_wait_drain(clean ? empty(j % S) : full(j % S), (uint32_t)(j / S) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = mma_idesc<NCOL>();
            int it = 0;
            for (long long t = blockIdx.x; t < T; t += gridDim.x) {
                int b, g, row0, n;
                if (!tile_of(t, b, g, row0, n, false)) continue;
                const int s = it % S, a = it & 1;
                const uint32_t ph = (uint32_t)(it / S) & 1u, aph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait_bounded(tempty(a), aph ^ 1u, s_abort)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                if (!mbar_wait_bounded(full(s), ph, s_abort)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t a_s = base + (uint32_t)(s * C::kStage), b_s = a_s + (uint32_t)C::kA;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t h = (uint32_t)(kk >> 2), k32 = (uint32_t)(kk & 3) * 32u;
                    tc_mma(tmem + (uint32_t)(a * NCOL), sw128_desc(a_s + h * (kTcRows * 128) + k32),
                           sw128_desc(b_s + h * (NCOL * 128) + k32), idesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(empty(s));
                tc_commit(tfull(a));
                ++it;
            }
            tc_commit(done);  // every product issued above has finished once this arrives
            mbar_wait_drain(done, 0u);
        }
        __syncwarp();
    } else {
        const int wq = warp & 3;  // TMEM lanes 32 wq .. 32 wq + 31 (accumulator rows)
        int it = 0;
        for (long long t = blockIdx.x; t < T; t += gridDim.x) {
            int b, g, row0, n;
            if (!tile_of(t, b, g, row0, n, warp == 2 && lane == 0)) continue;
            const int a = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            const bool ok = mbar_wait_bounded(tfull(a), aph, s_abort);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            uint32_t v[NCOL];
#pragma unroll
            for (int c = 0; c < NCOL / 16; ++c)
                tmem_ld16(tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(a * NCOL + c * 16), v + c * 16);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(a));
            const int row = row0 + wq * 32 + lane;
            if (row < n) {
                float* dst = p.scores + ((int64_t)b * p.Hq + (int64_t)g * p.G) * p.n_cap + row;
#pragma unroll
                for (int hh = 0; hh < NCOL / 3; ++hh) {
                    if (hh < p.G)
                        dst[(int64_t)hh * p.n_cap] =
                            (__uint_as_float(v[3 * hh]) + __uint_as_float(v[3 * hh + 1])) + __uint_as_float(v[3 * hh + 2]);
                }
            }
            ++it;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn load_encode_fn() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
}

EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = load_encode_fn();
    return fn;
}

template <int D, int NCOL>
cudaError_t launch_tc_t(const ExactParams& p, cudaStream_t st, bool* used) {
    using C = TcCfg<D, NCOL>;
    const EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaSuccess;
    // K [B][Hkv][n_cap][D] bf16 with the caller's strides; boxes of 128 rows x 64 values.
    // A stride of 0 (a cache shared by every batch entry or head) becomes an
    // extent of 1 read at coordinate 0.
    CUtensorMap tmK, tmQ;
    const cuuint64_t span = (cuuint64_t)p.n_cap * p.k_sn * 2;
    const cuuint64_t kdim[4] = {(cuuint64_t)D, (cuuint64_t)p.n_cap, p.k_sh ? (cuuint64_t)p.Hkv : 1u,
                                p.k_sb ? (cuuint64_t)p.B : 1u};
    const cuuint64_t kstr[3] = {(cuuint64_t)p.k_sn * 2, p.k_sh ? (cuuint64_t)p.k_sh * 2 : span,
                                p.k_sb ? (cuuint64_t)p.k_sb * 2 : span};
    const cuuint32_t kbox[4] = {64u, (cuuint32_t)kTcRows, 1u, 1u};
    const cuuint32_t unit[4] = {1u, 1u, 1u, 1u};
    if (enc(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<char*>(p.K), kdim, kstr, kbox, unit,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaSuccess;  // a layout TMA cannot describe: the caller takes the CUDA-core kernel
    const cuuint64_t qdim[2] = {(cuuint64_t)D, (cuuint64_t)p.B * p.Hkv * NCOL};
    const cuuint64_t qstr[1] = {(cuuint64_t)D * 2};
    const cuuint32_t qbox[2] = {64u, (cuuint32_t)NCOL};
    if (enc(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.qt, qdim, qstr, qbox, unit, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaSuccess;
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_dot_scores_tc<D, NCOL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    const int tiles_per_bg = (p.n_cap + kTcRows - 1) / kTcRows;
    const long long T = (long long)p.B * p.Hkv * tiles_per_bg;
    const unsigned grid = (unsigned)(T < nsm ? T : nsm);
    k_qsplit<NCOL><<<p.B * p.Hkv, 256, 0, st>>>(p, D);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_dot_scores_tc<D, NCOL><<<grid, kTcThreads, C::kSmem, st>>>(tmK, tmQ, p, tiles_per_bg);
    e = cudaGetLastError();
    if (e == cudaSuccess) *used = true;
    return e;
}

}  // namespace

cudaError_t launch_scores_tc(const ExactParams& p, int d, cudaStream_t st, bool* used) {
    *used = false;
    if (p.qt == nullptr || 3 * p.G > 64) return cudaSuccess;
    const int ncol = (3 * p.G + 15) / 16 * 16;  // three parts per query head, in units of 16 columns
    if (d == 128) {
        if (ncol == 16) return launch_tc_t<128, 16>(p, st, used);
        if (ncol == 32) return launch_tc_t<128, 32>(p, st, used);
        if (ncol == 48) return launch_tc_t<128, 48>(p, st, used);
        return launch_tc_t<128, 64>(p, st, used);
    }
    if (d == 64) {
        if (ncol == 16) return launch_tc_t<64, 16>(p, st, used);
        if (ncol == 32) return launch_tc_t<64, 32>(p, st, used);
        if (ncol == 48) return launch_tc_t<64, 48>(p, st, used);
        return launch_tc_t<64, 64>(p, st, used);
    }
    return cudaSuccess;
}

}  // namespace ha
