// Multi-segment merge of partial attentions.
//
// Nectar: Neural Estimation of Cached-Token Attention via Regression, Sec. 3:
// a segment whose scores are not materialised enters the softmax as one
// virtual logit lse_s carrying the value out_s, and Eq. (3.4) applied to every
// segment gives L = log sum_s e^{lse_s}, out = sum_s e^{lse_s - L} out_s for any
// number of segments (a sparse document part, a dense local part, generated
// tokens).
#include "ha_internal.cuh"

#include <math_constants.h>

#include <algorithm>

namespace ha {
namespace {

// Exact merge of nseg partial attentions (Nectar Sec. 3, Eq. (3.4) over every
// segment); one warp per row, the warps of the grid striding over the rows. Per
// row every lane starts the loads of its dims of the first four segments, then
// turns the segments' lse into the row's peak, mass and per-segment weights
// e^{lse_s - L} while they are in flight, and sums its dims over the segments,
// four segments' loads in flight at a time (16-byte loads when d and the
// strides allow).
template <bool VEC>
__global__ void __launch_bounds__(256, 5) k_merge_n(const MergeNParams p) {
    const int lane = threadIdx.x & 31;
    constexpr int W = VEC ? 4 : 1;  // floats per load
    const int nwarps = gridDim.x * 8;
    for (int row = blockIdx.x * 8 + (threadIdx.x >> 5); row < p.rows; row += nwarps) {
        const float* lr = p.lses + row;
        const int64_t base = (int64_t)row * p.d;
        // the values of segments s0 .. s0 + 3 at dims k .. k + W - 1
        auto load4 = [&](int s0, int k, float (&v)[4][W]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = s0 + u;
                const float* src = p.outs + (int64_t)(s < p.nseg ? s : 0) * p.out_seg_stride + base + k;
                if (VEC) {
                    const float4 x = *reinterpret_cast<const float4*>(src);
                    v[u][0] = x.x;
                    v[u][W > 1 ? 1 : 0] = x.y;
                    v[u][W > 2 ? 2 : 0] = x.z;
                    v[u][W > 3 ? 3 : 0] = x.w;
                } else {
                    v[u][0] = *src;
                }
            }
        };
        float v[4][W];  // the first block is loaded before the weights are formed
        if (lane * W < p.d) load4(0, lane * W, v);
        float M = -CUDART_INF_F;
        for (int s = 0; s < p.nseg; ++s) M = fmaxf(M, lr[(int64_t)s * p.lse_seg_stride]);
        const bool empty = (M == -CUDART_INF_F);
        float S = 0.f;
        if (!empty)
            for (int s = 0; s < p.nseg; ++s) S += expf(lr[(int64_t)s * p.lse_seg_stride] - M);
        const float inv = empty ? 0.f : 1.f / S;
        for (int k = lane * W; k < p.d; k += 32 * W) {
            float acc[W];
#pragma unroll
            for (int e = 0; e < W; ++e) acc[e] = 0.f;
            for (int s0 = 0; s0 < p.nseg; s0 += 4) {  // an empty row has all weights 0
                if (s0 != 0 || k != lane * W) load4(s0, k, v);
                float wgt[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int s = s0 + u;
                    const float l = (s < p.nseg) ? lr[(int64_t)s * p.lse_seg_stride] : -CUDART_INF_F;
                    wgt[u] = (empty || l == -CUDART_INF_F) ? 0.f : expf(l - M) * inv;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int e = 0; e < W; ++e) acc[e] += (wgt[u] != 0.f) ? wgt[u] * v[u][e] : 0.f;
            }
            if (VEC) {
                *reinterpret_cast<float4*>(p.out + base + k) = make_float4(acc[0], acc[W > 1 ? 1 : 0],
                                                                          acc[W > 2 ? 2 : 0], acc[W > 3 ? 3 : 0]);
            } else {
                p.out[base + k] = acc[0];
            }
        }
        __syncwarp();  // every lane has read the segments' lse before lane 0 may overwrite one
        if (lane == 0) p.lse[row] = empty ? -CUDART_INF_F : M + logf(S);
    }
}

}  // namespace

cudaError_t launch_merge_n(const MergeNParams& p, cudaStream_t st) {
    if (p.rows <= 0) return cudaSuccess;
    const bool vec = (p.d % 4 == 0) && (p.out_seg_stride % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.outs) | reinterpret_cast<uintptr_t>(p.out)) & 15u) == 0;
    // five 256-thread CTAs per SM (48 registers) at most; the warps stride over the rows
    const int grid = std::min((p.rows + 7) / 8, 5 * kSMs);
    if (vec) k_merge_n<true><<<grid, 256, 0, st>>>(p);
    else k_merge_n<false><<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ha
