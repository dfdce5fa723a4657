// Codes by sign projection: the step before SCORE.
//
// HashAttention: Semantic Sparsity for Faster Inference, Sec. 4.1: the signature
// of a query or key is ReLU(sign(F(x))), i.e. bit j is 1 iff the j-th output of
// the map is positive (0 maps to bit 0). F is learned on the pages; here it is a
// given 32 x d projection W per KV head (sign random projection), so the codes of
// the decode step's queries and of the newly appended keys are 32 GEMVs per
// vector.
//
// k_encode: one CTA per (KV head g, group of 8 vectors of g). The CTA stages
// W[g] transposed in shared memory ([d][33]: lane j reads column j, no bank
// conflict); each warp stages its vector, lane j accumulates projection j in
// float32 as four interleaved partial sums (dims k = 4i + u), and a ballot of
// (projection > 0) is the code.
#include "ha_internal.cuh"

namespace ha {
namespace {

constexpr int kEncWarps = 8;

__device__ __forceinline__ float load_elem(const void* base, int64_t off, int bf16) {
    if (bf16) return __uint_as_float(((uint32_t) reinterpret_cast<const uint16_t*>(base)[off]) << 16);
    return reinterpret_cast<const float*>(base)[off];
}

__global__ void __launch_bounds__(kEncWarps * 32) k_encode(const EncodeParams p) {
    extern __shared__ float s_wt[];  // [d][33], then [kEncWarps][d] vectors
    const int g = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float* Wg = p.W + (int64_t)g * 32 * p.d;
    for (int i = tid; i < 32 * p.d; i += kEncWarps * 32) {
        const int j = i / p.d, k = i - j * p.d;
        s_wt[k * 33 + j] = Wg[i];
    }
    __syncthreads();

    const int v = blockIdx.x * kEncWarps + warp;  // vector of KV head g
    const int per_g = p.keys ? p.B : p.B * p.G;
    if (v >= per_g) return;
    int64_t xoff;
    uint32_t* dst;
    if (p.keys) {
        const int b = v;
        const int pos = p.pos[b];
        if (pos < 0 || pos >= p.n_cap) {
            if (lane == 0 && p.flags != nullptr) atomicOr(p.flags, HA_DEVERR_INDEX);
            return;
        }
        xoff = (int64_t)b * p.x_sb + (int64_t)g * p.x_sh + (int64_t)pos * p.x_sn;
        dst = p.codes + (int64_t)b * p.c_sb + (int64_t)g * p.c_sh + pos;
    } else {
        const int b = v / p.G, h = g * p.G + v % p.G;
        xoff = (int64_t)b * p.x_sb + (int64_t)h * p.x_sh;
        dst = p.codes + (int64_t)b * p.Hq + h;
    }
    float* s_x = s_wt + p.d * 33 + warp * p.d;
    for (int k = lane; k < p.d; k += 32) s_x[k] = load_elem(p.x, xoff + k, p.x_bf16);
    __syncwarp();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < p.d; k += 4) {  // d is a multiple of 4 (64 or 128)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = fmaf(s_wt[(k + u) * 33 + lane], s_x[k + u], acc[u]);
    }
    const float proj = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    const uint32_t code = __ballot_sync(0xffffffffu, proj > 0.f);
    if (lane == 0) *dst = code;
}

}  // namespace

cudaError_t launch_encode(const EncodeParams& p, cudaStream_t st) {
    const int per_g = p.keys ? p.B : p.B * p.G;
    if (per_g <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((per_g + kEncWarps - 1) / kEncWarps), (unsigned)p.Hkv);
    const size_t smem = ((size_t)p.d * 33 + (size_t)kEncWarps * p.d) * sizeof(float);
    k_encode<<<grid, kEncWarps * 32, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ha
