// Codes by sign projection: the step before SCORE.
//
// HashAttention: Semantic Sparsity for Faster Inference, Sec. 4.1: the signature
// of a query or key is ReLU(sign(F(x))), i.e. bit j is 1 iff the j-th output of
// the map is positive (0 maps to bit 0). F is learned on the pages; here it is a
// given 32 x d projection W per KV head (sign random projection), so the codes of
// the decode step's queries and of the newly appended keys are 32 GEMVs per
// vector.
//
// k_encode_mlp: the same codes under the map as an MLP d -> H -> H -> 32
// (HashAttention Sec. 5 runs F as 128 -> 128 -> 128 -> 32), with a ReLU after
// each hidden layer (biases throughout): F = W3 relu(W2 relu(W1 x + b1) + b2) + b3.
// One CTA per (KV head, 8 vectors): the head's three weight matrices are copied
// into shared memory by 16-byte cp.async, rows padded by 4 floats so that the
// float4 reads of 8 consecutive rows fall on distinct banks; each layer is
// then computed for the 8 vectors with thread j owning output j (float32
// accumulation over the input in order), and the last layer's signs are a
// warp ballot per vector.
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

constexpr int kMlpVec = 8;        // vectors per CTA
constexpr int kMlpThreads = 256;

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Rows [R][C] of a row-major float matrix into shared memory with pitch C + 4.
__device__ __forceinline__ void stage_rows(const float* src, int R, int C, float* dst) {
    const int c4 = C >> 2, n4 = R * c4;
    for (int i = threadIdx.x; i < n4; i += kMlpThreads) {
        const int r = i / c4, c = (i - r * c4) * 4;
        cp_async16(smem_addr(dst + r * (C + 4) + c), src + (int64_t)r * C + c);
    }
}

// out[v][j] = act(sum_k W[j][k] in[v][k] + b[j]) for the CTA's 8 vectors; J in
// {32, 64, 128} outputs, thread t owns j = t % J for vectors (t / J) * vpt ...
__device__ __forceinline__ void mlp_layer(const float* in, int K, const float* W, const float* bias, int J,
                                          float* out) {
    const int t = threadIdx.x, j = t % J, vg = t / J, vpt = kMlpVec * J / kMlpThreads;
    const float* wj = W + j * (K + 4);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < K; k += 4) {
        const float4 w = *reinterpret_cast<const float4*>(wj + k);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (u < vpt) {
                const float4 x = *reinterpret_cast<const float4*>(in + (vg * vpt + u) * K + k);
                acc[u] = fmaf(w.x, x.x, acc[u]);
                acc[u] = fmaf(w.y, x.y, acc[u]);
                acc[u] = fmaf(w.z, x.z, acc[u]);
                acc[u] = fmaf(w.w, x.w, acc[u]);
            }
        }
    }
    const float bj = bias[j];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        if (u < vpt) out[(vg * vpt + u) * J + j] = fmaxf(acc[u] + bj, 0.f);
}

__global__ void __launch_bounds__(kMlpThreads) k_encode_mlp(const EncodeParams p) {
    extern __shared__ float s_m[];
    const int H = p.hidden, d = p.d, g = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* w1 = s_m;                       // [H][d + 4]
    float* w2 = w1 + H * (d + 4);          // [H][H + 4]
    float* w3 = w2 + H * (H + 4);          // [32][H + 4]
    float* xs = w3 + 32 * (H + 4);         // [8][d]
    float* h1 = xs + kMlpVec * d;          // [8][H]
    float* h2 = h1 + kMlpVec * H;          // [8][H]
    stage_rows(p.W1 + (int64_t)g * H * d, H, d, w1);
    stage_rows(p.W2 + (int64_t)g * H * H, H, H, w2);
    stage_rows(p.W3 + (int64_t)g * 32 * H, 32, H, w3);

    // the CTA's vectors (keys: the token at pos[b] of every batch entry b)
    const int per_g = p.keys ? p.B : p.B * p.G;
    const int v0 = blockIdx.x * kMlpVec;
    for (int i = tid; i < kMlpVec * d; i += kMlpThreads) {
        const int v = i / d, k = i - v * d, vv = v0 + v;
        float x = 0.f;
        if (vv < per_g) {
            int64_t off;
            if (p.keys) {
                const int pos = p.pos[vv];
                off = (pos >= 0 && pos < p.n_cap)
                          ? (int64_t)vv * p.x_sb + (int64_t)g * p.x_sh + (int64_t)pos * p.x_sn + k
                          : -1;
            } else {
                off = (int64_t)(vv / p.G) * p.x_sb + (int64_t)(g * p.G + vv % p.G) * p.x_sh + k;
            }
            if (off >= 0) x = load_elem(p.x, off, p.x_bf16);
        }
        xs[i] = x;
    }
    cp_async_wait_all();
    __syncthreads();
    mlp_layer(xs, d, w1, p.b1 + (int64_t)g * H, H, h1);
    __syncthreads();
    mlp_layer(h1, H, w2, p.b2 + (int64_t)g * H, H, h2);
    __syncthreads();
    // last layer: warp v, lane j -> F_j of vector v; the code is the ballot of F > 0
    const float* w3j = w3 + lane * (H + 4);
    const float* hv = h2 + warp * H;
    float f = 0.f;
    for (int k = 0; k < H; k += 4) {
        const float4 w = *reinterpret_cast<const float4*>(w3j + k);
        const float4 x = *reinterpret_cast<const float4*>(hv + k);
        f = fmaf(w.x, x.x, f);
        f = fmaf(w.y, x.y, f);
        f = fmaf(w.z, x.z, f);
        f = fmaf(w.w, x.w, f);
    }
    f += p.b3[(int64_t)g * 32 + lane];
    const uint32_t code = __ballot_sync(0xffffffffu, f > 0.f);
    const int vv = v0 + warp;
    if (lane != 0 || vv >= per_g) return;
    if (p.keys) {
        const int pos = p.pos[vv];
        if (pos < 0 || pos >= p.n_cap) {
            if (p.flags != nullptr) atomicOr(p.flags, HA_DEVERR_INDEX);
            return;
        }
        p.codes[(int64_t)vv * p.c_sb + (int64_t)g * p.c_sh + pos] = code;
    } else {
        p.codes[(int64_t)(vv / p.G) * p.Hq + g * p.G + vv % p.G] = code;
    }
}

}  // namespace

cudaError_t launch_encode_mlp(const EncodeParams& p, cudaStream_t st) {
    const int per_g = p.keys ? p.B : p.B * p.G;
    if (per_g <= 0) return cudaSuccess;
    const int H = p.hidden, d = p.d;
    const size_t smem = ((size_t)H * (d + 4) + (size_t)H * (H + 4) + 32 * (size_t)(H + 4) +
                         (size_t)kMlpVec * d + 2 * (size_t)kMlpVec * H) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_encode_mlp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((per_g + kMlpVec - 1) / kMlpVec), (unsigned)p.Hkv);
    k_encode_mlp<<<grid, kMlpThreads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_encode(const EncodeParams& p, cudaStream_t st) {
    const int per_g = p.keys ? p.B : p.B * p.G;
    if (per_g <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((per_g + kEncWarps - 1) / kEncWarps), (unsigned)p.Hkv);
    const size_t smem = ((size_t)p.d * 33 + (size_t)kEncWarps * p.d) * sizeof(float);
    k_encode<<<grid, kEncWarps * 32, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ha
