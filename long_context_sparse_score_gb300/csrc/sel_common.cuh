// Device helpers of the fused selection shared by k_sel_scan / k_sel_emit and
// k_group_att: warp reductions and the byte-wise threshold masks over a lane
// block of 32 packed distance words.
#pragma once

#include "ha_internal.cuh"

namespace ha {

static __device__ __forceinline__ uint32_t warp_sum_u(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

static __device__ __forceinline__ int warp_excl_scan(int v, int* total) {
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

static __device__ __forceinline__ void red_add_shared(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

static __device__ __forceinline__ uint32_t half_field(uint32_t w01, uint32_t w23, int e) {
    const uint32_t w = (e < 2) ? w01 : w23;
    return (e & 1) ? (w >> 16) : (w & 0xffffu);
}

// Bits [0, k) set, k clamped to [0, 32].
static __device__ __forceinline__ uint32_t low_bits(int k) {
    return k <= 0 ? 0u : (k >= 32 ? 0xffffffffu : ((1u << k) - 1u));
}

// Per-head masks over a lane block of 32 tokens: bit j of m[e] is set iff byte e
// of D[j] is at most byte e of the threshold word, where TE holds 0x80 + T_e in
// byte e (T_e in [-1, 32]; distances are at most 32, so no byte borrows from its
// neighbour and bit 7 of byte e of TE - D[j] is set exactly when D_e <= T_e).
static __device__ __forceinline__ void le_masks(const uint32_t (&D)[32], uint32_t TE, uint32_t (&m)[4]) {
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
static __device__ __forceinline__ uint32_t thresh_word(const int (&T)[4], int nh) {
    uint32_t w = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) w |= (uint32_t)((e < nh) ? (0x80 + T[e]) : 0x7F) << (8 * e);
    return w;
}

// Keep the first q set bits of x (q >= 0).
static __device__ __forceinline__ uint32_t first_bits(uint32_t x, int q) {
    uint32_t keep = 0u;
    while (x != 0u && q > 0) {
        const uint32_t low = x & (0u - x);
        keep |= low;
        x ^= low;
        --q;
    }
    return keep;
}


}  // namespace ha
