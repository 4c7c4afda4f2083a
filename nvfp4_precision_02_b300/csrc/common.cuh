// common.cuh -- device helpers of the NVFP4 kernels (sm_103a).
//
// Numerics follow the recipe stated in include/nvfp4.h: E2M1 elements in
// 16-element blocks with E4M3 block scales and an FP32 tensor scale
// ("Nemotron 3 Super -- technical report summary", gkm0120.cn, section 1
// pre-training table), SR driven by Philox with 5 rounds ("Nemotron 3 Super"
// summary, papers.lianghsun.dev, section 4.3).  Every FP32 step uses the
// explicit round-to-nearest intrinsics so that no FMA contraction or
// reassociation can change a bit.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace nvfp4 {

// ------------------------------------------------------------------ status
// Sticky device status word; read and cleared by nvfp4_device_status().
__device__ int g_dev_status;

constexpr int DEV_TIMEOUT = 1;
constexpr int DEV_BAD_OFFSETS = 2;

__device__ __forceinline__ void raise_status(int flag) { atomicOr(&g_dev_status, flag); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ formats
// Tensor encode scale: 2688 / amax (1 when amax == 0, FLT_MAX on overflow).
__device__ __forceinline__ float tensor_encode_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    float s = __fdiv_rn(2688.0f, amax);
    if (isinf(s)) s = 3.402823466e38f;
    return s;
}

__device__ __forceinline__ float tensor_decode_scale(float amax) {
    return __fdiv_rn(1.0f, tensor_encode_scale(amax));
}

// E4M3 (OCP OFP8) byte of a non-negative finite float: round to nearest
// even, saturating to 448.  Uses the hardware conversion (.satfinite); both
// halves of the packed result convert x, so the byte order does not matter.
__device__ __forceinline__ uint32_t e4m3_from_float(float x) {
    uint16_t packed;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(packed) : "f"(x));
    return packed & 0xFFu;
}

// Value of a non-negative E4M3 byte (exact in FP32).
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    uint32_t e = (b >> 3) & 15u, m = b & 7u;
    if (e == 0) return __fmul_rn((float)m, 0.001953125f);          // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));         // 2^(e-7) * (1 + m/8)
}

// Block scale byte of a block with largest magnitude bamax.
__device__ __forceinline__ uint32_t block_scale(float bamax, float s_enc) {
    return e4m3_from_float(__fmul_rn(__fdiv_rn(bamax, 6.0f), s_enc));
}

// Per-element multiplier S_enc / sf (only used when sf != 0).
__device__ __forceinline__ float element_ratio(float s_enc, uint32_t sf) {
    return __fdiv_rn(s_enc, e4m3_to_float(sf));
}

// E2M1 magnitude index (0..7) of m >= 0 with round-to-nearest-even and
// saturation: the decision points are the grid midpoints; a midpoint goes
// to the even index (0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2,
// 3.5->4, 5->4).
__device__ __forceinline__ uint32_t e2m1_rne_mag(float m) {
    return (uint32_t)(m > 0.25f) + (uint32_t)(m >= 0.75f) + (uint32_t)(m > 1.25f) +
           (uint32_t)(m >= 1.75f) + (uint32_t)(m > 2.5f) + (uint32_t)(m >= 3.5f) +
           (uint32_t)(m > 5.0f);
}

// E2M1 code (sign << 3 | magnitude) of v with RNE; the sign is copied.
__device__ __forceinline__ uint32_t e2m1_rne(float v) {
    return ((__float_as_uint(v) >> 28) & 8u) | e2m1_rne_mag(fabsf(v));
}

// E2M1 code of v with stochastic rounding by the 32-bit word u: with grid
// neighbours lo <= |v| < hi, p = (|v| - lo) / (hi - lo) (the gaps are powers
// of two, so the product with the reciprocal below is the exact quotient),
// and the magnitude rounds up iff (u >> 8) < p * 2^24.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t u) {
    const uint32_t sign = (__float_as_uint(v) >> 28) & 8u;
    const float m = fabsf(v);
    if (m >= 6.0f) return sign | 7u;
    uint32_t c = (uint32_t)(m >= 0.5f) + (uint32_t)(m >= 1.0f) + (uint32_t)(m >= 1.5f) +
                 (uint32_t)(m >= 2.0f) + (uint32_t)(m >= 3.0f) + (uint32_t)(m >= 4.0f);
    // lo and 1/(hi - lo) for c = 0..6
    const float lo = (c < 4) ? __fmul_rn((float)c, 0.5f) : (c == 4 ? 2.0f : (c == 5 ? 3.0f : 4.0f));
    const float inv_gap = (c < 4) ? 2.0f : (c < 6 ? 1.0f : 0.5f);
    const float p = __fmul_rn(__fsub_rn(m, lo), inv_gap);
    const float thr = __fmul_rn(p, 16777216.0f);
    c += (__uint2float_rn(u >> 8) < thr) ? 1u : 0u;
    return sign | c;
}

// ------------------------------------------------------------------ Philox
// Philox4x32 with R rounds (Salmon et al., SC'11): per round two 32x32->64
// products of counter words 0 and 2, words recombined with the key; the key
// advances by the Weyl constants between rounds.
template <int R>
__device__ __forceinline__ uint4 philox4x32(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r > 0) { k.x += 0x9E3779B9u; k.y += 0xBB67AE85u; }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    }
    return c;
}

// Four random words for output elements 4q .. 4q+3 under seed.
__device__ __forceinline__ uint4 sr_words(uint64_t seed, uint64_t q) {
    return philox4x32<5>(make_uint4((uint32_t)q, (uint32_t)(q >> 32), 0u, 0u),
                         make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}

// ------------------------------------------------------------------ layout
// Byte offset of block scale (r, c) of a [rows, cols] operand (128x4 atoms).
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t cols) {
    const int64_t catoms = (cols / 16 + 3) / 4;
    return ((r >> 7) * catoms + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

__host__ __device__ __forceinline__ int64_t sf_bytes(int64_t rows, int64_t cols) {
    return ((rows + 127) / 128) * 128 * (((cols / 16) + 3) / 4) * 4;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Zero the padding bytes of a swizzled scale buffer (rows beyond `rows` up to
// the next multiple of 128, and scale columns beyond cols/16 up to the next
// multiple of 4), spread over `nthreads` threads with id `tid`.
__device__ __forceinline__ void zero_sf_padding(uint8_t* sf, int64_t rows, int64_t cols,
                                                int64_t tid, int64_t nthreads) {
    const int64_t nc = cols / 16, pc = ((nc + 3) / 4) * 4;
    const int64_t pr = ((rows + 127) / 128) * 128;
    const int64_t right = rows * (pc - nc);           // (r < rows, c >= nc)
    const int64_t bottom = (pr - rows) * pc;          // (r >= rows, any c)
    for (int64_t i = tid; i < right + bottom; i += nthreads) {
        int64_t r, c;
        if (i < right) { r = i / (pc - nc); c = nc + i % (pc - nc); }
        else { const int64_t j = i - right; r = rows + j / pc; c = j % pc; }
        sf[sf_offset(r, c, cols)] = 0;
    }
}

}  // namespace nvfp4
