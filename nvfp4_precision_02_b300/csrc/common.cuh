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

// RN(x / 6) without a division for x >= 2^-125: q0 = RN(x * RN(1/6)),
// r = x - 6 q0 (exact, one fused multiply-add), q = RN(q0 + r * RN(1/6)).
// It equals the IEEE quotient for every float in [2^-125, FLT_MAX] (checked
// exhaustively on the host against x / 6.0f); smaller x take the division.
__device__ __forceinline__ float div6_rn(float x) {
    if (x < 2.35098870e-38f) return __fdiv_rn(x, 6.0f);        // 2^-125
    const float c = 0.16666667f;                              // RN(1/6)
    const float q0 = __fmul_rn(x, c);
    const float r = __fmaf_rn(-q0, 6.0f, x);
    return __fmaf_rn(r, c, q0);
}

// Block scale byte of a block with largest magnitude bamax: RN(RN(bamax / 6)
// * S_enc) converted to E4M3.
__device__ __forceinline__ uint32_t block_scale(float bamax, float s_enc) {
    return e4m3_from_float(__fmul_rn(div6_rn(bamax), s_enc));
}

// Per-element multiplier S_enc / sf (only used when sf != 0).  An infinite
// quotient clamps to FLT_MAX, as the tensor scale does: it overflows only
// when S_enc is already clamped and sf is a small subnormal E4M3 value, and
// the clamp keeps 0 * multiplier at 0 instead of NaN.
__device__ __forceinline__ float element_ratio(float s_enc, uint32_t sf) {
    const float r = __fdiv_rn(s_enc, e4m3_to_float(sf));
    return isinf(r) ? 3.402823466e38f : r;
}

// Eight E2M1 codes (round to nearest even, saturating at 6, sign copied)
// of f[0..7], element j in nibble j, by the hardware conversion
// cvt.rn.satfinite.e2m1x2.f32 (its first source goes to the high nibble).
// The GPU parity tests compare it with the oracle's nearest-value search,
// ties and signed zeros included.
__device__ __forceinline__ uint32_t e2m1x8_rne(const float (&f)[8]) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return out;
}

// E2M1 code of v with stochastic rounding by the 32-bit word u.  With grid
// neighbours lo <= |v| < hi and p = (|v| - lo) / (hi - lo), the magnitude
// rounds up iff (u >> 8) < p * 2^24, i.e. iff u < 256 * ceil(p * 2^24).
// Integer form: X holds m = min(|v|, 6) in code steps with 24 fraction bits
// (X >> 24 = the code rounded down, X mod 2^24 = ceil(p * 2^24)), so adding
// 2^24 - 1 - (u >> 8) carries into bit 24 exactly when the word rounds up:
//   m < 1:  the steps are 0.5 wide, X = ceil(m * 2^25) (the product is exact
//           in FP32; the conversion rounds up);
//   m >= 1: the grid is the FP32 grid with one mantissa bit, and X is four
//           times the FP32 bits of m minus those of 0.5 (exponent and top
//           mantissa bit give the code; the 22 lower mantissa bits, times 4,
//           are p * 2^24 exactly).
// Clamping at 6 gives every |v| >= 6 code 7 (rounding 6 <= |v| < 8 upwards
// included); fminf maps NaN to 6 as well.  It equals the FP32 statement above
// at both sides of every threshold for every finite FP32 input (checked
// exhaustively on the host); the decision is monotone in u, so that covers
// all words.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t u) {
    const float m = fminf(fabsf(v), 6.0f);
    const uint32_t mb = __float_as_uint(m);
    const uint32_t x = mb >= 0x3F800000u ? mb * 4u + 0x04000000u            // 4 (mb - bits(0.5)) mod 2^32
                                         : __float2uint_ru(m * 33554432.0f);
    const uint32_t c = (x + 0x00FFFFFFu - (u >> 8)) >> 24;
    return ((__float_as_uint(v) >> 28) & 8u) | c;
}

// Eight E2M1 codes (RNE) of the 8 bf16 values of v (element 2j in the low
// half of word j) times ratio: per word the two values become FP32 exactly
// (shift / mask), one packed f32x2 multiply rounds each product once (as
// __fmul_rn would), and one hardware conversion encodes the pair.
__device__ __forceinline__ uint32_t e2m1x8_rne_bf16(const uint4 v, float ratio) {
    uint32_t out;
    asm("{\n\t.reg .b64 rr, x0, x1, x2, x3;\n\t.reg .b32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
        ".reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b64 rr, {%5, %5};\n\t"
        "shl.b32 l0, %1, 16;\n\tand.b32 h0, %1, 0xFFFF0000;\n\tmov.b64 x0, {l0, h0};\n\t"
        "shl.b32 l1, %2, 16;\n\tand.b32 h1, %2, 0xFFFF0000;\n\tmov.b64 x1, {l1, h1};\n\t"
        "shl.b32 l2, %3, 16;\n\tand.b32 h2, %3, 0xFFFF0000;\n\tmov.b64 x2, {l2, h2};\n\t"
        "shl.b32 l3, %4, 16;\n\tand.b32 h3, %4, 0xFFFF0000;\n\tmov.b64 x3, {l3, h3};\n\t"
        "mul.rn.f32x2 x0, x0, rr;\n\tmul.rn.f32x2 x1, x1, rr;\n\t"
        "mul.rn.f32x2 x2, x2, rr;\n\tmul.rn.f32x2 x3, x3, rr;\n\t"
        "mov.b64 {l0, h0}, x0;\n\tmov.b64 {l1, h1}, x1;\n\tmov.b64 {l2, h2}, x2;\n\tmov.b64 {l3, h3}, x3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, h0, l0;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, h1, l1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, h2, l2;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, h3, l3;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "f"(ratio));
    return out;
}

// The 8 products bf16(v) * ratio of a half-block, each rounded once (packed
// f32x2 multiplies), for the stochastic encoder.
__device__ __forceinline__ void scale8_bf16(const uint4 v, float ratio, float (&f)[8]) {
    asm("{\n\t.reg .b64 rr, x0, x1, x2, x3;\n\t.reg .b32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
        "mov.b64 rr, {%12, %12};\n\t"
        "shl.b32 l0, %8, 16;\n\tand.b32 h0, %8, 0xFFFF0000;\n\tmov.b64 x0, {l0, h0};\n\t"
        "shl.b32 l1, %9, 16;\n\tand.b32 h1, %9, 0xFFFF0000;\n\tmov.b64 x1, {l1, h1};\n\t"
        "shl.b32 l2, %10, 16;\n\tand.b32 h2, %10, 0xFFFF0000;\n\tmov.b64 x2, {l2, h2};\n\t"
        "shl.b32 l3, %11, 16;\n\tand.b32 h3, %11, 0xFFFF0000;\n\tmov.b64 x3, {l3, h3};\n\t"
        "mul.rn.f32x2 x0, x0, rr;\n\tmul.rn.f32x2 x1, x1, rr;\n\t"
        "mul.rn.f32x2 x2, x2, rr;\n\tmul.rn.f32x2 x3, x3, rr;\n\t"
        "mov.b64 {%0, %1}, x0;\n\tmov.b64 {%2, %3}, x1;\n\tmov.b64 {%4, %5}, x2;\n\tmov.b64 {%6, %7}, x3;\n\t}"
        : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]), "=f"(f[4]), "=f"(f[5]), "=f"(f[6]), "=f"(f[7])
        : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "f"(ratio));
}

// Largest |x| of 16 bf16 values (two uint4 of bf16 pairs) as the 15 magnitude
// bits: seven packed abs-max operations and one final halving.
__device__ __forceinline__ uint32_t bf16x16_absmax(const uint4 a, const uint4 b) {
    uint32_t m;
    asm("{\n\t.reg .b32 t0, t1, t2, t3, u0, u1;\n\t"
        "max.xorsign.abs.bf16x2 t0, %1, %2;\n\t"
        "max.xorsign.abs.bf16x2 t1, %3, %4;\n\t"
        "max.xorsign.abs.bf16x2 t2, %5, %6;\n\t"
        "max.xorsign.abs.bf16x2 t3, %7, %8;\n\t"
        "max.xorsign.abs.bf16x2 u0, t0, t1;\n\t"
        "max.xorsign.abs.bf16x2 u1, t2, t3;\n\t"
        "max.xorsign.abs.bf16x2 %0, u0, u1;\n\t}"
        : "=r"(m)
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w));
    m &= 0x7FFF7FFFu;
    return max(m & 0xFFFFu, m >> 16);
}

// 32 bytes (16 bf16) from global memory in one 256-bit load that bypasses
// L1 (streamed data, read once): a warp's 32 lanes read 1 KB contiguous
// with every 32-byte sector used by one instruction.  p: 32-byte aligned.
__device__ __forceinline__ void ldg32_stream(const void* p, uint4& a, uint4& b) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
}

// ------------------------------------------------------------------ Philox
// Philox4x32 with 5 rounds (Salmon et al., SC'11): per round two 32x32->64
// products of counter words 0 and 2, words recombined with the round key;
// the key advances by the Weyl constants between rounds.  The round keys
// depend on the seed only and are formed once per thread.
struct PhiloxKeys {
    uint32_t k0[5], k1[5];
};

__device__ __forceinline__ PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 5; ++r) {
        k.k0[r] = a;
        k.k1[r] = b;
        a += 0x9E3779B9u;
        b += 0xBB67AE85u;
    }
    return k;
}

// Four random words for output elements 4q .. 4q+3: counter (q, 0, 0).
__device__ __forceinline__ uint4 sr_words(const PhiloxKeys& k, uint64_t q) {
    uint4 c = make_uint4((uint32_t)q, (uint32_t)(q >> 32), 0u, 0u);
#pragma unroll
    for (int r = 0; r < 5; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.k0[r], lo1, hi0 ^ c.w ^ k.k1[r], lo0);
    }
    return c;
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
