/*
 * oracle.c -- plain, slow CPU statement of the NVFP4 training linear-layer
 * path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU
 * baseline leg of the benchmark are the only callers.  It shares no code,
 * header, table or constant generator with the CUDA library.
 *
 * What the pages fix (sources are web pages summarising the Nemotron 3
 * Super / Ultra technical reports):
 *   [S-recipe] "Nemotron 3 Super -- technical report summary" (gkm0120.cn),
 *       section 1, pre-training table, row "training precision": NVFP4 is E2M1
 *       elements in 16-element micro-blocks with E4M3 scaling.
 *   [S-infra]  same page, "Infra design" table: NVFP4 GEMMs for fprop, dgrad
 *       and wgrad; 2D block scaling for weights, 1D block scaling for
 *       gradients and activations; random Hadamard transforms and
 *       stochastic rounding.
 *   [U-2.2]    "Nemotron 3 Ultra: Open, Efficient Mixture-of-Experts Hybrid
 *       Mamba-Transformer Model for Agentic Reasoning" (papercache.org
 *       translation), section 2.2 "NVFP4 pretraining": E2M1, 2D block
 *       quantisation of weights, RHT on the inputs of wgrad, SR on gradients.
 *   [SL-2.2]   "Nemotron 3 Super" summary (papers.lianghsun.dev), section 2.2:
 *       routed-expert GEMMs run in NVFP4; small gradients underflow to zero.
 *   [SL-4.2]   same page, section 4.2: activations use dynamic, per-block,
 *       max-based scaling.
 *   [SL-4.3]   same page, section 4.3: RTNE is biased, SR is unbiased; SR
 *       driven by a Philox generator with 5 rounds.
 *
 * Readings where the pages are silent (each also stated at its function):
 *   R1 tensor scale  S_enc = 2688 / amax (6 * 448, one FP32 division);
 *      amax == 0 -> 1; an infinite quotient clamps to FLT_MAX; dec = 1/S_enc.
 *   R2 block scale   sf = E4M3_RNE_satfinite((bamax / 6) * S_enc), two FP32
 *      ops in that order.
 *   R3 element       sf == 0 -> code +0; else v = x * (S_enc / sf) in FP32 (an
 *      infinite quotient clamps to FLT_MAX, as in R1) and v is rounded to
 *      E2M1 (RNE, saturating at 6), sign copied from x.
 *   R4 SR            Philox4x32 with 5 rounds, key = seed, counter =
 *      (e >> 2, 0, 0), word e & 3, e = row-major index in the quantised
 *      output; round up iff (u >> 8) < p * 2^24.
 *   R5 RHT           16-point Sylvester Hadamard along the quantised K axis,
 *      y = 0.25 * H * (s .* x), FP32 butterfly with stages 1, 2, 4, 8.
 *   R8 grouped       one tensor amax per expert (oracle_quantize_1d_grouped,
 *      the batched oracle_quantize_2d).
 *   R9 2D tiles      rows and columns of a 2D-quantised weight are multiples
 *      of 16.
 *   Layouts (not a reading of the method): codes packed two per byte (even
 *      index in the low nibble); block scales in 128x4 atoms (see
 *      oracle_sf_offset).
 *   R14 expert segments of the grouped wgrad (oracle_rht_quantize_grouped).
 *   R15 FP16 SR of the SSM cache (oracle_fp16_sr).
 *   R16 PTQ block scales by minimum squared error (oracle_quantize_1d_mse).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * The FP32 steps must not be contracted into FMAs or reassociated.
 */
#include <math.h>
#include <float.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Element formats [S-recipe], [U-2.2].                                 */
/* ------------------------------------------------------------------ */

/* E2M1 magnitudes, indexed by the three low bits of a code (OCP MX E2M1). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Value of a 4-bit E2M1 code: bit 3 is the sign. */
double oracle_e2m1_value(int code)
{
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* Value of an E4M3 byte (OCP OFP8 E4M3: bias 7, no infinities,
 * 0x7F / 0xFF are NaN, subnormals 2^-6 * m/8). */
double oracle_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* E4M3 encode of a non-negative finite float, round to nearest with ties to
 * the even code, saturating at 448 (R2).  Exhaustive nearest search over the
 * 127 non-negative finite codes: slow and obviously correct. */
uint8_t oracle_e4m3_encode(float x)
{
    int best = 0, c;
    double bestd, d;
    if (x >= 448.0f) return 0x7E;
    bestd = fabs((double)x);                      /* distance to code 0 */
    for (c = 1; c <= 0x7E; ++c) {
        d = fabs((double)x - oracle_e4m3_value(c));
        if (d < bestd || (d == bestd && (c & 1) == 0)) { best = c; bestd = d; }
    }
    return (uint8_t)best;
}

/* E2M1 magnitude code (0..7) of m >= 0: nearest grid value, ties to the
 * even code, |m| > 6 saturates to 6 (R3). */
static int e2m1_rne_mag(float m)
{
    int best = 0, c;
    double bestd, d;
    if (m > 6.0f) return 7;
    bestd = fabs((double)m - E2M1_MAG[0]);
    for (c = 1; c < 8; ++c) {
        d = fabs((double)m - E2M1_MAG[c]);
        if (d < bestd || (d == bestd && (c & 1) == 0)) { best = c; bestd = d; }
    }
    return best;
}

/* E2M1 code of v, round to nearest even; sign copied from v (so a negative
 * value that rounds to zero gives code 0x8). */
int oracle_e2m1_rne(float v)
{
    int s = signbit(v) ? 8 : 0;
    return s | e2m1_rne_mag(fabsf(v));
}

/* E2M1 code of v with stochastic rounding driven by the 32-bit word u (R4):
 * m = |v|; m >= 6 gives 6; otherwise lo <= m < hi are the neighbouring grid
 * values, p = (m - lo) / (hi - lo) (exact in FP32: Sterbenz, power-of-two
 * gap), and the result is hi iff (u >> 8) < p * 2^24. */
int oracle_e2m1_sr(float v, uint32_t u)
{
    int s = signbit(v) ? 8 : 0;
    float m = fabsf(v), p, lo, hi;
    int c;
    if (m >= 6.0f) return s | 7;
    c = 0;
    while (c < 7 && (float)E2M1_MAG[c + 1] <= m) ++c;     /* lo = grid[c] */
    lo = (float)E2M1_MAG[c];
    hi = (float)E2M1_MAG[c + 1];
    p = (m - lo) / (hi - lo);
    if ((float)(u >> 8) < p * 16777216.0f) ++c;
    return s | c;
}

/* ------------------------------------------------------------------ */
/* Philox4x32 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as  */
/* easy as 1, 2, 3", SC'11): R rounds of the Philox S-box, key bumped by */
/* the Weyl constants between rounds.  [SL-4.3] names Philox<5>.          */
/* ------------------------------------------------------------------ */
void oracle_philox4x32(const uint32_t ctr_in[4], const uint32_t key_in[2],
                       int rounds, uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    int r;
    for (r = 0; r < rounds; ++r) {
        uint64_t p0, p1;
        uint32_t n0, n1, n2, n3;
        if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        p0 = (uint64_t)0xD2511F53u * c0;
        p1 = (uint64_t)0xCD9E8D57u * c2;
        n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        n1 = (uint32_t)p1;
        n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The random word for element e of a quantised output under seed (R4). */
uint32_t oracle_sr_word(uint64_t seed, uint64_t e)
{
    uint32_t ctr[4], key[2], out[4];
    uint64_t q = e >> 2;
    ctr[0] = (uint32_t)q; ctr[1] = (uint32_t)(q >> 32); ctr[2] = 0; ctr[3] = 0;
    key[0] = (uint32_t)seed; key[1] = (uint32_t)(seed >> 32);
    oracle_philox4x32(ctr, key, 5, out);
    return out[e & 3];
}

/* ------------------------------------------------------------------ */
/* Scales (R1, R2).                                                     */
/* ------------------------------------------------------------------ */

/* Per-tensor encode scale: largest block maps to E4M3 448, element to 6. */
float oracle_tensor_scale(float amax)
{
    float s;
    if (amax == 0.0f) return 1.0f;
    s = 2688.0f / amax;
    if (isinf(s)) s = FLT_MAX;
    return s;
}

/* Per-tensor decode scale used for dequantisation and the GEMM alpha. */
float oracle_tensor_decode_scale(float amax)
{
    return 1.0f / oracle_tensor_scale(amax);
}

/* E4M3 block scale of a block whose largest magnitude is bamax (R2). */
uint8_t oracle_block_scale(float bamax, float s_enc)
{
    float t = bamax / 6.0f;
    float sf = t * s_enc;
    return oracle_e4m3_encode(sf);
}

/* Element multiplier S_enc / e4m3(sf) of a block (R3): one FP32 division;
 * an infinite quotient clamps to FLT_MAX, as R1's tensor scale does (it
 * overflows only when S_enc is already near FLT_MAX and sf is a small
 * subnormal E4M3 value; the clamp keeps 0 * multiplier at 0). */
static float element_multiplier(float s_enc, float sfv)
{
    float r = s_enc / sfv;
    if (isinf(r)) r = FLT_MAX;
    return r;
}

/* Encode one block of n values (n <= 16, all sharing block scale sf).
 * Output: one 4-bit code per byte of codes[].  For SR the element of value
 * j has output index e0 + j * estride. */
static void encode_block(const float *x, int n, float s_enc, uint8_t sf,
                         int mode, uint64_t seed, uint64_t e0, uint64_t estride,
                         uint8_t *codes)
{
    int j;
    float r;
    if (sf == 0) { for (j = 0; j < n; ++j) codes[j] = 0; return; }
    r = element_multiplier(s_enc, (float)oracle_e4m3_value(sf));
    for (j = 0; j < n; ++j) {
        float v = x[j] * r;
        if (mode == 0) codes[j] = (uint8_t)oracle_e2m1_rne(v);
        else codes[j] = (uint8_t)oracle_e2m1_sr(v, oracle_sr_word(seed, e0 + (uint64_t)j * estride));
    }
}

/* Exported single-block encoder (tests use it on hand-worked blocks). */
void oracle_encode_block(const float *x, int n, float s_enc, int mode,
                         uint64_t seed, uint64_t e0, uint8_t *sf_out, uint8_t *codes)
{
    float bamax = 0.0f;
    int j;
    for (j = 0; j < n; ++j) if (fabsf(x[j]) > bamax) bamax = fabsf(x[j]);
    *sf_out = oracle_block_scale(bamax, s_enc);
    encode_block(x, n, s_enc, *sf_out, mode, seed, e0, 1, codes);
}

/* ------------------------------------------------------------------ */
/* Layouts.                                                             */
/* ------------------------------------------------------------------ */

static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Block scales of a [rows, cols] tensor (cols/16 scale columns) are stored in
 * atoms of 128 rows x 4 scale columns (512 bytes).  Atoms are ordered by
 * row-atom, then column-atom; inside an atom the byte for (r, c) sits at
 * (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.  Rows pad to 128 and scale
 * columns to 4; padding bytes are zero. */
int64_t oracle_sf_offset(int64_t r, int64_t c, int64_t cols)
{
    int64_t catoms = (cols / 16 + 3) / 4;
    int64_t atom = (r / 128) * catoms + c / 4;
    return atom * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

size_t oracle_sf_bytes(int64_t rows, int64_t cols)
{
    return (size_t)((rows + 127) / 128) * 128 * (size_t)(((cols / 16) + 3) / 4) * 4;
}

static void put_code(uint8_t *codes, int64_t row, int64_t col, int64_t cols, uint8_t code)
{
    uint8_t *b = codes + row * (cols / 2) + col / 2;
    if (col & 1) *b = (uint8_t)((*b & 0x0F) | (code << 4));
    else         *b = (uint8_t)((*b & 0xF0) | (code & 0x0F));
}

/* ------------------------------------------------------------------ */
/* Amax.                                                                */
/* ------------------------------------------------------------------ */

float oracle_amax_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld)
{
    float a = 0.0f;
    int64_t r, c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c) {
            float v = fabsf(bf16_to_float(x[r * ld + c]));
            if (v > a) a = v;
        }
    return a;
}

/* ------------------------------------------------------------------ */
/* 1D (1x16) quantisation of activations and gradients [S-infra].       */
/* x: bf16 [rows, cols] with row stride ld (elements); cols % 16 == 0.   */
/* codes: [rows, cols/2]; sf: oracle_sf_bytes(rows, cols) bytes.         */
/* amax_in (nullable) replaces the computed tensor amax; the amax used   */
/* is written to *amax_out.  SR index e = r * cols + c.                  */
/* ------------------------------------------------------------------ */
static void quantize_rows(const uint16_t *x, int64_t row0, int64_t nrows, int64_t cols,
                          int64_t ld, int mode, uint64_t seed, float amax,
                          uint8_t *codes, uint8_t *sf, int64_t sf_row0)
{
    float s_enc = oracle_tensor_scale(amax);
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t r = row0 + i, b;
        float blk[16];
        uint8_t cd[16];
        for (b = 0; b < cols / 16; ++b) {
            float bamax = 0.0f;
            uint8_t s;
            int j;
            for (j = 0; j < 16; ++j) {
                blk[j] = bf16_to_float(x[r * ld + b * 16 + j]);
                if (fabsf(blk[j]) > bamax) bamax = fabsf(blk[j]);
            }
            s = oracle_block_scale(bamax, s_enc);
            sf[oracle_sf_offset(sf_row0 + i, b, cols)] = s;
            encode_block(blk, 16, s_enc, s, mode, seed, (uint64_t)(r * cols + b * 16), 1, cd);
            for (j = 0; j < 16; ++j) put_code(codes, r, b * 16 + j, cols, cd[j]);
        }
    }
}

void oracle_quantize_1d(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                        int mode, uint64_t seed, const float *amax_in,
                        uint8_t *codes, uint8_t *sf, float *amax_out)
{
    float amax = amax_in ? *amax_in : oracle_amax_bf16(x, rows, cols, ld);
    memset(sf, 0, oracle_sf_bytes(rows, cols));
    quantize_rows(x, 0, rows, cols, ld, mode, seed, amax, codes, sf, 0);
    *amax_out = amax;
}

/* Padded scale-row offset of group g: sum over earlier groups of their row
 * count rounded up to 128 (each group's block scales start on a fresh atom). */
int64_t oracle_group_sf_row(const int64_t *offsets, int32_t g)
{
    int64_t po = 0;
    int32_t i;
    for (i = 0; i < g; ++i) po += ((offsets[i + 1] - offsets[i] + 127) / 128) * 128;
    return po;
}

size_t oracle_sf_bytes_grouped(int64_t rows, int64_t cols, int32_t groups)
{
    /* worst case: every group adds up to 127 padding rows */
    return oracle_sf_bytes(rows + 127 * (int64_t)groups, cols);
}

/* Grouped 1D quantisation (LatentMoE experts, [SL-2.2]): rows
 * offsets[g] .. offsets[g+1]-1 form group g with its own tensor scale
 * (reading: each expert is its own linear layer).  SR index e = r*cols+c
 * over the whole [rows, cols] output. */
void oracle_quantize_1d_grouped(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                                const int64_t *offsets, int32_t groups, int mode,
                                uint64_t seed, const float *amax_in,
                                uint8_t *codes, uint8_t *sf, float *amax_out)
{
    int32_t g;
    (void)rows;
    memset(sf, 0, oracle_sf_bytes_grouped(rows, cols, groups));
    for (g = 0; g < groups; ++g) {
        int64_t o = offsets[g], n = offsets[g + 1] - offsets[g];
        float amax = amax_in ? amax_in[g] : oracle_amax_bf16(x + o * ld, n, cols, ld);
        amax_out[g] = amax;
        if (n > 0)
            quantize_rows(x, o, n, cols, ld, mode, seed, amax, codes, sf,
                          oracle_group_sf_row(offsets, g));
    }
}

/* ------------------------------------------------------------------ */
/* 2D (16x16) quantisation of weights [S-infra], [U-2.2].               */
/* w: bf16 [batch][rows, cols], row stride ld, batch stride rows*ld;     */
/* rows % 16 == 0 and cols % 16 == 0.  One E4M3 scale per 16x16 tile, so */
/* W and W^T get identical codes.  Outputs per batch (each nullable      */
/* except codes/sf/amax_out):                                            */
/*   codes   [rows, cols/2],  sf   swizzled for [rows, cols] (tile scale  */
/*           repeated on each of the tile's rows);                       */
/*   codes_t [cols, rows/2],  sf_t swizzled for [cols, rows];            */
/*   tile_sf [rows/16, cols/16] row-major.                               */
/* Batch strides: codes rows*cols/2, sf oracle_sf_bytes(rows, cols),     */
/* sf_t oracle_sf_bytes(cols, rows), tile_sf rows*cols/256.              */
/* ------------------------------------------------------------------ */
void oracle_quantize_2d(const uint16_t *w, int64_t batch, int64_t rows, int64_t cols,
                        int64_t ld, const float *amax_in,
                        uint8_t *codes, uint8_t *sf, uint8_t *codes_t, uint8_t *sf_t,
                        uint8_t *tile_sf, float *amax_out)
{
    int64_t b;
    for (b = 0; b < batch; ++b) {
        const uint16_t *wb = w + b * rows * ld;
        uint8_t *cb = codes + b * rows * cols / 2;
        uint8_t *sb = sf + b * (int64_t)oracle_sf_bytes(rows, cols);
        uint8_t *ctb = codes_t ? codes_t + b * rows * cols / 2 : NULL;
        uint8_t *stb = sf_t ? sf_t + b * (int64_t)oracle_sf_bytes(cols, rows) : NULL;
        uint8_t *tb = tile_sf ? tile_sf + b * (rows / 16) * (cols / 16) : NULL;
        float amax = amax_in ? amax_in[b] : oracle_amax_bf16(wb, rows, cols, ld);
        float s_enc = oracle_tensor_scale(amax);
        int64_t t;
        amax_out[b] = amax;
        memset(sb, 0, oracle_sf_bytes(rows, cols));
        if (stb) memset(stb, 0, oracle_sf_bytes(cols, rows));
#pragma omp parallel for schedule(static)
        for (t = 0; t < (rows / 16) * (cols / 16); ++t) {
            int64_t ti = t / (cols / 16), tj = t % (cols / 16), i, j;
            float tile[16][16], bamax = 0.0f;
            uint8_t s, cd[16];
            for (i = 0; i < 16; ++i)
                for (j = 0; j < 16; ++j) {
                    tile[i][j] = bf16_to_float(wb[(ti * 16 + i) * ld + tj * 16 + j]);
                    if (fabsf(tile[i][j]) > bamax) bamax = fabsf(tile[i][j]);
                }
            s = oracle_block_scale(bamax, s_enc);
            if (tb) tb[ti * (cols / 16) + tj] = s;
            for (i = 0; i < 16; ++i) {
                int64_t n = ti * 16 + i;
                sb[oracle_sf_offset(n, tj, cols)] = s;
                encode_block(tile[i], 16, s_enc, s, 0, 0, 0, 0, cd);
                for (j = 0; j < 16; ++j) {
                    int64_t k = tj * 16 + j;
                    put_code(cb, n, k, cols, cd[j]);
                    if (ctb) put_code(ctb, k, n, rows, cd[j]);
                }
            }
            if (stb)
                for (j = 0; j < 16; ++j) stb[oracle_sf_offset(tj * 16 + j, ti, rows)] = s;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Random Hadamard transform [S-infra], [U-2.2] (R5).                   */
/* ------------------------------------------------------------------ */

/* y = 0.25 * H16 * (s .* x): negate x_j where bit j of sign_mask is set,
 * then the Sylvester butterfly with strides 1, 2, 4, 8 in FP32, then a
 * multiply by 0.25.  H16[i][j] = (-1)^popcount(i & j). */
void oracle_rht16(const float *in, uint16_t sign_mask, float *out)
{
    float x[16];
    int h, i;
    for (i = 0; i < 16; ++i) x[i] = ((sign_mask >> i) & 1) ? -in[i] : in[i];
    for (h = 1; h < 16; h <<= 1)
        for (i = 0; i < 16; ++i)
            if ((i & h) == 0) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
    for (i = 0; i < 16; ++i) out[i] = x[i] * 0.25f;
}

/* Amax of the RHT output of x (bf16 [tokens, cols], row stride ld). */
float oracle_rht_amax(const uint16_t *x, int64_t tokens, int64_t cols, int64_t ld,
                      uint16_t sign_mask)
{
    float a = 0.0f;
    int64_t c, t;
    for (c = 0; c < cols; ++c)
        for (t = 0; t < tokens; t += 16) {
            float in[16], y[16];
            int i;
            for (i = 0; i < 16; ++i) in[i] = bf16_to_float(x[(t + i) * ld + c]);
            oracle_rht16(in, sign_mask, y);
            for (i = 0; i < 16; ++i) if (fabsf(y[i]) > a) a = fabsf(y[i]);
        }
    return a;
}

/* RHT + 1D quantisation of a wgrad input.  x is bf16 [tokens, cols]
 * (tokens % 16 == 0); the transform runs over each 16-token chunk of each
 * column; the output is the TRANSPOSED operand [cols, tokens]: codes_t
 * [cols, tokens/2], sf_t swizzled for [cols, tokens].  The tensor scale
 * comes from the amax of the transformed values.  SR index e = c*tokens+t. */
void oracle_rht_quantize(const uint16_t *x, int64_t tokens, int64_t cols, int64_t ld,
                         uint16_t sign_mask, int mode, uint64_t seed,
                         const float *amax_in, uint8_t *codes_t, uint8_t *sf_t,
                         float *amax_out)
{
    float amax = amax_in ? *amax_in : oracle_rht_amax(x, tokens, cols, ld, sign_mask);
    float s_enc = oracle_tensor_scale(amax);
    int64_t c;
    memset(sf_t, 0, oracle_sf_bytes(cols, tokens));
#pragma omp parallel for schedule(static)
    for (c = 0; c < cols; ++c) {
        int64_t t;
        for (t = 0; t < tokens; t += 16) {
            float in[16], y[16], bamax = 0.0f;
            uint8_t s, cd[16];
            int i;
            for (i = 0; i < 16; ++i) in[i] = bf16_to_float(x[(t + i) * ld + c]);
            oracle_rht16(in, sign_mask, y);
            for (i = 0; i < 16; ++i) if (fabsf(y[i]) > bamax) bamax = fabsf(y[i]);
            s = oracle_block_scale(bamax, s_enc);
            sf_t[oracle_sf_offset(c, t / 16, tokens)] = s;
            encode_block(y, 16, s_enc, s, mode, seed, (uint64_t)(c * tokens + t), 1, cd);
            for (i = 0; i < 16; ++i) put_code(codes_t, c, t + i, tokens, cd[i]);
        }
    }
    *amax_out = amax;
}

/* Expert-segmented RHT quantisation for the wgrad of the LatentMoE
 * expert GEMMs ([SL-2.2] routed-expert GEMMs in NVFP4 in every pass; [U-2.2]
 * RHT on the wgrad inputs).  Reading R14: the pages do not say how an
 * expert's token segment meets the 16-token transform; here each expert's
 * segment of cnt_g tokens (rows offsets[g] .. offsets[g+1] of the
 * expert-sorted x [rows, cols]) is padded with zero tokens to
 * kp_g = ceil(cnt_g / 64) * 64 and placed at columns ko_g = sum_{i<g} kp_i
 * of the transposed operand [cols, kt] (kt >= ko_G; columns from ko_G on
 * are left as they are).  Padding to 64 rather than 16 puts every expert on
 * a boundary of the 128x4 scale atoms (64 tokens per atom column), so the
 * grouped wgrad GEMM can take one expert's K range as a plain K slice.
 * Each padded segment is transformed in 16-token chunks (R5) and quantised
 * in 1x16 blocks along tokens with its own tensor amax (the largest
 * magnitude of the segment's transformed values) or amax_in[g]; SR index
 * e = c * kt + ko_g + t. */
int64_t oracle_group_k_offset(const int64_t *offsets, int32_t g)
{
    int64_t k = 0;
    int32_t i;
    for (i = 0; i < g; ++i) k += (offsets[i + 1] - offsets[i] + 63) / 64 * 64;
    return k;
}

void oracle_rht_quantize_grouped(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                                 const int64_t *offsets, int32_t groups, int64_t kt,
                                 uint16_t sign_mask, int mode, uint64_t seed,
                                 const float *amax_in, uint8_t *codes_t, uint8_t *sf_t,
                                 float *amax_out)
{
    int32_t g;
    (void)rows;
    for (g = 0; g < groups; ++g) {
        const int64_t o0 = offsets[g], cnt = offsets[g + 1] - offsets[g];
        const int64_t kp = (cnt + 63) / 64 * 64, ko = oracle_group_k_offset(offsets, g);
        float amax = 0.0f, s_enc;
        int64_t c, t;
        /* the segment's transformed values, chunk by chunk; zero tokens past cnt */
        if (amax_in) {
            amax = amax_in[g];
        } else {
            for (c = 0; c < cols; ++c)
                for (t = 0; t < kp; t += 16) {
                    float in[16], y[16];
                    int i;
                    for (i = 0; i < 16; ++i)
                        in[i] = (t + i < cnt) ? bf16_to_float(x[(o0 + t + i) * ld + c]) : 0.0f;
                    oracle_rht16(in, sign_mask, y);
                    for (i = 0; i < 16; ++i) if (fabsf(y[i]) > amax) amax = fabsf(y[i]);
                }
        }
        amax_out[g] = amax;
        s_enc = oracle_tensor_scale(amax);
        for (c = 0; c < cols; ++c)
            for (t = 0; t < kp; t += 16) {
                float in[16], y[16], bamax = 0.0f;
                uint8_t sc, cd[16];
                int i;
                for (i = 0; i < 16; ++i)
                    in[i] = (t + i < cnt) ? bf16_to_float(x[(o0 + t + i) * ld + c]) : 0.0f;
                oracle_rht16(in, sign_mask, y);
                for (i = 0; i < 16; ++i) if (fabsf(y[i]) > bamax) bamax = fabsf(y[i]);
                sc = oracle_block_scale(bamax, s_enc);
                sf_t[oracle_sf_offset(c, (ko + t) / 16, kt)] = sc;
                encode_block(y, 16, s_enc, sc, mode, seed, (uint64_t)(c * kt + ko + t), 1, cd);
                for (i = 0; i < 16; ++i) put_code(codes_t, c, ko + t + i, kt, cd[i]);
            }
    }
}

/* ------------------------------------------------------------------ */
/* Dequantisation and the GEMM definition [S-infra].                    */
/* ------------------------------------------------------------------ */

/* x_hat = e2m1(code) * e4m3(sf) * dec, in FP64, for the listed rows of a
 * quantised [*, cols] tensor; the block scales of row r sit at scale row
 * sf_row0 + r.  out is [nrows, cols]. */
void oracle_dequantize_rows(const uint8_t *codes, const uint8_t *sf, int64_t sf_row0,
                            int64_t cols, float amax, const int64_t *row_idx,
                            int64_t nrows, double *out)
{
    double dec = (double)oracle_tensor_decode_scale(amax);
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t r = row_idx[i], k;
        for (k = 0; k < cols; ++k) {
            uint8_t byte = codes[r * (cols / 2) + k / 2];
            int code = (k & 1) ? (byte >> 4) : (byte & 15);
            double s = oracle_e4m3_value(sf[oracle_sf_offset(sf_row0 + r, k / 16, cols)]);
            out[i * cols + k] = oracle_e2m1_value(code) * s * dec;
        }
    }
}

/* ref[m][n] = sum_k A[m][k] * B[n][k] and bnd[m][n] = sum_k |A[m][k] * B[n][k]|,
 * both in FP64 over the dequantised operands (A [M,K], B [N,K]). */
void oracle_gemm(const double *A, const double *B, int64_t M, int64_t N, int64_t K,
                 double *ref, double *absum)
{
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        int64_t n, k;
        for (n = 0; n < N; ++n) {
            double s = 0.0, a = 0.0;
            for (k = 0; k < K; ++k) {
                double p = A[m * K + k] * B[n * K + k];
                s += p;
                a += fabs(p);
            }
            ref[m * N + n] = s;
            absum[m * N + n] = a;
        }
    }
}

/* ------------------------------------------------------------------ */
/* PTQ weight scales by minimum squared error ([SL-4.2]).                */
/* ------------------------------------------------------------------ */

/* Reading R16: [SL-4.2] calibrates the per-block weight scales of the NVFP4
 * PTQ checkpoint by minimising the weight MSE instead of taking them from
 * the block maximum.  Here: 1x16 blocks along the row, the tensor scale of
 * R1 from the tensor amax.  A block whose largest magnitude is 0 gets scale
 * 0 (R2).  Otherwise every finite positive E4M3 code c = 1 .. 126 is tried:
 * codes q_j = E2M1_RNE(x_j * (S_enc / e4m3(c))) (R3) and the FP32 error
 *     err_c = sum over j = 0 .. 15, in order, of d_j * d_j,
 *     d_j = x_j - value(q_j) * step_c,  step_c = e4m3(c) * dec  (dec of R1),
 * every product and sum one FP32 rounding; the block takes the c with the
 * smallest err_c, the largest such c on ties, and its codes. */
static uint8_t mse_block(const float *x, float s_enc, float dec, uint8_t *codes)
{
    float bamax = 0.0f, best = 0.0f;
    int j, c, bestc = 0;
    for (j = 0; j < 16; ++j) if (fabsf(x[j]) > bamax) bamax = fabsf(x[j]);
    if (bamax == 0.0f) { for (j = 0; j < 16; ++j) codes[j] = 0; return 0; }
    for (c = 1; c <= 126; ++c) {
        const float sc = (float)oracle_e4m3_value(c);
        const float r = element_multiplier(s_enc, sc);
        const float step = sc * dec;
        float err = 0.0f;
        for (j = 0; j < 16; ++j) {
            const int q = oracle_e2m1_rne(x[j] * r);
            const float rec = (float)oracle_e2m1_value(q) * step;
            const float d = x[j] - rec;
            const float d2 = d * d;
            err = err + d2;
        }
        if (bestc == 0 || err <= best) { best = err; bestc = c; }
    }
    {
        const float r = element_multiplier(s_enc, (float)oracle_e4m3_value(bestc));
        for (j = 0; j < 16; ++j) codes[j] = (uint8_t)oracle_e2m1_rne(x[j] * r);
    }
    return (uint8_t)bestc;
}

void oracle_quantize_1d_mse(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld,
                            const float *amax_in, uint8_t *codes, uint8_t *sf, float *amax_out)
{
    const float amax = amax_in ? *amax_in : oracle_amax_bf16(x, rows, cols, ld);
    const float s_enc = oracle_tensor_scale(amax), dec = oracle_tensor_decode_scale(amax);
    int64_t r;
    memset(sf, 0, oracle_sf_bytes(rows, cols));
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t b;
        for (b = 0; b < cols / 16; ++b) {
            float blk[16];
            uint8_t cd[16];
            int j;
            for (j = 0; j < 16; ++j) blk[j] = bf16_to_float(x[r * ld + b * 16 + j]);
            sf[oracle_sf_offset(r, b, cols)] = mse_block(blk, s_enc, dec, cd);
            for (j = 0; j < 16; ++j) put_code(codes, r, b * 16 + j, cols, cd[j]);
        }
    }
    *amax_out = amax;
}

/* ------------------------------------------------------------------ */
/* FP16 stochastic rounding for the SSM cache ([SL-4.3]).                */
/* ------------------------------------------------------------------ */

/* Reading R15: [SL-4.3] keeps the Mamba SSM cache in FP16 with stochastic
 * rounding driven by Philox with 5 rounds and gives no further rule.  Here,
 * for a finite x with m = |x| < 65504: lo = the largest FP16 magnitude <= m,
 * hi = the next FP16 magnitude, p = (m - lo) / (hi - lo) (exact in FP64);
 * the magnitude becomes hi iff u < 256 * ceil(p * 2^24) (the resolution of
 * R4), u = the R4 word of element e; the sign is kept (so -0 stays -0).
 * m >= 65504 (and infinities) saturate to 65504; NaN becomes the FP16
 * quiet NaN 0x7E00 with the sign of x. */
static double fp16_spacing(double m)
{
    int e;
    if (m < ldexp(1.0, -14)) return ldexp(1.0, -24);
    frexp(m, &e);                                    /* m = f * 2^e, f in [0.5, 1) */
    return ldexp(1.0, e - 1 - 10);
}

static uint16_t fp16_bits_of(double v)               /* v: an FP16 magnitude <= 65504 */
{
    int e;
    if (v < ldexp(1.0, -14)) return (uint16_t)(v * ldexp(1.0, 24));
    frexp(v, &e);
    return (uint16_t)(((e - 1 + 15) << 10) | (uint16_t)((v / ldexp(1.0, e - 1) - 1.0) * 1024.0));
}

uint16_t oracle_fp16_sr(float x, uint32_t u)
{
    uint32_t bits;
    uint16_t sign;
    double m, sp, lo, p, c;
    memcpy(&bits, &x, 4);
    sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    m = fabs((double)x);
    if (m >= 65504.0) return (uint16_t)(sign | 0x7BFFu);
    sp = fp16_spacing(m);
    lo = floor(m / sp) * sp;
    p = (m - lo) / sp;
    c = ceil(p * 16777216.0);
    if ((double)u < 256.0 * c) lo += sp;
    return (uint16_t)(sign | fp16_bits_of(lo));
}

/* out[e] = SR of x[e] to FP16 with the R4 word of index e under seed. */
void oracle_sr_fp16(const float *x, int64_t n, uint64_t seed, uint16_t *out)
{
    int64_t e;
#pragma omp parallel for schedule(static)
    for (e = 0; e < n; ++e) out[e] = oracle_fp16_sr(x[e], oracle_sr_word(seed, (uint64_t)e));
}

/* Number of threads the parallel loops above use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
