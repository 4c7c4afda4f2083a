/*
 * nvfp4.h -- C ABI of libnvfp4.so: NVFP4 training linear layers on one
 * B300 (sm_103a).
 *
 * The method (web pages summarising the Nemotron 3 Super / Ultra technical
 * reports):
 *   - "Nemotron 3 Super -- technical report summary" (gkm0120.cn), section 1,
 *     pre-training table, row "training precision": NVFP4 = E2M1 elements in
 *     16-element micro-blocks with E4M3 scaling.
 *   - same page, "Infra design" table: NVFP4 GEMMs for fprop, dgrad and wgrad;
 *     2D block scaling for weights, 1D block scaling for activations and
 *     gradients; random Hadamard transforms plus stochastic rounding.
 *   - "Nemotron 3 Ultra: Open, Efficient Mixture-of-Experts Hybrid
 *     Mamba-Transformer Model for Agentic Reasoning" (papercache.org
 *     translation), section 2.2: 2D block quantisation of weights, the RHT
 *     on the inputs of wgrad, SR on gradients.
 *   - "Nemotron 3 Super" summary (papers.lianghsun.dev), section 2.2: the
 *     MoE routed-expert GEMMs run in NVFP4.
 *
 * Numerics (the pages give the format, not the formulas; these readings are
 * fixed here and every entry point follows them bit for bit):
 *   tensor scale  S_enc = 2688 / amax in FP32 (1 if amax == 0, FLT_MAX if the
 *                 quotient overflows); decode scale dec = 1 / S_enc.
 *   block scale   sf = E4M3(round-nearest-even, saturating at 448) of
 *                 (bamax / 6) * S_enc, computed as two FP32 operations.
 *   element       sf == 0 gives code +0; otherwise v = x * (S_enc / sf) in
 *                 FP32, rounded to E2M1 {0,.5,1,1.5,2,3,4,6} (nearest-even,
 *                 saturating at 6) or stochastically (below); the sign bit
 *                 is copied from x.
 *   SR            element e (row-major index in the quantised output) draws
 *                 word e & 3 of Philox4x32 with 5 rounds, key = seed,
 *                 counter = (e >> 2 as two 32-bit halves, 0, 0); with grid
 *                 neighbours lo <= |v| < hi and p = (|v|-lo)/(hi-lo), the
 *                 magnitude rounds up iff (word >> 8) < p * 2^24.
 *   RHT           per column, per 16 consecutive rows: y = 0.25 * H16 * (s .* x),
 *                 s_j = -1 where bit j of sign_mask is set, H16 the Sylvester
 *                 Hadamard matrix, evaluated as the FP32 butterfly with strides
 *                 1, 2, 4, 8.
 *
 * Layouts:
 *   codes  uint8 [rows, cols/2], rows cols/2 bytes apart; element 2j of a
 *          row is the low nibble of byte j, element 2j+1 the high nibble;
 *          nibble = sign << 3 | E2M1 magnitude index.
 *   sf     block scale (r, c) of a [rows, cols] operand (c < cols/16) sits at
 *          byte ((r/128) * ceil(cols/64) + c/4) * 512
 *               + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *          i.e. 128x4 atoms of 512 bytes, rows padded to 128 and scale
 *          columns to 4; padding bytes are written as 0 by the quantisers.
 *          nvfp4_sf_bytes() gives the size.
 *   grouped operands: group g's rows are offsets[g] .. offsets[g+1]-1 of the
 *          codes, and its block scales start at scale row
 *          P_g = sum_{i<g} ceil((offsets[i+1]-offsets[i]) / 128) * 128.
 *   batched 2D weights: entry b of a [batch, rows, cols] weight owns codes
 *          bytes [b*rows*cols/2, ...) and sf bytes
 *          [b*nvfp4_sf_bytes(rows, cols), ...).
 *
 * Ownership and errors:
 *   The caller allocates every device buffer and owns the stream; the
 *   library allocates no device memory.  Every call validates its
 *   arguments on the host before launching anything and returns a status;
 *   work is enqueued asynchronously on `stream` (NULL = legacy default
 *   stream).  Launch failures return NVFP4_ERR_CUDA with the CUDA message in
 *   nvfp4_last_error().  Values that live in device memory (group offsets)
 *   cannot be checked on the host: kernels clamp them into range and record
 *   NVFP4_DEV_* codes in a device status word read by nvfp4_device_status().
 *   Bounded waits inside kernels that give up record NVFP4_DEV_TIMEOUT there
 *   and return instead of hanging.
 *   All device pointers must be 16-byte aligned; all leading dimensions are
 *   in elements and must make every row start 16-byte aligned.
 *
 * State kept by the library (all calls may come from any host thread):
 *   a per-thread last-error string; a per-device cache of the device check
 *   and kernel attributes (guarded by a mutex); a launch counter and a
 *   one-shot failure-injection hook (atomics); in device memory, the status
 *   word and the counters of nvfp4_quantize_2d_fused_static.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *nvfp4_stream_t;

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_NULL = 1,        /* a required pointer is NULL */
    NVFP4_ERR_SHAPE = 2,       /* negative size, dimension not a multiple of 16 (32 for GEMM K), mismatch */
    NVFP4_ERR_ALIGN = 3,       /* pointer or leading dimension breaks 16-byte alignment */
    NVFP4_ERR_DEVICE = 4,      /* no CUDA device or not compute capability 10.3 */
    NVFP4_ERR_CUDA = 5,        /* a CUDA call failed; see nvfp4_last_error() */
    NVFP4_ERR_TIMEOUT = 6,     /* a kernel abandoned a bounded wait */
    NVFP4_ERR_LIMIT = 7        /* a size is beyond a documented limit */
} nvfp4_status;

typedef enum { NVFP4_ROUND_RNE = 0, NVFP4_ROUND_SR = 1 } nvfp4_round;
typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_FP32 = 1 } nvfp4_out_dtype;

/* Device status word codes (bit flags, sticky until read). */
#define NVFP4_DEV_TIMEOUT     1
#define NVFP4_DEV_BAD_OFFSETS 2

/* Largest group count of the grouped calls. */
#define NVFP4_MAX_GROUPS 1024

/* A quantised operand.  cols is the reduction (K) dimension. */
typedef struct {
    void    *codes;    /* device, uint8 [rows, cols/2] */
    uint8_t *sf;       /* device, swizzled E4M3 block scales */
    float   *amax;     /* device, FP32 amax: 1 value, or 1 per group / batch entry */
    int64_t  rows;
    int64_t  cols;
} nvfp4_tensor;

/* ------------------------------------------------------------- layout */

/* Bytes of the swizzled block-scale buffer of a [rows, cols] operand. */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);

/* Upper bound of the block-scale bytes of a grouped [rows, cols] operand with
 * num_groups groups (each group may add up to 127 padding rows). */
size_t nvfp4_sf_bytes_grouped(int64_t rows, int64_t cols, int32_t num_groups);

/* Byte offset of block scale (r, c) inside the swizzled buffer. */
int64_t nvfp4_sf_offset(int64_t r, int64_t c, int64_t cols);

/* ------------------------------------------------------------- amax */

/* amax[b] = max |x| over entry b of a bf16 [batch, rows, cols] tensor with
 * row stride ld (entries rows*ld elements apart).  amax: device, batch floats,
 * overwritten.  Inputs must be finite.  (Per-tensor FP32 scale of the
 * recipe; the max-based scaling of "Nemotron 3 Super" summary,
 * papers.lianghsun.dev, section 4.2.) */
nvfp4_status nvfp4_amax(const void *x, int64_t batch, int64_t rows, int64_t cols,
                        int64_t ld, float *amax, nvfp4_stream_t stream);

/* ------------------------------------------------------------- quantisers */

/* 1D (1x16) quantisation of activations (RNE) or gradients (SR) -- "Infra
 * design" table of the Super summary; SR of gradients, Ultra report 2.2.
 * x: bf16 [rows, cols], row stride ld; cols % 16 == 0.
 * out: codes, sf (nvfp4_sf_bytes(rows, cols)), amax (1 float), rows, cols
 * must equal the arguments.  amax_in (device, nullable): when given, its
 * value is the tensor amax (and is copied to out->amax); otherwise the
 * amax is computed first (an extra read of x).  seed is used only for SR. */
nvfp4_status nvfp4_quantize_1d(const void *x, int64_t rows, int64_t cols, int64_t ld,
                               nvfp4_round mode, uint64_t seed, const float *amax_in,
                               nvfp4_tensor *out, nvfp4_stream_t stream);

/* Grouped 1D quantisation of expert-sorted activations (LatentMoE routed
 * experts in NVFP4, Super summary papers.lianghsun.dev 2.2): group g is rows
 * offsets[g] .. offsets[g+1]-1 and has its own tensor amax (out->amax[g]).
 * offsets: device int64 [num_groups+1], non-decreasing, offsets[0] == 0,
 * offsets[num_groups] <= rows; empty groups allowed.  out->sf must hold
 * nvfp4_sf_bytes_grouped(rows, cols, num_groups) bytes; block scales of
 * group g start at scale row P_g (see Layouts).  SR index e = r*cols + c
 * over the whole output.  amax_in: device, num_groups floats, nullable.
 * 1 <= num_groups <= NVFP4_MAX_GROUPS. */
nvfp4_status nvfp4_quantize_1d_grouped(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                       const int64_t *offsets, int32_t num_groups,
                                       nvfp4_round mode, uint64_t seed, const float *amax_in,
                                       nvfp4_tensor *out, nvfp4_stream_t stream);

/* 2D (16x16) quantisation of weights, so that W and W^T quantise
 * identically (Super summary "Infra design"; Ultra report 2.2).
 * w: bf16 [batch, rows, cols], row stride ld, entry stride rows*ld;
 * rows % 16 == 0, cols % 16 == 0.  Always RNE.
 * out   (required): codes [batch][rows, cols/2], sf per entry
 *       nvfp4_sf_bytes(rows, cols) with each tile's scale on every one of its
 *       16 rows (GEMM-ready), amax[batch]; out->rows == rows, out->cols == cols.
 * out_t (nullable): the transposed operand W^T -- codes [batch][cols, rows/2],
 *       sf per entry nvfp4_sf_bytes(cols, rows); amax may be NULL (the
 *       amax lives in out->amax); out_t->rows == cols, out_t->cols == rows.
 * tile_sf (nullable): device uint8 [batch][rows/16, cols/16] row-major.
 * amax_in: device, batch floats, nullable. */
nvfp4_status nvfp4_quantize_2d(const void *w, int64_t batch, int64_t rows, int64_t cols,
                               int64_t ld, const float *amax_in, nvfp4_tensor *out,
                               nvfp4_tensor *out_t, uint8_t *tile_sf, nvfp4_stream_t stream);

/* Bytes of device workspace nvfp4_quantize_2d_fused needs for `batch`
 * entries (16-byte multiple). */
size_t nvfp4_quantize_2d_fused_workspace(int64_t batch);

/* The same W result as nvfp4_quantize_2d with amax_in == NULL and out_t ==
 * NULL (per-entry amax, W codes and GEMM-ready scales, optional tile scales)
 * for batched weights such as the LatentMoE expert weights (2D block scaling
 * of weights, Super summary "Infra design"), in one cooperative launch that
 * reads each element once from HBM.  When an entry has at most 18 units of
 * 16 x 256 elements per SM (5120 x 2048 on 148 SMs), every CTA keeps its share
 * of the entry on chip (TMA into shared memory, then registers) while the
 * entry's amax is exchanged through the workspace, and then encodes it;
 * larger entries are read a second time within a short window so that the
 * second read can hit L2.  Either way the entries are processed one after
 * another with one grid-wide exchange each, and for the LatentMoE expert
 * weights on B300 the two-launch nvfp4_quantize_2d (amax, then quantise) is
 * still faster, so this entry point is an alternative, not the default.
 * Requires w 16-byte aligned with ld % 8 == 0.  The transposed copy is not
 * produced (use nvfp4_quantize_2d for W^T).
 * workspace: device, caller-allocated, at least
 * nvfp4_quantize_2d_fused_workspace(batch) bytes, 16-byte aligned; the call
 * zeroes and uses it (per-entry arrival counters), so calls sharing one
 * workspace must not overlap on the GPU.  out->amax receives the amaxes.
 * Other arguments as for nvfp4_quantize_2d. */
nvfp4_status nvfp4_quantize_2d_fused(const void *w, int64_t batch, int64_t rows, int64_t cols, int64_t ld,
                                     void *workspace, size_t workspace_bytes, nvfp4_tensor *out,
                                     uint8_t *tile_sf, nvfp4_stream_t stream);

/* Largest batch of nvfp4_quantize_2d_fused_static. */
#define NVFP4_STATIC_MAX_BATCH 4096

/* nvfp4_quantize_2d_fused without a caller workspace, for callers that cannot
 * allocate device memory at the point of the call: code whose device memory
 * is owned by another allocator that has no workspace to lend, or a loop that
 * must not call cudaMalloc (it can synchronise the device and take locks).
 * The per-entry counters live in a fixed array inside the library
 * ((NVFP4_STATIC_MAX_BATCH + 8) * 4 bytes, held by every GPU that loads the
 * library until the process exits); the call allocates nothing.
 * batch > NVFP4_STATIC_MAX_BATCH returns NVFP4_ERR_LIMIT.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.
 * Every call zeroes and reuses the same array, so two calls that overlap on
 * the GPU (other streams, other host threads) race and corrupt each other.
 * Other arguments and results as for nvfp4_quantize_2d_fused.  The pages
 * have no counterpart of this entry point: it only changes where scratch
 * memory comes from. */
nvfp4_status nvfp4_quantize_2d_fused_static(const void *w, int64_t batch, int64_t rows, int64_t cols, int64_t ld,
                                            nvfp4_tensor *out, uint8_t *tile_sf, nvfp4_stream_t stream);

/* amax of the RHT output of x (bf16 [tokens, cols], row stride ld,
 * tokens % 16 == 0) -> amax (device, 1 float). */
nvfp4_status nvfp4_rht_amax(const void *x, int64_t tokens, int64_t cols, int64_t ld,
                            uint16_t sign_mask, float *amax, nvfp4_stream_t stream);

/* Both tensor amaxes of a gradient in one read: amax_plain = max |x| (the
 * 1x16 SR quantiser of dgrad) and amax_rht = max |RHT(x)| along tokens (the
 * RHT quantiser of wgrad), x: bf16 [tokens, cols], tokens % 16 == 0.  Each
 * result is the one nvfp4_amax / nvfp4_rht_amax would give; pass them as
 * amax_in.  amax_plain, amax_rht: device, 1 float each, zeroed by the call. */
nvfp4_status nvfp4_dual_amax(const void *x, int64_t tokens, int64_t cols, int64_t ld, uint16_t sign_mask,
                             float *amax_plain, float *amax_rht, nvfp4_stream_t stream);

/* Both stochastically rounded operands of a gradient dY from one read of it
 * (Super summary "Infra design": stochastic rounding of gradients, RHT on
 * the inputs of wgrad; Ultra report 2.2): out_row receives exactly what
 * nvfp4_quantize_1d(dy, NVFP4_ROUND_SR, seed_row, amax_row) gives (the dgrad
 * operand [tokens, cols]) and out_t exactly what nvfp4_rht_quantize(dy,
 * sign_mask, NVFP4_ROUND_SR, seed_rht, amax_rht) gives (the wgrad operand
 * [cols, tokens]); both are encoded from the same staged tile of dY.
 * amax_row, amax_rht: device, 1 float each (nvfp4_dual_amax gives both),
 * copied into out_row->amax and out_t->amax.  zero_count (device, one 64-bit
 * word, nullable): receives the number of zero-magnitude codes of out_row,
 * what nvfp4_count_zero_codes(out_row) would count (zeroed by the call).
 * dy: bf16 [tokens, cols], row stride ld, tokens % 16 == 0, cols % 16 == 0. */
nvfp4_status nvfp4_dual_sr_quantize(const void *dy, int64_t tokens, int64_t cols, int64_t ld, uint16_t sign_mask,
                                    uint64_t seed_row, uint64_t seed_rht, const float *amax_row,
                                    const float *amax_rht, nvfp4_tensor *out_row, nvfp4_tensor *out_t,
                                    uint64_t *zero_count, nvfp4_stream_t stream);

/* Number of E2M1 codes of magnitude zero (+0 and -0) in a quantised tensor
 * (rows * cols codes): the zero-gradient fraction the pages monitor (Super
 * summary "Infra design"; section 2.2: small gradients underflow to zero).
 * count: device, one 64-bit word, zeroed by the call.  codes 16-byte aligned. */
nvfp4_status nvfp4_count_zero_codes(const nvfp4_tensor *t, uint64_t *count, nvfp4_stream_t stream);

/* RHT + 1D quantisation of a wgrad input (Super summary "Infra design";
 * Ultra report 2.2: RHT on the inputs of wgrad).  x: bf16 [tokens, cols],
 * row stride ld, tokens % 16 == 0.  The transform runs along tokens (the
 * wgrad K axis); the result is the TRANSPOSED operand out_t: codes
 * [cols, tokens/2], sf nvfp4_sf_bytes(cols, tokens), amax (1 float) of the
 * transformed values; out_t->rows == cols, out_t->cols == tokens.
 * Use the same sign_mask for both operands of one wgrad GEMM.
 * SR index e = c*tokens + t.  amax_in: device, nullable. */
nvfp4_status nvfp4_rht_quantize(const void *x, int64_t tokens, int64_t cols, int64_t ld,
                                uint16_t sign_mask, nvfp4_round mode, uint64_t seed,
                                const float *amax_in, nvfp4_tensor *out_t,
                                nvfp4_stream_t stream);

/* 1x16 quantisation with block scales calibrated by minimum squared error:
 * the weight scales of the NVFP4 PTQ checkpoint (Super summary section 4.2:
 * per-block weight scales chosen to minimise the weight MSE rather than from
 * the block maximum).  x: bf16 [rows, cols] (cols % 16 == 0, row stride
 * ld % 8 == 0, 16-byte aligned); out as for nvfp4_quantize_1d (RNE codes,
 * GEMM-ready scales, amax).
 * The tensor scale is the usual 2688 / amax (amax computed, or amax_in).  A
 * block whose largest magnitude is 0 gets scale 0; otherwise every finite
 * positive E4M3 scale is tried and the block keeps the one with the smallest
 * FP32 squared error sum_j (x_j - value(q_j) * e4m3(c) * dec)^2 (summed in
 * element order; the larger scale on ties).  Offline work: 126 trial
 * encodings per block. */
nvfp4_status nvfp4_quantize_1d_mse(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                   const float *amax_in, nvfp4_tensor *out, nvfp4_stream_t stream);

/* FP32 -> FP16 with stochastic rounding: the Mamba SSM-cache recipe of the
 * Super summary (section 4.3: FP16 cache, stochastic rounding driven by
 * Philox with 5 rounds).  x: device FP32 [n] (4-byte aligned); out: device
 * FP16 bits [n] (2-byte aligned).  For m = |x[e]| < 65504 with FP16
 * neighbours lo <= m < hi, the magnitude becomes hi iff u < 256 * ceil(p *
 * 2^24), p = (m - lo) / (hi - lo), u = word e & 3 of Philox4x32-5 with key
 * seed and counter (e >> 2, 0, 0) (the same words as the SR quantisers);
 * m >= 65504 and infinities saturate to 65504, NaN becomes 0x7E00, the sign
 * is kept.  Not part of the NVFP4 recipe itself: a second user of its SR. */
nvfp4_status nvfp4_sr_fp16(const float *x, int64_t n, uint64_t seed, uint16_t *out, nvfp4_stream_t stream);

/* Columns needed by nvfp4_rht_quantize_grouped for `rows` expert-sorted
 * tokens in `groups` experts, whatever the split: ceil((rows + 63 * groups)
 * / 64) * 64 (every expert's segment is padded to a multiple of 64). */
int64_t nvfp4_group_k_capacity(int64_t rows, int32_t groups);

/* Expert-segmented RHT + 1D quantisation: the wgrad inputs of the LatentMoE
 * expert GEMMs (Super summary section 2.2: routed-expert GEMMs in NVFP4;
 * Ultra report 2.2: RHT on the inputs of wgrad).  x: bf16 [rows, cols],
 * rows sorted by expert, expert g owning rows offsets[g] .. offsets[g+1]
 * (device, num_groups + 1 values).  Expert g's segment is padded with zero
 * tokens to kp_g = ceil(cnt_g / 64) * 64 and written at columns ko_g =
 * sum_{i<g} kp_i of the transposed operand out_t ([cols, kt]: codes
 * [cols, kt/2], sf nvfp4_sf_bytes(cols, kt), amax num_groups floats); the
 * pages do not say how a segment meets the 16-token transform, 64 puts every
 * expert on a scale-atom boundary.  Each segment is transformed in 16-token
 * chunks and quantised with its own amax (computed, or amax_in[g]); SR index
 * e = c * kt + ko_g + t.  kt: a multiple of 64, at least
 * nvfp4_group_k_capacity(rows, num_groups); columns past the last segment
 * are not written.  Use the same sign_mask for both operands of a wgrad. */
nvfp4_status nvfp4_rht_quantize_grouped(const void *x, int64_t rows, int64_t cols, int64_t ld,
                                        const int64_t *offsets, int32_t num_groups, int64_t kt,
                                        uint16_t sign_mask, nvfp4_round mode, uint64_t seed,
                                        const float *amax_in, nvfp4_tensor *out_t, nvfp4_stream_t stream);

/* ------------------------------------------------------------- GEMMs */

/* C[m, n] = alpha * sum_k a_k * sa * b_k * sb with FP32 accumulation, where
 * alpha = dec(a->amax) * dec(b->amax) in FP32 -- the fprop / dgrad / wgrad
 * NVFP4 GEMMs (Super summary "Infra design"; Ultra report 2.2).
 * a: [M, K], b: [N, K] (both K-major, a->cols == b->cols == K, K % 16 == 0,
 * the 16-element micro-block of the recipe; K % 16 != 0 returns
 * NVFP4_ERR_SHAPE).  When K % 32 == 16 the K/2-byte code rows are not the
 * 16-byte multiple a TMA tensor map needs: the kernel then copies the code
 * rows into shared memory itself, on single CTAs.  c: device [M, N], row stride
 * ldc elements, bf16 (one RNE rounding of the FP32 result) or FP32.
 * M, N >= 1 arbitrary.  c_amax (device, 1 float, nullable): receives
 * max |c| over the written outputs (of the stored bf16 values for a bf16 c),
 * the tensor amax a following quantisation of c can take as amax_in instead
 * of reading c again; it is zeroed by the call (left untouched when M or N
 * is 0).
 * Kernel: pairs of CTAs on two SMs (tcgen05 cta_group::2, 256 x 256 tiles)
 * unless the environment variable NVFP4_GEMM_PAIR is "0" at the call, which
 * selects single CTAs (128 x 256 tiles); both give the same bits.  The same
 * holds for nvfp4_grouped_gemm. */
nvfp4_status nvfp4_gemm(const nvfp4_tensor *a, const nvfp4_tensor *b, void *c, int64_t ldc,
                        nvfp4_out_dtype c_dtype, float *c_amax, nvfp4_stream_t stream);

/* Grouped GEMM of the LatentMoE routed experts: for every group g,
 * C[offsets[g] .. offsets[g+1]-1, :] = alpha_g * A_g * W_g^T with
 * alpha_g = dec(a->amax[g]) * dec(b->amax[g]).  a: grouped operand from
 * nvfp4_quantize_1d_grouped ([R, K], K % 16 == 0, as for nvfp4_gemm).  b: batched operand from
 * nvfp4_quantize_2d with batch == num_groups, b->rows == n per expert,
 * b->cols == K.  offsets: device int64 [num_groups+1] as for the grouped
 * quantiser.  Rows of C outside [offsets[0], offsets[num_groups]) are not
 * written.  c: bf16 or FP32 [R, n], row stride ldc.  c_amax (device,
 * num_groups floats, nullable): per-group max |c| over the written outputs
 * (the amax_in of a following grouped quantisation of c), zeroed by the
 * call. */
nvfp4_status nvfp4_grouped_gemm(const nvfp4_tensor *a, const int64_t *offsets, int32_t num_groups,
                                const nvfp4_tensor *b, int64_t n, void *c, int64_t ldc,
                                nvfp4_out_dtype c_dtype, float *c_amax, nvfp4_stream_t stream);

/* ------------------------------------------------------------- status */

/* GEMM whose groups split K: the wgrad of the LatentMoE expert GEMMs,
 * dW_g = dH_g^T . A_g over expert g's tokens (Super summary section 2.2:
 * routed-expert GEMMs in NVFP4; Ultra report 2.2: wgrad on RHT operands).
 * a: [M, KT] and b: [N, KT], both from nvfp4_rht_quantize_grouped with the
 * same offsets and sign mask (amax: num_groups floats each); KT % 64 == 0.
 * offsets: device, num_groups + 1 token offsets; group g's K slice is
 * columns ko_g .. ko_g + ceil(cnt_g / 64) * 64 (nvfp4_rht_quantize_grouped).
 * c: [num_groups * M, N], row stride ldc; rows g*M .. g*M + M - 1 receive
 * C_g = alpha_g * A[:, slice_g] . B[:, slice_g]^T, alpha_g =
 * dec(a->amax[g]) * dec(b->amax[g]); an expert without tokens gets zeros.
 * c_amax: nullable, num_groups floats, as for nvfp4_grouped_gemm. */
nvfp4_status nvfp4_grouped_gemm_k(const nvfp4_tensor *a, const nvfp4_tensor *b, const int64_t *offsets,
                                  int32_t num_groups, void *c, int64_t ldc, nvfp4_out_dtype c_dtype,
                                  float *c_amax, nvfp4_stream_t stream);

const char *nvfp4_status_string(nvfp4_status status);

/* Message of the last failed call on this host thread ("" if none). */
const char *nvfp4_last_error(void);

/* Synchronises the current device, returns the device status word
 * (NVFP4_DEV_* bit flags, 0 if clean) in *flags and clears it.  Returns
 * NVFP4_ERR_TIMEOUT if NVFP4_DEV_TIMEOUT was set, NVFP4_OK otherwise. */
nvfp4_status nvfp4_device_status(int32_t *flags);

/* Number of kernels this library has launched in this process (diagnostic;
 * counts every successful launch of every entry point). */
uint64_t nvfp4_launch_count(void);

/* Test hook: the next call to any entry point above returns `status`
 * without launching (NVFP4_OK clears the hook).  Host-side only. */
void nvfp4_debug_inject(nvfp4_status status);

/* Test hook: launches one block that waits on a barrier nothing will
 * complete, giving up after timeout_ns nanoseconds; the give-up is recorded
 * as NVFP4_DEV_TIMEOUT in the device status word. */
nvfp4_status nvfp4_debug_wait_timeout(int64_t timeout_ns, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H */
