// nvfp4.cu -- the C ABI of libnvfp4.so (declared in include/nvfp4.h).
//
// Host side only validates arguments, builds TMA tensor maps and launches the
// kernels of quant.cuh and gemm.cuh on the caller's stream.  It allocates no
// device memory.
#include <cuda.h>
#include <cstdlib>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "nvfp4.h"
#include "common.cuh"
#include "quant.cuh"
#include "gemm.cuh"
#include "quant2d_resident.cuh"
#include "quant2d_w.cuh"

using namespace nvfp4;

namespace {

thread_local char g_last_error[512] = "";
std::atomic<int> g_inject{0};
std::atomic<uint64_t> g_launches{0};

nvfp4_status fail(nvfp4_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

#define NVFP4_INJECT_CHECK()                                                              \
    do {                                                                                  \
        const int inj = g_inject.exchange(0);                                             \
        if (inj != 0) return fail((nvfp4_status)inj, "injected failure (test hook)");     \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device ordinals this library serves: per-device tables below are indexed by
// the ordinal, and check_device() refuses ordinals at or above the bound.
constexpr int MAX_DEVICES = 64;

struct DeviceInfo {
    bool checked = false;
    bool ok = false;
    int sms = 0;
    bool gemm_attr = false;
    int pair_clusters = 0;
    bool q2r_attr = false;
    bool rht_attr = false;
};
DeviceInfo g_dev[MAX_DEVICES];
std::mutex g_dev_mu;

// Current device must be compute capability 10.3 (B300, sm_103a).
nvfp4_status check_device(int* sms = nullptr, int* dev_out = nullptr) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return fail(NVFP4_ERR_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.checked) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(NVFP4_ERR_DEVICE, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
        }
        d.ok = (prop.major == 10 && prop.minor == 3);
        d.sms = prop.multiProcessorCount;
        d.checked = true;
        if (!d.ok) return fail(NVFP4_ERR_DEVICE, "device %d is sm_%d%d, this library is built for sm_103a", dev, prop.major, prop.minor);
    }
    if (!d.ok) return fail(NVFP4_ERR_DEVICE, "device %d is not sm_103", dev);
    if (sms) *sms = d.sms;
    if (dev_out) *dev_out = dev;
    return NVFP4_OK;
}

nvfp4_status launched(const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return NVFP4_OK;
}

nvfp4_status cuda_call(cudaError_t e, const char* what) {
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(NVFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    }
    return NVFP4_OK;
}

#define NVFP4_TRY(expr)                           \
    do {                                          \
        const nvfp4_status st_ = (expr);          \
        if (st_ != NVFP4_OK) return st_;          \
    } while (0)

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shared checks of a bf16 input [rows, cols] with row stride ld.
// vec_rows: the kernel reads rows with 16-byte vectors (ld % 8 == 0 and a
// 16-byte aligned base); otherwise 2-byte alignment suffices.
nvfp4_status check_input(const void* x, int64_t rows, int64_t cols, int64_t ld, int64_t mult, const char* name,
                         bool vec_rows = true) {
    if (x == nullptr && rows > 0) return fail(NVFP4_ERR_NULL, "%s is NULL", name);
    if (rows < 0 || cols < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative size", name);
    if (cols % mult != 0) return fail(NVFP4_ERR_SHAPE, "%s: cols=%lld is not a multiple of %lld", name, (long long)cols, (long long)mult);
    if (ld < cols) return fail(NVFP4_ERR_SHAPE, "%s: ld=%lld < cols=%lld", name, (long long)ld, (long long)cols);
    if (vec_rows && (ld % 8 != 0 || !aligned16(x)))
        return fail(NVFP4_ERR_ALIGN, "%s: rows must start 16-byte aligned (ld %% 8 == 0, aligned base)", name);
    if (!vec_rows && ((uintptr_t)x & 1u)) return fail(NVFP4_ERR_ALIGN, "%s: not 2-byte aligned", name);
    if ((rows * cols) / 8 >= (int64_t(1) << 32)) return fail(NVFP4_ERR_LIMIT, "%s: more than 2^35 elements", name);
    return NVFP4_OK;
}

nvfp4_status check_out(const nvfp4_tensor* t, int64_t rows, int64_t cols, bool need_amax, const char* name) {
    if (t == nullptr) return fail(NVFP4_ERR_NULL, "%s is NULL", name);
    if (t->rows != rows || t->cols != cols)
        return fail(NVFP4_ERR_SHAPE, "%s: shape [%lld, %lld] != expected [%lld, %lld]", name, (long long)t->rows,
                    (long long)t->cols, (long long)rows, (long long)cols);
    if (rows > 0 && (t->codes == nullptr || t->sf == nullptr)) return fail(NVFP4_ERR_NULL, "%s: codes/sf NULL", name);
    if (need_amax && t->amax == nullptr) return fail(NVFP4_ERR_NULL, "%s: amax NULL", name);
    if (!aligned16(t->codes) || !aligned16(t->sf)) return fail(NVFP4_ERR_ALIGN, "%s: codes/sf not 16-byte aligned", name);
    return NVFP4_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

// 2D uint8 tensor map over packed codes [rows, row_bytes] with a box of
// {128 bytes, box_rows} and 128-byte swizzle (the tcgen05 K-major layout).
nvfp4_status make_code_map(CUtensorMap* map, const void* codes, int64_t rows, int64_t row_bytes, int box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return NVFP4_OK;
}

int quant_blocks(int64_t rows, int sms) {
    const int64_t b = cdiv(rows, 8);
    return (int)std::max<int64_t>(1, std::min<int64_t>(b, (int64_t)sms * 8));
}

// Strips of 16 x 64 per warp in the W-only 2D quantiser.  Measured on the
// Ultra expert weights (5.4 G elements, amax supplied): 1 (k_quant2d) 2.41 ms,
// 2 1.93-1.98 ms, 3 1.94 ms, 4 1.98 ms.
constexpr int Q2D_W_STRIPS = 2;

// Scale buffers above this size are written in band order by k_quant1d
// (the 126 MB L2 keeps smaller ones until their sectors are complete).
constexpr int64_t G_QUANT_SF_L2_BYTES = 48ll << 20;

// Blocks of 8 warps for k_quant1d: one warp per 512-element segment at most,
// and no more blocks than can be resident at once (the kernel splits its
// segments statically over the warps of the grid, so a second wave would be
// a tail).
template <bool SR, bool GROUPED, bool BAND>
int quant1d_blocks(int64_t rows, int64_t cols, int sms, size_t smem) {
    static int per_sm[64][2] = {};      // per device; [0]: computed, [1]: blocks per SM
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!per_sm[dev][0]) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_quant1d<SR, GROUPED, BAND>, 256, smem) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = 1;
        }
        per_sm[dev][1] = n;
        per_sm[dev][0] = 1;
    }
    // segments: 128 scale rows per band, 32 blocks per segment (grouped: one
    // partial band per expert at most)
    const int64_t segs = (cdiv(rows, 128) + (GROUPED ? NVFP4_MAX_GROUPS : 0)) * 128 * cdiv(cols / 16, 32);
    return (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(segs, 8), (int64_t)sms * per_sm[dev][1]));
}

int amax_blocks(int64_t units) {
    return (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(units, 256 * 8), 4096));
}

}  // namespace

// One mode of the RHT kernel over a dense operand (amax 0, RNE 1, SR 2, both
// amaxes 3, dual SR encoder 4): for modes 0, 1 and 3 the persistent streaming
// kernel when the rows can be copied in 16-byte pieces, else one CTA per tile.
template <int MODE>
static nvfp4_status launch_rht_dense(const void* x, int64_t tokens, int64_t cols, int64_t ld, uint16_t sign_mask,
                                     float* am, uint8_t* codes, uint8_t* sf, float* copy, nvfp4_stream_t stream,
                                     uint64_t seed = 0, const RowSR& rsr = RowSR{}) {
    int sms = 0, dev = 0;
    NVFP4_TRY(check_device(&sms, &dev));
    if constexpr (MODE == 0 || MODE == 1 || MODE == 3) {
        if (ld % 8 == 0 && cols % 8 == 0 && aligned16(x)) {
            {
                std::lock_guard<std::mutex> lk(g_dev_mu);
                if (!g_dev[dev].rht_attr) {
                    NVFP4_TRY(cuda_call(cudaFuncSetAttribute(k_rht_stream<0>,
                                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                             RHT_STREAM_SMEM), "smem attr"));
                    NVFP4_TRY(cuda_call(cudaFuncSetAttribute(k_rht_stream<1>,
                                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                             RHT_STREAM_SMEM), "smem attr"));
                    NVFP4_TRY(cuda_call(cudaFuncSetAttribute(k_rht_stream<3>,
                                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                             RHT_STREAM_SMEM), "smem attr"));
                    g_dev[dev].rht_attr = true;
                }
            }
            const int64_t tiles = cdiv(cols, 256) * cdiv(tokens, 64);
            const int grid = (int)std::min<int64_t>(tiles, (int64_t)sms * 3);
            k_rht_stream<MODE><<<grid, 256, RHT_STREAM_SMEM, stream>>>((const uint16_t*)x, tokens, cols, ld, sign_mask,
                                                                     am, codes, sf, copy);
            return launched("k_rht_stream");
        }
    }
    k_rht<MODE><<<dim3((unsigned)cdiv(cols, 256), (unsigned)cdiv(tokens, 64)), 256, 0, stream>>>(
        (const uint16_t*)x, tokens, cols, ld, sign_mask, am, seed, codes, sf, copy, nullptr, 1, 0, rsr);
    return launched("k_rht");
}


extern "C" {

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)sf_bytes(rows, cols);
}

size_t nvfp4_sf_bytes_grouped(int64_t rows, int64_t cols, int32_t num_groups) {
    if (rows < 0 || cols <= 0 || num_groups <= 0) return 0;
    return (size_t)sf_bytes(rows + 127 * (int64_t)num_groups, cols);
}

int64_t nvfp4_sf_offset(int64_t r, int64_t c, int64_t cols) { return sf_offset(r, c, cols); }

const char* nvfp4_status_string(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_NULL: return "null pointer";
        case NVFP4_ERR_SHAPE: return "invalid shape";
        case NVFP4_ERR_ALIGN: return "misaligned pointer or leading dimension";
        case NVFP4_ERR_DEVICE: return "no sm_103 CUDA device";
        case NVFP4_ERR_CUDA: return "CUDA error";
        case NVFP4_ERR_TIMEOUT: return "kernel wait timed out";
        case NVFP4_ERR_LIMIT: return "size beyond a documented limit";
    }
    return "unknown status";
}

const char* nvfp4_last_error(void) { return g_last_error; }

void nvfp4_debug_inject(nvfp4_status status) { g_inject.store((int)status); }

uint64_t nvfp4_launch_count(void) { return g_launches.load(); }

nvfp4_status nvfp4_amax(const void* x, int64_t batch, int64_t rows, int64_t cols, int64_t ld, float* amax,
                        nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (amax == nullptr) return fail(NVFP4_ERR_NULL, "amax is NULL");
    if (batch < 1 || batch > 65535) return fail(NVFP4_ERR_SHAPE, "batch must be in [1, 65535]");
    NVFP4_TRY(check_input(x, rows, cols, ld, 16, "x"));
    if (((uintptr_t)amax & 3u) != 0) return fail(NVFP4_ERR_ALIGN, "amax not 4-byte aligned");
    NVFP4_TRY(check_device());
    NVFP4_TRY(cuda_call(cudaMemsetAsync(amax, 0, sizeof(float) * batch, stream), "memset amax"));
    if (rows == 0 || cols == 0) return NVFP4_OK;
    k_amax<<<dim3(amax_blocks(rows * cols / 8), (unsigned)batch), 256, 0, stream>>>(
        (const uint16_t*)x, rows, cols, ld, rows * ld, amax);
    return launched("k_amax");
}

nvfp4_status nvfp4_quantize_1d(const void* x, int64_t rows, int64_t cols, int64_t ld, nvfp4_round mode,
                               uint64_t seed, const float* amax_in, nvfp4_tensor* out, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_input(x, rows, cols, ld, 16, "x"));
    NVFP4_TRY(check_out(out, rows, cols, true, "out"));
    if (mode != NVFP4_ROUND_RNE && mode != NVFP4_ROUND_SR) return fail(NVFP4_ERR_SHAPE, "bad rounding mode");
    int sms = 0;
    NVFP4_TRY(check_device(&sms));
    const float* am = amax_in;
    float* copy = nullptr;
    if (am == nullptr) {
        NVFP4_TRY(cuda_call(cudaMemsetAsync(out->amax, 0, sizeof(float), stream), "memset amax"));
        if (rows > 0 && cols > 0) {
            k_amax<<<dim3(amax_blocks(rows * cols / 8), 1), 256, 0, stream>>>((const uint16_t*)x, rows, cols, ld, 0,
                                                                               out->amax);
            NVFP4_TRY(launched("k_amax"));
        }
        am = out->amax;
    } else if (amax_in != out->amax) {
        copy = out->amax;
    }
    if (rows == 0 || cols == 0) {
        if (copy) NVFP4_TRY(cuda_call(cudaMemcpyAsync(copy, amax_in, 4, cudaMemcpyDeviceToDevice, stream), "amax copy"));
        return NVFP4_OK;
    }
    const bool band = (int64_t)sf_bytes(rows, cols) > G_QUANT_SF_L2_BYTES;
    const bool sr = mode == NVFP4_ROUND_SR;
    uint8_t* codes = (uint8_t*)out->codes;
    const uint16_t* xp = (const uint16_t*)x;
#define NVFP4_Q1D(SR_, BAND_)                                                                              \
    k_quant1d<SR_, false, BAND_><<<quant1d_blocks<SR_, false, BAND_>(rows, cols, sms, 0), 256, 0, stream>>>( \
        xp, rows, cols, ld, am, seed, codes, out->sf, nullptr, 0, copy)
    if (sr) { if (band) NVFP4_Q1D(true, true); else NVFP4_Q1D(true, false); }
    else { if (band) NVFP4_Q1D(false, true); else NVFP4_Q1D(false, false); }
#undef NVFP4_Q1D
    return launched("k_quant1d");       // it also writes the zero scales of the padding rows
}

nvfp4_status nvfp4_quantize_1d_grouped(const void* x, int64_t rows, int64_t cols, int64_t ld, const int64_t* offsets,
                                       int32_t num_groups, nvfp4_round mode, uint64_t seed, const float* amax_in,
                                       nvfp4_tensor* out, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_input(x, rows, cols, ld, 16, "x"));
    NVFP4_TRY(check_out(out, rows, cols, true, "out"));
    if (offsets == nullptr) return fail(NVFP4_ERR_NULL, "offsets is NULL");
    if (num_groups < 1 || num_groups > NVFP4_MAX_GROUPS) return fail(NVFP4_ERR_LIMIT, "num_groups must be in [1, %d]", NVFP4_MAX_GROUPS);
    if (rows >= (int64_t(1) << 31) - 128 * (int64_t)num_groups) return fail(NVFP4_ERR_LIMIT, "rows too large");
    if (mode != NVFP4_ROUND_RNE && mode != NVFP4_ROUND_SR) return fail(NVFP4_ERR_SHAPE, "bad rounding mode");
    int sms = 0;
    NVFP4_TRY(check_device(&sms));
    const size_t tab = sizeof(int32_t) * 2 * (num_groups + 1);
    const float* am = amax_in;
    float* copy = nullptr;
    if (am == nullptr) {
        NVFP4_TRY(cuda_call(cudaMemsetAsync(out->amax, 0, sizeof(float) * num_groups, stream), "memset amax"));
        if (rows > 0 && cols > 0) {
            k_amax_grouped<<<quant_blocks(rows, sms), 256, tab, stream>>>((const uint16_t*)x, rows, cols, ld, offsets,
                                                                           num_groups, out->amax);
            NVFP4_TRY(launched("k_amax_grouped"));
        }
        am = out->amax;
    } else if (amax_in != out->amax) {
        copy = out->amax;
    }
    if (rows == 0 || cols == 0) {
        if (copy)
            NVFP4_TRY(cuda_call(cudaMemcpyAsync(copy, amax_in, 4 * num_groups, cudaMemcpyDeviceToDevice, stream), "amax copy"));
        return NVFP4_OK;
    }
    // the group tables are sized for NVFP4_MAX_GROUPS in the occupancy query
    const size_t tab_max = sizeof(int32_t) * 2 * (NVFP4_MAX_GROUPS + 1);
    const bool band = (int64_t)sf_bytes(rows + 127 * (int64_t)num_groups, cols) > G_QUANT_SF_L2_BYTES;
    const bool sr = mode == NVFP4_ROUND_SR;
    uint8_t* codes = (uint8_t*)out->codes;
    const uint16_t* xp = (const uint16_t*)x;
#define NVFP4_Q1G(SR_, BAND_)                                                                                   \
    k_quant1d<SR_, true, BAND_><<<quant1d_blocks<SR_, true, BAND_>(rows, cols, sms, tab_max), 256, tab, stream>>>( \
        xp, rows, cols, ld, am, seed, codes, out->sf, offsets, num_groups, copy)
    if (sr) { if (band) NVFP4_Q1G(true, true); else NVFP4_Q1G(true, false); }
    else { if (band) NVFP4_Q1G(false, true); else NVFP4_Q1G(false, false); }
#undef NVFP4_Q1G
    return launched("k_quant1d grouped");   // it also writes the zero scales of each expert's padding rows
}

nvfp4_status nvfp4_quantize_2d(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ld,
                               const float* amax_in, nvfp4_tensor* out, nvfp4_tensor* out_t, uint8_t* tile_sf,
                               nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (batch < 1 || batch > 65535) return fail(NVFP4_ERR_SHAPE, "batch must be in [1, 65535]");
    NVFP4_TRY(check_input(w, rows * batch, cols, ld, 16, "w"));
    if (rows % 16 != 0) return fail(NVFP4_ERR_SHAPE, "rows=%lld is not a multiple of 16", (long long)rows);
    if (cdiv(rows, 64) > 65535) return fail(NVFP4_ERR_LIMIT, "rows too large");
    NVFP4_TRY(check_out(out, rows, cols, true, "out"));
    if (out_t != nullptr) NVFP4_TRY(check_out(out_t, cols, rows, false, "out_t"));
    int sms = 0;
    NVFP4_TRY(check_device(&sms));
    const float* am = amax_in;
    float* copy = nullptr;
    if (am == nullptr) {
        NVFP4_TRY(cuda_call(cudaMemsetAsync(out->amax, 0, sizeof(float) * batch, stream), "memset amax"));
        if (rows > 0 && cols > 0) {
            k_amax<<<dim3(amax_blocks(rows * cols / 8), (unsigned)batch), 256, 0, stream>>>((const uint16_t*)w, rows, cols,
                                                                                          ld, rows * ld, out->amax);
            NVFP4_TRY(launched("k_amax"));
        }
        am = out->amax;
    } else if (amax_in != out->amax) {
        copy = out->amax;
    }
    if (rows == 0 || cols == 0) {
        if (copy) NVFP4_TRY(cuda_call(cudaMemcpyAsync(copy, amax_in, 4 * batch, cudaMemcpyDeviceToDevice, stream), "amax copy"));
        return NVFP4_OK;
    }
    if (out_t == nullptr) {
        dim3 grid((unsigned)cdiv(cols, 64 * Q2D_W_STRIPS), (unsigned)cdiv(rows, 64), (unsigned)batch);
        k_quant2d_w<Q2D_W_STRIPS><<<grid, 128, 0, stream>>>((const uint16_t*)w, rows, cols, ld, am,
                                                           (uint8_t*)out->codes, out->sf, tile_sf, copy);
        NVFP4_TRY(launched("k_quant2d_w"));
    } else {
        dim3 grid((unsigned)cdiv(cols, 64), (unsigned)cdiv(rows, 64), (unsigned)batch);
        k_quant2d<<<grid, 128, 0, stream>>>((const uint16_t*)w, rows, cols, ld, am, (uint8_t*)out->codes, out->sf,
                                            (uint8_t*)out_t->codes, out_t->sf, tile_sf, copy);
        NVFP4_TRY(launched("k_quant2d"));
    }
    const bool pad = (rows % 128) || ((cols / 16) % 4) || (out_t && ((cols % 128) || ((rows / 16) % 4)));
    if (pad) {
        k_quant2d_pad<<<dim3(16, (unsigned)batch), 256, 0, stream>>>(out->sf, out_t ? out_t->sf : nullptr, rows, cols);
        NVFP4_TRY(launched("k_quant2d_pad"));
    }
    return NVFP4_OK;
}

size_t nvfp4_quantize_2d_fused_workspace(int64_t batch) {
    if (batch < 1) return 0;
    // per-entry counters, the abort word and a spare word, rounded up to 16 bytes
    return (size_t)(((batch + 2) * 4 + 15) / 16 * 16);
}

nvfp4_status nvfp4_quantize_2d_fused(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ld,
                                     void* workspace, size_t workspace_bytes, nvfp4_tensor* out, uint8_t* tile_sf,
                                     nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (batch < 1 || batch > 65535) return fail(NVFP4_ERR_SHAPE, "batch must be in [1, 65535]");
    NVFP4_TRY(check_input(w, rows * batch, cols, ld, 16, "w"));
    if (rows % 16 != 0) return fail(NVFP4_ERR_SHAPE, "rows=%lld is not a multiple of 16", (long long)rows);
    NVFP4_TRY(check_out(out, rows, cols, true, "out"));
    if (workspace == nullptr) return fail(NVFP4_ERR_NULL, "workspace is NULL");
    if (!aligned16(workspace)) return fail(NVFP4_ERR_ALIGN, "workspace not 16-byte aligned");
    if (workspace_bytes < nvfp4_quantize_2d_fused_workspace(batch))
        return fail(NVFP4_ERR_SHAPE, "workspace of %zu bytes, %zu needed", workspace_bytes,
                    nvfp4_quantize_2d_fused_workspace(batch));
    int sms = 0, dev = 0;
    NVFP4_TRY(check_device(&sms, &dev));
    NVFP4_TRY(cuda_call(cudaMemsetAsync(out->amax, 0, sizeof(float) * batch, stream), "memset amax"));
    if (rows == 0 || cols == 0) return NVFP4_OK;
    NVFP4_TRY(cuda_call(cudaMemsetAsync(workspace, 0, nvfp4_quantize_2d_fused_workspace(batch), stream), "memset workspace"));
    if ((rows / 16) * cdiv(cols, Q2F_ITEM_COLS) > (int64_t)0x7FFFFFFF)
        return fail(NVFP4_ERR_LIMIT, "an entry of %lld x %lld is too large", (long long)rows, (long long)cols);
    const int64_t col_units = cdiv(cols, Q2R_UNIT_COLS);
    const int64_t units = (rows / 16) * col_units;
    if (units <= (int64_t)Q2R_MAX_UNITS * sms && batch * rows <= (int64_t)0x7FFFFFFF) {
        // every entry fits in the CTAs' registers: one read of HBM
        {
            std::lock_guard<std::mutex> lk(g_dev_mu);
            if (!g_dev[dev].q2r_attr) {
                NVFP4_TRY(cuda_call(cudaFuncSetAttribute(k_quant2d_resident, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         Q2R_SMEM_BYTES), "smem attr"));
                g_dev[dev].q2r_attr = true;
            }
        }
        int per_sm = 0;
        NVFP4_TRY(cuda_call(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quant2d_resident, Q2R_THREADS,
                                                                          Q2R_SMEM_BYTES), "occupancy"));
        if (per_sm < 1) return fail(NVFP4_ERR_CUDA, "resident 2D quantiser cannot be resident");
        auto fn = encode_fn();
        if (fn == nullptr) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
        const int64_t box_cols = std::min<int64_t>(cols, Q2R_UNIT_COLS);
        CUtensorMap map;
        cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(batch * rows)};
        cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
        cuuint32_t box[2] = {(cuuint32_t)box_cols, 16u};
        cuuint32_t estr[2] = {1u, 1u};
        const CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled (weights) failed (%d)", (int)r);
        Quant2dResidentArgs qa{batch, rows, cols, units, col_units, (int32_t)(box_cols * 2), out->amax,
                               (uint32_t*)workspace, (uint8_t*)out->codes, out->sf, tile_sf};
        const int64_t grid = std::min<int64_t>(sms, units);
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(Q2R_THREADS);
        cfg.dynamicSmemBytes = Q2R_SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        NVFP4_TRY(cuda_call(cudaLaunchKernelEx(&cfg, k_quant2d_resident, map, qa), "k_quant2d_resident launch"));
        NVFP4_TRY(launched("k_quant2d_resident"));
        if ((rows % 128) || ((cols / 16) % 4)) {
            k_quant2d_pad<<<dim3(16, (unsigned)batch), 256, 0, stream>>>(out->sf, nullptr, rows, cols);
            NVFP4_TRY(launched("k_quant2d_pad"));
        }
        return NVFP4_OK;
    }
    int per_sm = 0;
    NVFP4_TRY(cuda_call(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quant2d_fused, Q2F_THREADS, 0), "occupancy"));
    if (per_sm < 1) return fail(NVFP4_ERR_CUDA, "fused 2D quantiser cannot be resident");
    // every block must be resident (cooperative launch); a small problem takes fewer warps
    const int64_t items = batch * (rows / 16) * cdiv(cols, Q2F_ITEM_COLS);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(items, Q2F_THREADS / 32), (int64_t)per_sm * sms));
    const uint16_t* wp = (const uint16_t*)w;
    float* am = out->amax;
    uint32_t* cnt = (uint32_t*)workspace;
    uint8_t* codes = (uint8_t*)out->codes;
    uint8_t* sf = out->sf;
    void* args[] = {&wp, &batch, &rows, &cols, &ld, &am, &cnt, &codes, &sf, &tile_sf};
    NVFP4_TRY(cuda_call(cudaLaunchCooperativeKernel((const void*)k_quant2d_fused, dim3(grid), dim3(Q2F_THREADS), args, 0, stream),
                        "k_quant2d_fused launch"));
    NVFP4_TRY(launched("k_quant2d_fused"));
    if ((rows % 128) || ((cols / 16) % 4)) {
        k_quant2d_pad<<<dim3(16, (unsigned)batch), 256, 0, stream>>>(out->sf, nullptr, rows, cols);
        NVFP4_TRY(launched("k_quant2d_pad"));
    }
    return NVFP4_OK;
}

// ------------------------------------------------------------------ allocation-free variant
// Counter scratch of nvfp4_quantize_2d_fused_static: one word per batch entry
// plus the abort word, in a fixed array that every GPU loading this library
// holds until the process exits.  Host code must not pass the symbol itself
// to a kernel (on the host it only names a stand-in); the device address is
// looked up once per device with that device current.
static __device__ __align__(256) uint32_t g_q2f_static_scratch[NVFP4_STATIC_MAX_BATCH + 8];

namespace {
uint32_t* g_static_scratch_ptr[MAX_DEVICES] = {};   // by device ordinal (check_device bounds it)
}

nvfp4_status nvfp4_quantize_2d_fused_static(const void* w, int64_t batch, int64_t rows, int64_t cols, int64_t ld,
                                            nvfp4_tensor* out, uint8_t* tile_sf, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (batch > NVFP4_STATIC_MAX_BATCH)
        return fail(NVFP4_ERR_LIMIT, "batch=%lld exceeds the %d entries of the static scratch; use nvfp4_quantize_2d_fused "
                    "with a workspace", (long long)batch, NVFP4_STATIC_MAX_BATCH);
    int sms = 0, dev = 0;
    NVFP4_TRY(check_device(&sms, &dev));
    uint32_t* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (g_static_scratch_ptr[dev] == nullptr) {
            void* p = nullptr;
            NVFP4_TRY(cuda_call(cudaGetSymbolAddress(&p, g_q2f_static_scratch), "cudaGetSymbolAddress(static scratch)"));
            g_static_scratch_ptr[dev] = static_cast<uint32_t*>(p);
        }
        scratch = g_static_scratch_ptr[dev];
    }
    return nvfp4_quantize_2d_fused(w, batch, rows, cols, ld, scratch, sizeof(g_q2f_static_scratch), out, tile_sf,
                                   stream);
}

nvfp4_status nvfp4_rht_amax(const void* x, int64_t tokens, int64_t cols, int64_t ld, uint16_t sign_mask, float* amax,
                            nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (amax == nullptr) return fail(NVFP4_ERR_NULL, "amax is NULL");
    NVFP4_TRY(check_input(x, tokens, cols, ld, 1, "x", false));
    if (tokens % 16 != 0) return fail(NVFP4_ERR_SHAPE, "tokens=%lld is not a multiple of 16", (long long)tokens);
    if (cdiv(tokens, 64) > 65535) return fail(NVFP4_ERR_LIMIT, "tokens too large");
    NVFP4_TRY(check_device());
    NVFP4_TRY(cuda_call(cudaMemsetAsync(amax, 0, sizeof(float), stream), "memset amax"));
    if (tokens == 0 || cols == 0) return NVFP4_OK;
    return launch_rht_dense<0>(x, tokens, cols, ld, sign_mask, amax, nullptr, nullptr, nullptr, stream);
}

nvfp4_status nvfp4_dual_amax(const void* x, int64_t tokens, int64_t cols, int64_t ld, uint16_t sign_mask,
                             float* amax_plain, float* amax_rht, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (amax_plain == nullptr || amax_rht == nullptr) return fail(NVFP4_ERR_NULL, "amax_plain or amax_rht is NULL");
    NVFP4_TRY(check_input(x, tokens, cols, ld, 1, "x", false));
    if (tokens % 16 != 0) return fail(NVFP4_ERR_SHAPE, "tokens=%lld is not a multiple of 16", (long long)tokens);
    if (cdiv(tokens, 64) > 65535) return fail(NVFP4_ERR_LIMIT, "tokens too large");
    NVFP4_TRY(check_device());
    NVFP4_TRY(cuda_call(cudaMemsetAsync(amax_plain, 0, sizeof(float), stream), "memset amax"));
    NVFP4_TRY(cuda_call(cudaMemsetAsync(amax_rht, 0, sizeof(float), stream), "memset amax"));
    if (tokens == 0 || cols == 0) return NVFP4_OK;
    return launch_rht_dense<3>(x, tokens, cols, ld, sign_mask, amax_rht, nullptr, nullptr, amax_plain, stream);
}

nvfp4_status nvfp4_dual_sr_quantize(const void* dy, int64_t tokens, int64_t cols, int64_t ld, uint16_t sign_mask,
                                    uint64_t seed_row, uint64_t seed_rht, const float* amax_row, const float* amax_rht,
                                    nvfp4_tensor* out_row, nvfp4_tensor* out_t, uint64_t* zero_count,
                                    nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_input(dy, tokens, cols, ld, 16, "dy", false));
    if (tokens % 16 != 0) return fail(NVFP4_ERR_SHAPE, "tokens=%lld is not a multiple of 16", (long long)tokens);
    if (cdiv(tokens, 64) > 65535) return fail(NVFP4_ERR_LIMIT, "tokens too large");
    if (amax_row == nullptr || amax_rht == nullptr) return fail(NVFP4_ERR_NULL, "amax_row or amax_rht is NULL");
    NVFP4_TRY(check_out(out_row, tokens, cols, true, "out_row"));
    NVFP4_TRY(check_out(out_t, cols, tokens, true, "out_t"));
    if (zero_count != nullptr && ((uintptr_t)zero_count & 7u) != 0) return fail(NVFP4_ERR_ALIGN, "zero_count not 8-byte aligned");
    NVFP4_TRY(check_device());
    if (zero_count != nullptr) NVFP4_TRY(cuda_call(cudaMemsetAsync(zero_count, 0, sizeof(uint64_t), stream), "memset count"));
    if (tokens == 0 || cols == 0) {
        NVFP4_TRY(cuda_call(cudaMemcpyAsync(out_row->amax, amax_row, 4, cudaMemcpyDeviceToDevice, stream), "amax copy"));
        return cuda_call(cudaMemcpyAsync(out_t->amax, amax_rht, 4, cudaMemcpyDeviceToDevice, stream), "amax copy");
    }
    RowSR rsr;
    rsr.amax_row = amax_row;
    rsr.seed_row = seed_row;
    rsr.codes_r = (uint8_t*)out_row->codes;
    rsr.sf_r = out_row->sf;
    rsr.zero_count = reinterpret_cast<unsigned long long*>(zero_count);
    rsr.amax_row_copy = amax_row != out_row->amax ? out_row->amax : nullptr;
    float* copy_t = amax_rht != out_t->amax ? out_t->amax : nullptr;
    NVFP4_TRY(launch_rht_dense<4>(dy, tokens, cols, ld, sign_mask, const_cast<float*>(amax_rht),
                                  (uint8_t*)out_t->codes, out_t->sf, copy_t, stream, seed_rht, rsr));
    // scale padding rows of both operands (rows past tokens, or past cols)
    if (tokens % 128 != 0) {
        k_zero_pad_rows<<<64, 256, 0, stream>>>(out_row->sf, tokens, cols, nullptr, 0);
        NVFP4_TRY(launched("k_zero_pad_rows"));
    }
    if (cols % 128 != 0) {
        k_zero_pad_rows<<<64, 256, 0, stream>>>(out_t->sf, cols, tokens, nullptr, 0);
        NVFP4_TRY(launched("k_zero_pad_rows"));
    }
    return NVFP4_OK;
}

nvfp4_status nvfp4_count_zero_codes(const nvfp4_tensor* t, uint64_t* count, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (t == nullptr || count == nullptr) return fail(NVFP4_ERR_NULL, "t or count is NULL");
    if (t->rows < 0 || t->cols < 0 || (t->cols & 1)) return fail(NVFP4_ERR_SHAPE, "bad tensor shape");
    if (((uintptr_t)count & 7u) != 0) return fail(NVFP4_ERR_ALIGN, "count not 8-byte aligned");
    int sms = 0;
    NVFP4_TRY(check_device(&sms));
    NVFP4_TRY(cuda_call(cudaMemsetAsync(count, 0, sizeof(uint64_t), stream), "memset count"));
    const int64_t nbytes = t->rows * (t->cols / 2);
    if (nbytes == 0) return NVFP4_OK;
    if (t->codes == nullptr || !aligned16(t->codes)) return fail(NVFP4_ERR_ALIGN, "codes NULL or not 16-byte aligned");
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(nbytes, 256 * 16), (int64_t)sms * 8));
    k_count_zero_codes<<<grid, 256, 0, stream>>>((const uint8_t*)t->codes, nbytes,
                                                 reinterpret_cast<unsigned long long*>(count));
    return launched("k_count_zero_codes");
}

nvfp4_status nvfp4_rht_quantize(const void* x, int64_t tokens, int64_t cols, int64_t ld, uint16_t sign_mask,
                                nvfp4_round mode, uint64_t seed, const float* amax_in, nvfp4_tensor* out_t,
                                nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_input(x, tokens, cols, ld, 1, "x", false));
    if (tokens % 16 != 0) return fail(NVFP4_ERR_SHAPE, "tokens=%lld is not a multiple of 16", (long long)tokens);
    if (cdiv(tokens, 64) > 65535) return fail(NVFP4_ERR_LIMIT, "tokens too large");
    NVFP4_TRY(check_out(out_t, cols, tokens, true, "out_t"));
    if (mode != NVFP4_ROUND_RNE && mode != NVFP4_ROUND_SR) return fail(NVFP4_ERR_SHAPE, "bad rounding mode");
    NVFP4_TRY(check_device());
    const float* am = amax_in;
    float* copy = nullptr;
    if (am == nullptr) {
        NVFP4_TRY(cuda_call(cudaMemsetAsync(out_t->amax, 0, sizeof(float), stream), "memset amax"));
        if (tokens > 0 && cols > 0)
            NVFP4_TRY(launch_rht_dense<0>(x, tokens, cols, ld, sign_mask, out_t->amax, nullptr, nullptr, nullptr, stream));
        am = out_t->amax;
    } else if (amax_in != out_t->amax) {
        copy = out_t->amax;
    }
    if (tokens == 0 || cols == 0) {
        if (copy) NVFP4_TRY(cuda_call(cudaMemcpyAsync(copy, amax_in, 4, cudaMemcpyDeviceToDevice, stream), "amax copy"));
        return NVFP4_OK;
    }
    if (mode == NVFP4_ROUND_SR) {
        NVFP4_TRY(launch_rht_dense<2>(x, tokens, cols, ld, sign_mask, const_cast<float*>(am), (uint8_t*)out_t->codes,
                                      out_t->sf, copy, stream, seed));
    } else {
        NVFP4_TRY(launch_rht_dense<1>(x, tokens, cols, ld, sign_mask, const_cast<float*>(am), (uint8_t*)out_t->codes,
                                      out_t->sf, copy, stream));
    }
    if (cols % 128 != 0) {
        k_zero_pad_rows<<<64, 256, 0, stream>>>(out_t->sf, cols, tokens, nullptr, 0);
        NVFP4_TRY(launched("k_zero_pad_rows"));
    }
    return NVFP4_OK;
}

nvfp4_status nvfp4_quantize_1d_mse(const void* x, int64_t rows, int64_t cols, int64_t ld, const float* amax_in,
                                   nvfp4_tensor* out, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_input(x, rows, cols, ld, 16, "x"));       // 16-byte aligned rows (vector loads)
    NVFP4_TRY(check_out(out, rows, cols, true, "out"));
    int sms = 0;
    NVFP4_TRY(check_device(&sms));
    const float* am = amax_in;
    float* copy = nullptr;
    if (am == nullptr) {
        NVFP4_TRY(cuda_call(cudaMemsetAsync(out->amax, 0, sizeof(float), stream), "memset amax"));
        if (rows > 0 && cols > 0) {
            k_amax<<<dim3(amax_blocks(rows * cols / 8), 1), 256, 0, stream>>>((const uint16_t*)x, rows, cols, ld, 0,
                                                                           out->amax);
            NVFP4_TRY(launched("k_amax"));
        }
        am = out->amax;
    } else if (amax_in != out->amax) {
        copy = out->amax;
    }
    NVFP4_TRY(cuda_call(cudaMemsetAsync(out->sf, 0, nvfp4_sf_bytes(rows, cols), stream), "memset sf"));
    if (rows == 0 || cols == 0) {
        if (copy) NVFP4_TRY(cuda_call(cudaMemcpyAsync(copy, amax_in, 4, cudaMemcpyDeviceToDevice, stream), "amax copy"));
        return NVFP4_OK;
    }
    const int64_t blocks = rows * (cols / 16);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(blocks, 256), (int64_t)sms * 16));
    k_quant1d_mse<<<grid, 256, 0, stream>>>((const uint16_t*)x, rows, cols, ld, am, (uint8_t*)out->codes, out->sf,
                                            copy);
    return launched("k_quant1d_mse");
}

nvfp4_status nvfp4_sr_fp16(const float* x, int64_t n, uint64_t seed, uint16_t* out, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (n < 0) return fail(NVFP4_ERR_SHAPE, "n < 0");
    if (n == 0) return NVFP4_OK;
    if (x == nullptr || out == nullptr) return fail(NVFP4_ERR_NULL, "x or out is NULL");
    if (((uintptr_t)x & 3u) || ((uintptr_t)out & 1u)) return fail(NVFP4_ERR_ALIGN, "x or out misaligned");
    int sms = 0;
    NVFP4_TRY(check_device(&sms));
    const int64_t nq = cdiv(n, 4);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(nq, 256), (int64_t)sms * 8));
    k_sr_fp16<<<grid, 256, 0, stream>>>(x, n, seed, out);
    return launched("k_sr_fp16");
}

int64_t nvfp4_group_k_capacity(int64_t rows, int32_t groups) {
    if (rows < 0 || groups < 1) return 0;
    return cdiv(rows + 63 * (int64_t)groups, 64) * 64;
}

nvfp4_status nvfp4_rht_quantize_grouped(const void* x, int64_t rows, int64_t cols, int64_t ld, const int64_t* offsets,
                                        int32_t num_groups, int64_t kt, uint16_t sign_mask, nvfp4_round mode,
                                        uint64_t seed, const float* amax_in, nvfp4_tensor* out_t,
                                        nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_input(x, rows, cols, ld, 1, "x", false));
    if (offsets == nullptr) return fail(NVFP4_ERR_NULL, "offsets is NULL");
    if (num_groups < 1 || num_groups > NVFP4_MAX_GROUPS)
        return fail(NVFP4_ERR_LIMIT, "num_groups must be in [1, %d]", NVFP4_MAX_GROUPS);
    if (kt % 64 != 0 || kt < nvfp4_group_k_capacity(rows, num_groups))
        return fail(NVFP4_ERR_SHAPE, "kt=%lld must be a multiple of 64 and at least nvfp4_group_k_capacity = %lld",
                    (long long)kt, (long long)nvfp4_group_k_capacity(rows, num_groups));
    if (kt / 64 > 65535 || rows >= (int64_t(1) << 31)) return fail(NVFP4_ERR_LIMIT, "too many tokens");
    NVFP4_TRY(check_out(out_t, cols, kt, true, "out_t"));
    if (mode != NVFP4_ROUND_RNE && mode != NVFP4_ROUND_SR) return fail(NVFP4_ERR_SHAPE, "bad rounding mode");
    NVFP4_TRY(check_device());
    const int tab = 2 * 4 * (num_groups + 1);
    const float* am = amax_in;
    float* copy = nullptr;
    const dim3 grid((unsigned)cdiv(cols, 256), (unsigned)(kt / 64));
    if (am == nullptr) {
        NVFP4_TRY(cuda_call(cudaMemsetAsync(out_t->amax, 0, sizeof(float) * num_groups, stream), "memset amax"));
        if (rows > 0 && cols > 0) {
            k_rht<0, true><<<grid, 256, tab, stream>>>((const uint16_t*)x, rows, cols, ld, sign_mask, out_t->amax, 0,
                                                      nullptr, nullptr, nullptr, offsets, num_groups, kt);
            NVFP4_TRY(launched("k_rht amax grouped"));
        }
        am = out_t->amax;
    } else if (amax_in != out_t->amax) {
        copy = out_t->amax;
    }
    if (rows == 0 || cols == 0) {
        if (copy)
            NVFP4_TRY(cuda_call(cudaMemcpyAsync(copy, amax_in, 4 * num_groups, cudaMemcpyDeviceToDevice, stream),
                                "amax copy"));
        return NVFP4_OK;
    }
    if (mode == NVFP4_ROUND_SR)
        k_rht<2, true><<<grid, 256, tab, stream>>>((const uint16_t*)x, rows, cols, ld, sign_mask, const_cast<float*>(am),
                                                  seed, (uint8_t*)out_t->codes, out_t->sf, copy, offsets, num_groups, kt);
    else
        k_rht<1, true><<<grid, 256, tab, stream>>>((const uint16_t*)x, rows, cols, ld, sign_mask, const_cast<float*>(am),
                                                  seed, (uint8_t*)out_t->codes, out_t->sf, copy, offsets, num_groups, kt);
    NVFP4_TRY(launched("k_rht quantize grouped"));
    if (cols % 128 != 0) {
        k_zero_pad_rows<<<64, 256, 0, stream>>>(out_t->sf, cols, kt, nullptr, 0);
        NVFP4_TRY(launched("k_zero_pad_rows"));
    }
    return NVFP4_OK;
}

static nvfp4_status check_operand(const nvfp4_tensor* t, const char* name) {
    if (t == nullptr) return fail(NVFP4_ERR_NULL, "%s is NULL", name);
    if (t->rows < 0 || t->cols < 0) return fail(NVFP4_ERR_SHAPE, "%s: negative size", name);
    if (t->rows > 0 && (t->codes == nullptr || t->sf == nullptr || t->amax == nullptr))
        return fail(NVFP4_ERR_NULL, "%s: codes/sf/amax NULL", name);
    if (!aligned16(t->codes) || !aligned16(t->sf)) return fail(NVFP4_ERR_ALIGN, "%s: codes/sf not 16-byte aligned", name);
    return NVFP4_OK;
}

}  // extern "C"

// CTA pairs (cta_group::2) unless NVFP4_GEMM_PAIR=0 is set in the
// environment (read at every call, so a process can compare both kernels).
static bool use_pair() {
    const char* e = std::getenv("NVFP4_GEMM_PAIR");
    return !(e != nullptr && e[0] == '0');
}

template <bool F32, bool TS, bool PAIR, int SCHED>
static nvfp4_status launch_one(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                               const GemmParams& p, int grid, int smem, nvfp4_stream_t stream) {
    auto kern = k_gemm_nvfp4<F32, TS, PAIR, SCHED>;
    if (!PAIR) {
        kern<<<grid, G_THREADS, smem, stream>>>(ma, mb, mc, p);
        return launched("k_gemm_nvfp4");
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    NVFP4_TRY(cuda_call(cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, p), "k_gemm_nvfp4 pair launch"));
    return launched("k_gemm_nvfp4 pair");
}

template <bool F32, bool TS, bool PAIR, int SCHED>
static nvfp4_status set_gemm_attr() {
    const int groups = SCHED == G_DENSE ? 1 : NVFP4_MAX_GROUPS;
    NVFP4_TRY(cuda_call(cudaFuncSetAttribute(k_gemm_nvfp4<F32, TS, PAIR, SCHED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             gemm_smem_bytes(TS, groups, PAIR, SCHED == G_DENSE)),
                        "smem attr"));
    if (PAIR)
        NVFP4_TRY(cuda_call(cudaFuncSetAttribute(k_gemm_nvfp4<F32, TS, PAIR, SCHED>,
                                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 0),
                            "cluster attr"));
    return NVFP4_OK;
}

// Attributes of the four output modes (bf16 / FP32, direct / TMA store) of
// one schedule and CTA arrangement.
template <bool PAIR, int SCHED>
static nvfp4_status set_gemm_attrs() {
    NVFP4_TRY((set_gemm_attr<false, false, PAIR, SCHED>()));
    NVFP4_TRY((set_gemm_attr<false, true, PAIR, SCHED>()));
    NVFP4_TRY((set_gemm_attr<true, false, PAIR, SCHED>()));
    NVFP4_TRY((set_gemm_attr<true, true, PAIR, SCHED>()));
    return NVFP4_OK;
}

// Largest number of co-resident CTA pairs of the pair kernel in its largest
// layout (the grid is sized to it: the kernel is persistent over tiles).
static nvfp4_status pair_clusters(int* out) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = std::max(gemm_smem_bytes(true, 1, true, true), gemm_smem_bytes(true, NVFP4_MAX_GROUPS, true, false));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    NVFP4_TRY(cuda_call(cudaOccupancyMaxActiveClusters(&n, k_gemm_nvfp4<false, true, true, G_DENSE>, &cfg),
                        "cluster occupancy"));
    *out = n;
    return NVFP4_OK;
}

template <bool PAIR, int SCHED>
static nvfp4_status launch_mode(bool f32, bool ts, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                                const GemmParams& p, int grid, int smem, nvfp4_stream_t stream) {
    if (f32) return ts ? launch_one<true, true, PAIR, SCHED>(ma, mb, mc, p, grid, smem, stream)
                       : launch_one<true, false, PAIR, SCHED>(ma, mb, mc, p, grid, smem, stream);
    return ts ? launch_one<false, true, PAIR, SCHED>(ma, mb, mc, p, grid, smem, stream)
              : launch_one<false, false, PAIR, SCHED>(ma, mb, mc, p, grid, smem, stream);
}

// tiles_1cta: output tiles of 128 x 256 (grid bound of the single-CTA
// kernel); pair_tiles: tiles of 256 x 256.  sched: G_DENSE, G_MGROUP or
// G_KGROUP.  tma_store: C's rows are 16-byte aligned and mc maps it.
static nvfp4_status launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                                const GemmParams& p, int64_t tiles_1cta, int64_t pair_tiles, int sms,
                                nvfp4_out_dtype dt, bool tma_store, bool pair, nvfp4_stream_t stream, int dev,
                                int sched) {
    const bool f32 = dt == NVFP4_OUT_FP32;
    const int smem = gemm_smem_bytes(tma_store, p.groups, pair, sched == G_DENSE);
    int clusters = 0;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!g_dev[dev].gemm_attr) {
            NVFP4_TRY((set_gemm_attrs<false, G_DENSE>()));
            NVFP4_TRY((set_gemm_attrs<false, G_MGROUP>()));
            NVFP4_TRY((set_gemm_attrs<false, G_KGROUP>()));
            NVFP4_TRY((set_gemm_attrs<true, G_DENSE>()));
            NVFP4_TRY((set_gemm_attrs<true, G_MGROUP>()));
            NVFP4_TRY((set_gemm_attrs<true, G_KGROUP>()));
            int c = 0;
            NVFP4_TRY(pair_clusters(&c));
            g_dev[dev].pair_clusters = c;
            g_dev[dev].gemm_attr = true;
        }
        clusters = g_dev[dev].pair_clusters;
    }
    if (sched == G_KGROUP && !f32 && !tma_store)
        return fail(NVFP4_ERR_ALIGN, "bf16 output of a K-grouped GEMM needs 16-byte rows");
    if (!pair) {
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles_1cta, sms));
        if (sched == G_KGROUP) return launch_mode<false, G_KGROUP>(f32, tma_store, ma, mb, mc, p, grid, smem, stream);
        if (sched == G_MGROUP) return launch_mode<false, G_MGROUP>(f32, tma_store, ma, mb, mc, p, grid, smem, stream);
        return launch_mode<false, G_DENSE>(f32, tma_store, ma, mb, mc, p, grid, smem, stream);
    }
    if (clusters < 1) return fail(NVFP4_ERR_CUDA, "the CTA-pair GEMM cannot be resident");
    const int grid = 2 * (int)std::max<int64_t>(1, std::min<int64_t>(pair_tiles, clusters));
    if (sched == G_KGROUP) return launch_mode<true, G_KGROUP>(f32, tma_store, ma, mb, mc, p, grid, smem, stream);
    if (sched == G_MGROUP) return launch_mode<true, G_MGROUP>(f32, tma_store, ma, mb, mc, p, grid, smem, stream);
    return launch_mode<true, G_DENSE>(f32, tma_store, ma, mb, mc, p, grid, smem, stream);
}

extern "C" {

// Store tensor map of a bf16 or FP32 output [rows, n] with row stride ldc:
// boxes of 32 rows x 64 bytes (32 bf16 or 16 FP32 columns) with 64-byte
// swizzle.  Only built when C's rows are 16-byte aligned; otherwise the
// kernel stores directly.
static nvfp4_status make_store_map(CUtensorMap* map, void* c, int64_t rows, int64_t n, int64_t ldc, bool f32,
                                   bool* enabled) {
    std::memset(map, 0, sizeof(*map));
    *enabled = false;
    const int esz = f32 ? 4 : 2;
    if (!aligned16(c) || (ldc * esz) % 16 != 0) return NVFP4_OK;
    auto fn = encode_fn();
    if (fn == nullptr) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ldc * esz)};
    cuuint32_t box[2] = {f32 ? 16u : 32u, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c, dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled (store) failed (%d)", (int)r);
    *enabled = true;
    return NVFP4_OK;
}

nvfp4_status nvfp4_gemm(const nvfp4_tensor* a, const nvfp4_tensor* b, void* c, int64_t ldc, nvfp4_out_dtype c_dtype,
                        float* c_amax, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_operand(a, "a"));
    NVFP4_TRY(check_operand(b, "b"));
    const int64_t M = a->rows, N = b->rows, K = a->cols;
    if (b->cols != K) return fail(NVFP4_ERR_SHAPE, "a->cols=%lld != b->cols=%lld", (long long)K, (long long)b->cols);
    if (K % 16 != 0 || K == 0) return fail(NVFP4_ERR_SHAPE, "K=%lld must be a positive multiple of 16", (long long)K);
    if (c_dtype != NVFP4_OUT_BF16 && c_dtype != NVFP4_OUT_FP32) return fail(NVFP4_ERR_SHAPE, "bad output dtype");
    if (ldc < N) return fail(NVFP4_ERR_SHAPE, "ldc < N");
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return fail(NVFP4_ERR_LIMIT, "M or N >= 2^31");
    if (M == 0 || N == 0) return NVFP4_OK;
    if (c == nullptr) return fail(NVFP4_ERR_NULL, "c is NULL");
    const int esz = c_dtype == NVFP4_OUT_FP32 ? 4 : 2;
    if (((uintptr_t)c % esz) != 0) return fail(NVFP4_ERR_ALIGN, "c is not aligned to its element size");
    int sms = 0, dev = 0;
    NVFP4_TRY(check_device(&sms, &dev));
    // K % 32 == 16: code rows are not a 16-byte multiple (no tensor map); the
    // single-CTA kernel copies them
    const bool copy_ab = K % 32 != 0;
    const bool pair = use_pair() && !copy_ab;
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof(ma));
    std::memset(&mb, 0, sizeof(mb));
    if (!copy_ab) {
        NVFP4_TRY(make_code_map(&ma, a->codes, M, K / 2, G_BM));
        NVFP4_TRY(make_code_map(&mb, b->codes, N, K / 2, pair ? G_BN / 2 : G_BN));
    }
    GemmParams p{};
    p.copy_ab = copy_ab;
    p.a_codes = (const uint8_t*)a->codes; p.b_codes = (const uint8_t*)b->codes;
    p.a_rows = M; p.b_rows = N;
    p.M = M; p.N = N; p.K = K;
    p.offsets = nullptr; p.groups = 1;
    p.sfa = a->sf; p.sfb = b->sf; p.sfb_group_stride = 0;
    p.amax_a = a->amax; p.amax_b = b->amax;
    p.c = c; p.ldc = ldc;
    p.c_amax = c_amax;
    p.vec_store = aligned16(c) && (ldc * esz) % 16 == 0;
    if (c_amax != nullptr) {
        if (((uintptr_t)c_amax & 3u) != 0) return fail(NVFP4_ERR_ALIGN, "c_amax not 4-byte aligned");
        NVFP4_TRY(cuda_call(cudaMemsetAsync(c_amax, 0, sizeof(float), stream), "memset c_amax"));
    }
    CUtensorMap mc;
    bool tma_store = false;
    std::memset(&mc, 0, sizeof(mc));
    NVFP4_TRY(make_store_map(&mc, c, M, N, ldc, c_dtype == NVFP4_OUT_FP32, &tma_store));
    const int64_t tiles = cdiv(M, G_BM) * cdiv(N, G_BN);
    const int64_t pair_tiles = cdiv(M, 2 * G_BM) * cdiv(N, G_BN);
    return launch_gemm(ma, mb, mc, p, tiles, pair_tiles, sms, c_dtype, tma_store, pair, stream, dev, G_DENSE);
}

nvfp4_status nvfp4_grouped_gemm(const nvfp4_tensor* a, const int64_t* offsets, int32_t num_groups,
                                const nvfp4_tensor* b, int64_t n, void* c, int64_t ldc, nvfp4_out_dtype c_dtype,
                                float* c_amax, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_operand(a, "a"));
    NVFP4_TRY(check_operand(b, "b"));
    if (offsets == nullptr) return fail(NVFP4_ERR_NULL, "offsets is NULL");
    if (num_groups < 1 || num_groups > NVFP4_MAX_GROUPS) return fail(NVFP4_ERR_LIMIT, "num_groups must be in [1, %d]", NVFP4_MAX_GROUPS);
    const int64_t R = a->rows, K = a->cols;
    if (b->rows != n || b->cols != K) return fail(NVFP4_ERR_SHAPE, "b must be [n, K] per expert");
    if (K % 16 != 0 || K == 0) return fail(NVFP4_ERR_SHAPE, "K=%lld must be a positive multiple of 16", (long long)K);
    if (n < 1) return fail(NVFP4_ERR_SHAPE, "n must be >= 1");
    if (c_dtype != NVFP4_OUT_BF16 && c_dtype != NVFP4_OUT_FP32) return fail(NVFP4_ERR_SHAPE, "bad output dtype");
    if (ldc < n) return fail(NVFP4_ERR_SHAPE, "ldc < n");
    if (R >= (int64_t(1) << 31) - 128 * (int64_t)num_groups || n * (int64_t)num_groups >= (int64_t(1) << 31))
        return fail(NVFP4_ERR_LIMIT, "rows or experts*n >= 2^31");
    if (R == 0) return NVFP4_OK;
    if (c == nullptr) return fail(NVFP4_ERR_NULL, "c is NULL");
    const int esz = c_dtype == NVFP4_OUT_FP32 ? 4 : 2;
    if (((uintptr_t)c % esz) != 0) return fail(NVFP4_ERR_ALIGN, "c is not aligned to its element size");
    int sms = 0, dev = 0;
    NVFP4_TRY(check_device(&sms, &dev));
    const bool copy_ab = K % 32 != 0;     // as for nvfp4_gemm
    const bool pair = use_pair() && !copy_ab;
    CUtensorMap ma, mb;
    std::memset(&ma, 0, sizeof(ma));
    std::memset(&mb, 0, sizeof(mb));
    if (!copy_ab) {
        NVFP4_TRY(make_code_map(&ma, a->codes, R, K / 2, G_BM));
        NVFP4_TRY(make_code_map(&mb, b->codes, n * num_groups, K / 2, pair ? G_BN / 2 : G_BN));
    }
    GemmParams p{};
    p.copy_ab = copy_ab;
    p.a_codes = (const uint8_t*)a->codes; p.b_codes = (const uint8_t*)b->codes;
    p.a_rows = R; p.b_rows = n * num_groups;
    p.M = R; p.N = n; p.K = K;
    p.offsets = offsets; p.groups = num_groups;
    p.sfa = a->sf; p.sfb = b->sf; p.sfb_group_stride = sf_bytes(n, K);
    p.amax_a = a->amax; p.amax_b = b->amax;
    p.c = c; p.ldc = ldc;
    p.c_amax = c_amax;
    p.vec_store = aligned16(c) && (ldc * esz) % 16 == 0;
    if (c_amax != nullptr) {
        if (((uintptr_t)c_amax & 3u) != 0) return fail(NVFP4_ERR_ALIGN, "c_amax not 4-byte aligned");
        NVFP4_TRY(cuda_call(cudaMemsetAsync(c_amax, 0, sizeof(float) * num_groups, stream), "memset c_amax"));
    }
    CUtensorMap mc;
    bool tma_store = false;
    std::memset(&mc, 0, sizeof(mc));
    NVFP4_TRY(make_store_map(&mc, c, R, n, ldc, c_dtype == NVFP4_OUT_FP32, &tma_store));
    // tiles depend on the group sizes (device data): the grid is the SM count
    return launch_gemm(ma, mb, mc, p, sms, sms / 2, sms, c_dtype, tma_store, pair, stream, dev, G_MGROUP);
}

nvfp4_status nvfp4_grouped_gemm_k(const nvfp4_tensor* a, const nvfp4_tensor* b, const int64_t* offsets,
                                  int32_t num_groups, void* c, int64_t ldc, nvfp4_out_dtype c_dtype, float* c_amax,
                                  nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    NVFP4_TRY(check_operand(a, "a"));
    NVFP4_TRY(check_operand(b, "b"));
    if (offsets == nullptr) return fail(NVFP4_ERR_NULL, "offsets is NULL");
    if (num_groups < 1 || num_groups > NVFP4_MAX_GROUPS)
        return fail(NVFP4_ERR_LIMIT, "num_groups must be in [1, %d]", NVFP4_MAX_GROUPS);
    const int64_t M = a->rows, N = b->rows, KT = a->cols;
    if (b->cols != KT) return fail(NVFP4_ERR_SHAPE, "a->cols=%lld != b->cols=%lld", (long long)KT, (long long)b->cols);
    if (KT % 64 != 0 || KT == 0) return fail(NVFP4_ERR_SHAPE, "K=%lld must be a positive multiple of 64", (long long)KT);
    if (c_dtype != NVFP4_OUT_BF16 && c_dtype != NVFP4_OUT_FP32) return fail(NVFP4_ERR_SHAPE, "bad output dtype");
    if (ldc < N) return fail(NVFP4_ERR_SHAPE, "ldc < N");
    if (M * (int64_t)num_groups >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || KT >= (int64_t(1) << 31))
        return fail(NVFP4_ERR_LIMIT, "groups * M, N or K >= 2^31");
    if (M == 0 || N == 0) return NVFP4_OK;
    if (c == nullptr) return fail(NVFP4_ERR_NULL, "c is NULL");
    const int esz = c_dtype == NVFP4_OUT_FP32 ? 4 : 2;
    if (((uintptr_t)c % esz) != 0) return fail(NVFP4_ERR_ALIGN, "c is not aligned to its element size");
    int sms = 0, dev = 0;
    NVFP4_TRY(check_device(&sms, &dev));
    const bool pair = use_pair();
    CUtensorMap ma, mb;
    NVFP4_TRY(make_code_map(&ma, a->codes, M, KT / 2, G_BM));
    NVFP4_TRY(make_code_map(&mb, b->codes, N, KT / 2, pair ? G_BN / 2 : G_BN));
    GemmParams p{};
    p.M = M; p.N = N; p.K = KT;
    p.offsets = offsets; p.groups = num_groups;
    p.sfa = a->sf; p.sfb = b->sf; p.sfb_group_stride = 0;
    p.amax_a = a->amax; p.amax_b = b->amax;
    p.c = c; p.ldc = ldc;
    p.c_amax = c_amax;
    p.vec_store = aligned16(c) && (ldc * esz) % 16 == 0;
    if (c_amax != nullptr) {
        if (((uintptr_t)c_amax & 3u) != 0) return fail(NVFP4_ERR_ALIGN, "c_amax not 4-byte aligned");
        NVFP4_TRY(cuda_call(cudaMemsetAsync(c_amax, 0, sizeof(float) * num_groups, stream), "memset c_amax"));
    }
    CUtensorMap mc;
    bool tma_store = false;
    std::memset(&mc, 0, sizeof(mc));
    NVFP4_TRY(make_store_map(&mc, c, M * num_groups, N, ldc, c_dtype == NVFP4_OUT_FP32, &tma_store));
    const int64_t tiles = (int64_t)num_groups * cdiv(M, G_BM) * cdiv(N, G_BN);
    const int64_t pair_tiles = (int64_t)num_groups * cdiv(M, 2 * G_BM) * cdiv(N, G_BN);
    return launch_gemm(ma, mb, mc, p, tiles, pair_tiles, sms, c_dtype, tma_store, pair, stream, dev, G_KGROUP);
}

nvfp4_status nvfp4_device_status(int32_t* flags) {
    NVFP4_INJECT_CHECK();
    if (flags == nullptr) return fail(NVFP4_ERR_NULL, "flags is NULL");
    NVFP4_TRY(check_device());
    NVFP4_TRY(cuda_call(cudaDeviceSynchronize(), "cudaDeviceSynchronize"));
    int v = 0, zero = 0;
    NVFP4_TRY(cuda_call(cudaMemcpyFromSymbol(&v, g_dev_status, sizeof(int)), "read status"));
    NVFP4_TRY(cuda_call(cudaMemcpyToSymbol(g_dev_status, &zero, sizeof(int)), "clear status"));
    *flags = v;
    return (v & DEV_TIMEOUT) ? NVFP4_ERR_TIMEOUT : NVFP4_OK;
}

nvfp4_status nvfp4_debug_wait_timeout(int64_t timeout_ns, nvfp4_stream_t stream) {
    NVFP4_INJECT_CHECK();
    if (timeout_ns <= 0 || timeout_ns > 10000000000ll) return fail(NVFP4_ERR_SHAPE, "timeout must be in (0, 10 s]");
    NVFP4_TRY(check_device());
    k_wait_probe<<<1, 32, 0, stream>>>((uint64_t)timeout_ns);
    return launched("k_wait_probe");
}

}  // extern "C"
