// Entry points of the BitLinear matmul: argument checks, engine choice,
// status reporting.  The kernels live in pack.cu, quant.cu, gemv.cu and
// gemm.cu.
#include <atomic>

#include "bl_device.cuh"

namespace bl {
cudaError_t launch_gemv(const int8_t *q, const float *tok_scale, const uint8_t *packed,
                        const float *gamma, int M, int N, int K, __nv_bfloat16 *out,
                        int32_t *acc_out, cudaStream_t st, int num_sms);
cudaError_t launch_gemm(const int8_t *q, const float *tok_scale, const uint8_t *packed,
                        const float *gamma, int M, int N, int K, __nv_bfloat16 *out,
                        int32_t *acc_out, cudaStream_t st, uint32_t wait_limit, int split);
cudaError_t launch_gemm16(const void *q16, const float *tok_scale, const uint8_t *packed,
                          const float *gamma, int M, int N, int K, __nv_bfloat16 *out,
                          int32_t *acc_out, cudaStream_t st, uint32_t wait_limit, int split);
cudaError_t gemm_status(unsigned int *out, cudaStream_t st);

namespace {
constexpr uint32_t kDefaultWaitLimit = 1u << 22;
std::atomic<uint32_t> g_wait_limit{kDefaultWaitLimit};
int g_sms[64] = {0};

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!g_sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        g_sms[dev] = v;
    }
    return g_sms[dev];
}
}  // namespace
}  // namespace bl

extern "C" const char *bitlinear_status_string(int status) {
    switch (status) {
        case BITLINEAR_OK: return "ok";
        case BITLINEAR_ERR_INVALID_ARG: return "invalid argument";
        case BITLINEAR_ERR_UNSUPPORTED: return "unsupported device or shape";
        case BITLINEAR_ERR_CUDA: return "CUDA runtime error";
        case BITLINEAR_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
        case BITLINEAR_ERR_STATE: return "a pending factor buffer was produced into again";
        case BITLINEAR_ERR_BOUNDS: return "a device bounds check failed (debug build)";
        default: return "unknown status";
    }
}

extern "C" int bitlinear_version(void) { return 101; }

#ifdef BITLINEAR_DEBUG
#include <cstdio>
#include <mutex>
#include <vector>
namespace bl {
namespace {
struct DebugEntry {
    DebugTake take;
    const char *unit;
};
// Function-local statics: the units register from their static
// initialisers, in whatever order the loader runs them.
std::vector<DebugEntry> &debug_units() {
    static std::vector<DebugEntry> v;
    return v;
}
std::mutex &debug_mutex() {
    static std::mutex m;
    return m;
}
// Records a failed check without any memory access: the reporting path,
// testable without an out-of-bounds access.
__global__ void debug_selftest_kernel() { dbg_ok(false, 31u); }
}  // namespace
void debug_register(DebugTake take, const char *unit) {
    std::lock_guard<std::mutex> lock(debug_mutex());
    debug_units().push_back({take, unit});
}
}  // namespace bl
#endif

extern "C" bitlinear_status_t bitlinear_debug_selftest(void *stream) {
#ifdef BITLINEAR_DEBUG
    bl::debug_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>();
    return cudaGetLastError() == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
#else
    (void)stream;
    return BITLINEAR_ERR_UNSUPPORTED;
#endif
}

namespace bl {
uint32_t current_wait_limit() { return g_wait_limit.load(); }
}  // namespace bl

extern "C" void bitlinear_set_wait_limit(uint32_t iterations) {
    bl::g_wait_limit.store(iterations ? iterations : bl::kDefaultWaitLimit);
}

// Batches up to gemv_max_tokens run on the decode GEMV engine (16-token
// chunks in one launch, at most kGemvMaxM); larger ones on the tensor-core
// GEMM.
constexpr int64_t kGemvMaxM = 64;
namespace bl {
namespace {
std::atomic<int32_t> g_gemv_max_tokens{-1};  // -1: the measured default below
std::atomic<int32_t> g_split_k{0};

// The default engine choice (B300 measurements, weights from HBM): the GEMV
// up to 32 tokens (two 16-token chunks); at 33-48 tokens (three chunks) the
// split-K GEMM on widened activations for matrices with K >= 8192, N <= K
// and at least 2^24 weights - 8192x28672 68 against 88 us, 8192x8192 25.0
// against 27.4, 3200x8640 15.1 against 17.5 - and the GEMV elsewhere
// (28672x8192 79 against 81, 1024x8192 8.5 against 10.7, 2560x6912 11.7
// against 12.5, 6912x2560 10.8 against 13.2); at 49-64 tokens (four chunks)
// the GEMM where K is large and the matrix is big - 8192x8192 34.8 us
// against 43.0, 8192x28672 94 against 125-141, 2560x6912 18.4 against 19.7
// - and the GEMV elsewhere (2560x2560 12.3 against 14.3, 6912x2560 16.4
// against 18.4, 1024x8192 14.3 against 16.4); the GEMM above 64.
bool use_gemv(int64_t M, int64_t N, int64_t K) {
    const int32_t forced = g_gemv_max_tokens.load();
    if (forced >= 0) return M <= forced;
    if (M > kGemvMaxM) return false;
    if (M > 48 && K >= 6912 && N * K >= (1ll << 24)) return false;
    if (M > 32 && K >= 8192 && N <= K && N * K >= (1ll << 24)) return false;
    return true;
}
}  // namespace
}  // namespace bl

extern "C" bitlinear_status_t bitlinear_set_engine(int32_t gemv_max_tokens, int32_t split_k) {
    if (gemv_max_tokens < -1 || gemv_max_tokens > kGemvMaxM || split_k < 0 || split_k > 16)
        return BITLINEAR_ERR_INVALID_ARG;
    bl::g_gemv_max_tokens.store(gemv_max_tokens);
    bl::g_split_k.store(split_k);
    return BITLINEAR_OK;
}

extern "C" bitlinear_status_t bitlinear_forward(const int8_t *q, const float *tok_scale,
                                                const uint8_t *packed, const float *gamma,
                                                int64_t M, int64_t N, int64_t K, void *out_bf16,
                                                int32_t *acc_out, void *stream) {
    using namespace bl;
    if (M < 0 || N < 1 || K < 16 || (K % 16) != 0 || K > 65536 || N > (1ll << 30) ||
        M > (1ll << 30))
        return BITLINEAR_ERR_INVALID_ARG;
    if (M == 0) return BITLINEAR_OK;
    if (!q || !tok_scale || !packed || !gamma || !out_bf16) return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned4(tok_scale) || !aligned16(packed) || !aligned4(gamma) ||
        !aligned16(out_bf16) || (acc_out && !aligned16(acc_out)))
        return BITLINEAR_ERR_INVALID_ARG;
    const bool gemv = use_gemv(M, N, K);
    if ((N + 15) / 16 > 65535 * 4 && gemv) return BITLINEAR_ERR_UNSUPPORTED;
    if ((M + 63) / 64 > 65535) return BITLINEAR_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto *out = static_cast<__nv_bfloat16 *>(out_bf16);
    cudaError_t e;
    if (gemv)  // the decode GEMV, in 16-token chunks above 16
        e = launch_gemv(q, tok_scale, packed, gamma, static_cast<int>(M), static_cast<int>(N),
                        static_cast<int>(K), out, acc_out, st, num_sms());
    else
        e = launch_gemm(q, tok_scale, packed, gamma, static_cast<int>(M), static_cast<int>(N),
                        static_cast<int>(K), out, acc_out, st, g_wait_limit.load(), g_split_k.load());
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" bitlinear_status_t bitlinear_forward_f16(const void *q_f16, const float *tok_scale,
                                                    const uint8_t *packed, const float *gamma,
                                                    int64_t M, int64_t N, int64_t K, void *out_bf16,
                                                    int32_t *acc_out, void *stream) {
    using namespace bl;
    if (M < 0 || N < 1 || K < 16 || (K % 16) != 0 || K > 65536 || N > (1ll << 30) || M > (1ll << 30))
        return BITLINEAR_ERR_INVALID_ARG;
    if (M == 0) return BITLINEAR_OK;
    if (!q_f16 || !tok_scale || !packed || !gamma || !out_bf16) return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(q_f16) || !aligned4(tok_scale) || !aligned16(packed) || !aligned4(gamma) ||
        !aligned16(out_bf16) || (acc_out && !aligned16(acc_out)))
        return BITLINEAR_ERR_INVALID_ARG;
    if ((M + 63) / 64 > 65535 || M > 0x7fffffffll) return BITLINEAR_ERR_UNSUPPORTED;
    const cudaError_t e =
        launch_gemm16(q_f16, tok_scale, packed, gamma, static_cast<int>(M), static_cast<int>(N),
                      static_cast<int>(K), static_cast<__nv_bfloat16 *>(out_bf16), acc_out,
                      static_cast<cudaStream_t>(stream), g_wait_limit.load(), g_split_k.load());
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" bitlinear_status_t bitlinear_check_status(void *stream) {
    unsigned int v = 0;
    if (bl::gemm_status(&v, static_cast<cudaStream_t>(stream)) != cudaSuccess) return BITLINEAR_ERR_CUDA;
#ifdef BITLINEAR_DEBUG
    {
        std::lock_guard<std::mutex> lock(bl::debug_mutex());
        unsigned int bounds = 0u;
        for (const auto &u : bl::debug_units()) {
            unsigned int w = 0u;
            if (u.take(&w, static_cast<cudaStream_t>(stream)) != cudaSuccess) return BITLINEAR_ERR_CUDA;
            if (w) std::fprintf(stderr, "bitlinear: device bounds check failed in %s (site bits 0x%08x)\n", u.unit, w);
            bounds |= w;
        }
        if (bounds) return BITLINEAR_ERR_BOUNDS;
    }
#endif
    // bit 0: a bounded wait gave up; bit 1: a pending factor buffer was produced into
    if (v & 1u) return BITLINEAR_ERR_TIMEOUT;
    return v ? BITLINEAR_ERR_STATE : BITLINEAR_OK;
}
