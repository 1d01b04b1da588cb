// Offline weight packer: absmean scale and 2-bit ternary codes.
//
// BitNet b1.58 (cheatsheet.md, "BitNet b1.58とは？"): weights are divided by
// their mean absolute value and rounded to the nearest integer in
// {-1, 0, +1}.  asi.tokyo, "マイクロソフトが偶然に作った史上最も効率的なAI"
// (2025-04-27), the paragraph on running the model on a GPU: four ternary
// weights are packed into each byte.
//
// gamma = mean|W| is computed exactly, so it does not depend on the order of
// a floating-point reduction (a different order would move weights across
// rounding boundaries).  Every fp32 |w| equals mant * 2^(e-150) with a
// 24-bit integer mant and biased exponent e (subnormals: e = 1, no hidden
// bit).  Integer atomics add `mant` into one of 256 64-bit buckets chosen by
// e; a single thread then forms the exact sum as a multi-word integer,
// rounds it once to double, divides by N*K in double and rounds to float.
#include <mutex>

#include "bl_device.cuh"

namespace bl {
namespace {

constexpr int kBuckets = 256;

__global__ void __launch_bounds__(256) absmean_buckets_kernel(const float4 *__restrict__ w,
                                                              int64_t n4,
                                                              unsigned long long *buckets) {
    __shared__ unsigned long long sb[kBuckets];
    for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) sb[i] = 0ull;
    __syncthreads();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += stride) {
        float4 v = w[i];
        float a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t bits = __float_as_uint(a[j]) & 0x7fffffffu;
            uint32_t e = bits >> 23;
            uint32_t mant = bits & 0x7fffffu;
            if (e != 0) mant |= 0x800000u;
            uint32_t idx = e == 0 ? 1u : e;  // subnormals share the scale of e = 1
            if (mant) atomicAdd(&sb[idx], static_cast<unsigned long long>(mant));
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kBuckets; i += blockDim.x)
        if (sb[i]) atomicAdd(&buckets[i], sb[i]);
}

// Exact sum -> double (round to nearest even) -> / count -> float.
__global__ void gamma_finish_kernel(const unsigned long long *buckets, int64_t count,
                                    float *gamma_out) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    // value = sum_e B[e] * 2^(e-1) in units of 2^-149; 12 x 32-bit limbs.
    uint32_t limb[12];
    for (int i = 0; i < 12; ++i) limb[i] = 0;
    bool nonfinite = buckets[255] != 0ull;
    for (int e = 1; e < 255; ++e) {
        unsigned long long b = buckets[e];
        if (!b) continue;
        int s = e - 1;
        int li = s >> 5, sh = s & 31;
        // b << sh spans up to three limbs
        const uint32_t p0 = static_cast<uint32_t>(b << sh);
        const uint32_t p1 = static_cast<uint32_t>(sh == 0 ? (b >> 32) : (b >> (32 - sh)));
        const uint32_t p2 = sh == 0 ? 0u : static_cast<uint32_t>(b >> (64 - sh));
        uint32_t add[3] = {p0, p1, p2};
        unsigned long long carry = 0;
        for (int k = li; k < 12; ++k) {
            unsigned long long sum = static_cast<unsigned long long>(limb[k]) + carry +
                                     (k - li < 3 ? add[k - li] : 0u);
            limb[k] = static_cast<uint32_t>(sum);
            carry = sum >> 32;
            if (k - li >= 2 && carry == 0) break;
        }
    }
    // highest set bit
    int top = -1;
    for (int k = 11; k >= 0 && top < 0; --k)
        if (limb[k]) top = k * 32 + 31 - __clz(limb[k]);
    double s;
    if (top < 0) {
        s = 0.0;
    } else if (top < 53) {
        unsigned long long v = (static_cast<unsigned long long>(limb[1]) << 32) | limb[0];
        s = ldexp(static_cast<double>(v), -149);  // exact: v < 2^53
    } else {
        // mantissa = bits [top-52, top]; round bit = top-53; sticky below.
        auto bit = [&](int i) -> uint32_t { return (limb[i >> 5] >> (i & 31)) & 1u; };
        unsigned long long m = 0;
        for (int i = top; i >= top - 52; --i) m = (m << 1) | bit(i);
        uint32_t rb = bit(top - 53);
        bool sticky = false;
        for (int i = top - 54; i >= 0 && !sticky; --i) sticky = bit(i) != 0;
        int exp = top - 52;
        if (rb && (sticky || (m & 1ull))) {
            ++m;
            if (m == (1ull << 53)) { m >>= 1; ++exp; }
        }
        s = ldexp(static_cast<double>(m), exp - 149);
    }
    double mean = __ddiv_rn(s, static_cast<double>(count));
    float g = __double2float_rn(mean);
    if (nonfinite) g = __int_as_float(0x7fc00000);
    *gamma_out = g;
}

// One thread per 16-byte lane chunk of the packed layout: lane 4g+t of tile
// (row group r, k block c) holds rows 16r+g and 16r+g+8 over
// k in [128c + 32t, 128c + 32t + 32).  Word 2P+u holds row 16r+8u+g and
// k = 128c + 32t + 16P + j (j < 16); inside the word the code of j sits at
// bit 16*(j%2) + 2*(2*((j%16)/4) + (j%4)/2).
template <bool kFromFloat>
__global__ void __launch_bounds__(256) pack_kernel(const void *__restrict__ src, int64_t N,
                                                   int64_t K, int64_t KT, int64_t nchunks,
                                                   float eps, const float *__restrict__ gamma,
                                                   uint4 *__restrict__ packed) {
    int64_t id = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (id >= nchunks) return;
    const int lane = static_cast<int>(id & 31);
    const int64_t tile = id >> 5;
    const int64_t r = tile / KT, c = tile % KT;
    const int g = lane >> 2, t = lane & 3;
    float d = 1.0f;
    if (kFromFloat) d = __fadd_rn(*gamma, eps);
    uint32_t words[4];
#pragma unroll
    for (int P = 0; P < 2; ++P) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t n = 16 * r + 8 * u + g;
            const int64_t k0 = 128 * c + 32 * t + 16 * P;
            int codes[16];
            if (n < N && k0 < K && dbg_ok(fits(n * K + k0, 16, N * K), 0)) {  // K % 16 == 0: all 16 in range
                if (kFromFloat) {
                    const float4 *row =
                        reinterpret_cast<const float4 *>(static_cast<const float *>(src) + n * K + k0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float4 v = __ldg(row + q);
                        float a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            int iv = __float2int_rn(__fdiv_rn(a[e], d));
                            iv = iv > 1 ? 1 : (iv < -1 ? -1 : iv);
                            codes[4 * q + e] = iv + 1;
                        }
                    }
                } else {
                    uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const int8_t *>(src) +
                                                                    n * K + k0));
                    uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            int iv = static_cast<int8_t>((a[q] >> (8 * e)) & 0xffu);
                            iv = iv > 1 ? 1 : (iv < -1 ? -1 : iv);
                            codes[4 * q + e] = iv + 1;
                        }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) codes[j] = 1;
            }
            uint32_t wv = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int p = 2 * (j >> 2) + ((j & 3) >> 1);
                const int bitpos = 16 * (j & 1) + 2 * p;
                wv |= static_cast<uint32_t>(codes[j]) << bitpos;
            }
            words[2 * P + u] = wv;
        }
    }
    // the packed layout holds RGN * KT tiles of 32 chunks
    if (dbg_ok(fits(id, 1, (N + 15) / 16 * KT * 32), 1)) packed[id] = make_uint4(words[0], words[1], words[2], words[3]);
}

// Per-device bucket workspace, allocated on first use and kept until exit.
std::mutex g_ws_mutex;
unsigned long long *g_ws[64] = {nullptr};

cudaError_t workspace(unsigned long long **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    if (!g_ws[dev]) {
        e = cudaMalloc(&g_ws[dev], kBuckets * sizeof(unsigned long long));
        if (e != cudaSuccess) {
            g_ws[dev] = nullptr;
            return e;
        }
    }
    *out = g_ws[dev];
    return cudaSuccess;
}

bool shape_ok(int64_t N, int64_t K) { return N >= 1 && K >= 16 && (K % 16) == 0 && N <= (1ll << 31) && K <= (1ll << 31); }

// Each exponent bucket gathers up to N*K mantissas below 2^24; keeping
// N*K <= 2^40 keeps every 64-bit counter below 2^64.
constexpr int64_t kMaxSumElems = 1ll << 40;

// The matmul kernels read packed weights before they wait for the kernel
// that precedes them in the stream (weights are static, so their loads can
// overlap that kernel).  The packers must therefore hand over weights that
// are complete and visible: pack_kernel is an ordinary launch that never lets
// its dependents start early, and it is followed by publish_kernel, another
// ordinary launch, which starts only once pack_kernel has finished and its
// writes are visible.  A kernel launched after the packer can start early
// only relative to publish_kernel, when the packed bytes are already final.
__global__ void publish_kernel() {}

cudaError_t launch_pack(const void *src, bool from_float, int64_t N, int64_t K, float eps,
                        const float *gamma, uint8_t *packed, cudaStream_t st) {
    const int64_t Np = (N + 15) / 16 * 16, KT = (K + 127) / 128;
    const int64_t nchunks = (Np / 16) * KT * 32;
    const unsigned blocks = static_cast<unsigned>((nchunks + 255) / 256);
    if (from_float)
        pack_kernel<true><<<blocks, 256, 0, st>>>(src, N, K, KT, nchunks, eps, gamma,
                                                  reinterpret_cast<uint4 *>(packed));
    else
        pack_kernel<false><<<blocks, 256, 0, st>>>(src, N, K, KT, nchunks, eps, gamma,
                                                   reinterpret_cast<uint4 *>(packed));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    publish_kernel<<<1, 32, 0, st>>>();
    return cudaGetLastError();
}

// Original binary BitNet (lumen-it.ai BitNet article): signum weights, one
// bit each (1 for W > 0, 0 otherwise), in tiles of 16 rows x 256 k: lane
// 4g+t holds rows g, g+8 at k in [64t, 64t+64), word 2P+u (row g+8u, k half
// P) holds k = 64t + 32P + j at bit 16(j%2) + 2(j/4) + (j%4)/2.  One thread
// per output word reads its row's 32 consecutive floats.
__global__ void __launch_bounds__(256) pack1_kernel(const float *__restrict__ W, int64_t N, int64_t K, int64_t KT1,
                                                    int64_t nwords, uint32_t *__restrict__ out) {
    const int64_t wi = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (wi >= nwords) return;
    const int64_t tile = wi / 128;
    const int lw = static_cast<int>(wi % 128);
    const int64_t r = tile / KT1, c = tile % KT1;
    const int lane = lw / 4, wd = lw % 4;
    const int P = wd / 2, u = wd % 2, g = lane / 4, t = lane % 4;
    const int64_t n = 16 * r + 8 * u + g;
    const int64_t kb = 256 * c + 64 * t + 32 * P;
    uint32_t word = 0;
    if (n < N) {
        const float *row = W + n * K;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const int64_t k = kb + j;
            if (k < K && dbg_ok(fits(n * K + k, 1, N * K), 2) && row[k] > 0.0f)
                word |= 1u << (16 * (j % 2) + 2 * (j / 4) + (j % 4) / 2);
        }
    }
    if (dbg_ok(fits(wi, 1, (N + 15) / 16 * KT1 * 128), 3)) out[wi] = word;
}

}  // namespace
}  // namespace bl

extern "C" size_t bitlinear_packed1_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1) return 0;
    return static_cast<size_t>((N + 15) / 16 * 16 * ((K + 255) / 256 * 256) / 8);
}

extern "C" bitlinear_status_t bitlinear_pack_binary(const float *W, int64_t N, int64_t K, int64_t groups,
                                                    uint8_t *packed1, float *beta, void *stream) {
    using namespace bl;
    if (!W || !packed1 || !beta || !shape_ok(N, K) || groups < 1 || N % groups != 0)
        return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(packed1) || !aligned4(beta)) return BITLINEAR_ERR_INVALID_ARG;
    if (N * K > kMaxSumElems || groups > 65536) return BITLINEAR_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long *ws = nullptr;
    if (workspace(&ws) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // beta_g = mean |W| over the g-th block of N/G rows, each by the exact
    // bucket sum (the blocks are contiguous and 64-byte aligned: K % 16 == 0)
    const int64_t per = N / groups * K;
    for (int64_t gi = 0; gi < groups; ++gi) {
        if (cudaMemsetAsync(ws, 0, kBuckets * sizeof(unsigned long long), st) != cudaSuccess)
            return BITLINEAR_ERR_CUDA;
        const int64_t n4 = per / 4, want = (n4 + 255) / 256;
        const unsigned blocks = static_cast<unsigned>(want < sms * 8 ? (want < 1 ? 1 : want) : sms * 8);
        absmean_buckets_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(W + gi * per), n4, ws);
        gamma_finish_kernel<<<1, 32, 0, st>>>(ws, per, beta + gi);
        if (cudaGetLastError() != cudaSuccess) return BITLINEAR_ERR_CUDA;
    }
    const int64_t KT1 = (K + 255) / 256;
    const int64_t nwords = static_cast<int64_t>(bitlinear_packed1_bytes(N, K)) / 4;
    pack1_kernel<<<static_cast<unsigned>((nwords + 255) / 256), 256, 0, st>>>(W, N, K, KT1, nwords,
                                                                             reinterpret_cast<uint32_t *>(packed1));
    if (cudaGetLastError() != cudaSuccess) return BITLINEAR_ERR_CUDA;
    publish_kernel<<<1, 32, 0, st>>>();  // as launch_pack: packed bytes final before any dependent starts
    return cudaGetLastError() == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" size_t bitlinear_packed_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1) return 0;
    const int64_t Np = (N + 15) / 16 * 16, Kp = (K + 127) / 128 * 128;
    return static_cast<size_t>(Np * Kp / 4);
}

extern "C" bitlinear_status_t bitlinear_pack_weights(const float *W, int64_t N, int64_t K,
                                                     float eps, uint8_t *packed, float *gamma,
                                                     void *stream) {
    using namespace bl;
    if (!W || !packed || !gamma || !shape_ok(N, K)) return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(packed) || !aligned4(gamma)) return BITLINEAR_ERR_INVALID_ARG;
    if (N * K > kMaxSumElems) return BITLINEAR_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long *ws = nullptr;
    if (workspace(&ws) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, kBuckets * sizeof(unsigned long long), st) != cudaSuccess)
        return BITLINEAR_ERR_CUDA;
    const int64_t n4 = N * K / 4;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t want = (n4 + 255) / 256;
    unsigned blocks = static_cast<unsigned>(want < sms * 8 ? (want < 1 ? 1 : want) : sms * 8);
    absmean_buckets_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(W), n4, ws);
    if (cudaGetLastError() != cudaSuccess) return BITLINEAR_ERR_CUDA;
    gamma_finish_kernel<<<1, 32, 0, st>>>(ws, N * K, gamma);
    if (cudaGetLastError() != cudaSuccess) return BITLINEAR_ERR_CUDA;
    if (launch_pack(W, true, N, K, eps, gamma, packed, st) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    return BITLINEAR_OK;
}

extern "C" bitlinear_status_t bitlinear_pack_ternary(const int8_t *Wq, int64_t N, int64_t K,
                                                     uint8_t *packed, void *stream) {
    using namespace bl;
    if (!Wq || !packed || !shape_ok(N, K)) return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(Wq) || !aligned16(packed)) return BITLINEAR_ERR_INVALID_ARG;
    if (launch_pack(Wq, false, N, K, 0.0f, nullptr, packed, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return BITLINEAR_ERR_CUDA;
    return BITLINEAR_OK;
}

// ---------------------------------------------------------------------------
// Packing without any allocation.
//
// Some callers cannot call cudaMalloc: code running under an allocator that
// owns all device memory (a serving runtime's arena, a memory pool that must
// not be fragmented), or code that must not take the driver's allocation
// lock at that moment.  bitlinear_pack_weights allocates its 2 KB bucket
// workspace on the first call per device; this variant instead keeps the
// 256 exponent buckets in the fixed device array below, which every GPU
// that loads the library holds until the process exits.
// ---------------------------------------------------------------------------
namespace bl {
namespace {

// 256 64-bit counters (2 KB): the whole scratch of the absmean sum.
static __device__ __align__(256) unsigned long long g_noalloc_buckets[kBuckets];

std::mutex g_noalloc_mutex;
unsigned long long *g_noalloc_ptr[64] = {nullptr};

// Device address of g_noalloc_buckets on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in;
// kernels must be given this address.
cudaError_t noalloc_scratch(unsigned long long **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_buckets);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<unsigned long long *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace bl

extern "C" bitlinear_status_t bitlinear_pack_weights_noalloc(const float *W, int64_t N, int64_t K,
                                                             float eps, uint8_t *packed,
                                                             float *gamma, void *stream) {
    using namespace bl;
    if (!W || !packed || !gamma || !shape_ok(N, K)) return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(packed) || !aligned4(gamma)) return BITLINEAR_ERR_INVALID_ARG;
    if (N * K > kMaxSumElems) return BITLINEAR_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long *ws = nullptr;
    if (noalloc_scratch(&ws) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    // The array keeps the previous call's sums: clear it first.
    if (cudaMemsetAsync(ws, 0, kBuckets * sizeof(unsigned long long), st) != cudaSuccess)
        return BITLINEAR_ERR_CUDA;
    const int64_t n4 = N * K / 4;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 148;
    const int64_t want = (n4 + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(want < sms * 8 ? (want < 1 ? 1 : want) : sms * 8);
    absmean_buckets_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(W), n4, ws);
    if (cudaGetLastError() != cudaSuccess) return BITLINEAR_ERR_CUDA;
    gamma_finish_kernel<<<1, 32, 0, st>>>(ws, N * K, gamma);
    if (cudaGetLastError() != cudaSuccess) return BITLINEAR_ERR_CUDA;
    if (launch_pack(W, true, N, K, eps, gamma, packed, st) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    return BITLINEAR_OK;
}
