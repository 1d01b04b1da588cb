// Fused RMSNorm + per-token absmax int8 quantisation of activations.
//
// BitNet b1.58 (cheatsheet.md, "BitNet b1.58とは？"): activations are scaled
// per token into the 8-bit range; the LLaMA-style parts include RMSNorm.
// lumen-it.ai: absmax quantisation of activations.
//
// Per token (v_k = x_k * gain_k in fp32, exact for bf16 inputs):
//   mx = max(max |v_k|, 1e-5f);  c = 127 / mx  (fp32);  q_k = rint(v_k * c)
//   tok_scale = rms^-1 * mx / 127, rms = sqrt(sum v_k^2 / K + eps)
// RMSNorm's positive factor cancels inside absmax, so q is decided by fp32
// products of the raw inputs only: it is the same on every device and in
// any reduction order.  The sum of squares is accumulated as an unevaluated
// pair of floats (two-sum plus the exact product residual) and combined
// across threads the same way; the scale is then formed with correctly
// rounded fp32 operations (B300's FP64 units are far too slow for this
// path), within a few 1e-7 of the double-precision definition.
#include "bl_device.cuh"

namespace bl {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Compensated fp32 sum: the squares of fp32 products get their exact
// rounding residual, the additions an error-free two-sum.
struct FF2 {
    float hi = 0.0f, lo = 0.0f;
    __device__ __forceinline__ void add(float p, float pe = 0.0f) {
        const float s = __fadd_rn(hi, p);
        const float bp = __fsub_rn(s, hi);
        lo = __fadd_rn(lo, __fadd_rn(__fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp)), pe));
        hi = s;
    }
    __device__ __forceinline__ void add(const FF2 &o) {
        add(o.hi);
        lo = __fadd_rn(lo, o.lo);
    }
    __device__ __forceinline__ void add_sq(float v) {
        const float p = __fmul_rn(v, v);
        add(p, __fmaf_rn(v, v, -p));
    }
    __device__ __forceinline__ float value() const { return __fadd_rn(hi, lo); }
};

// kF16: store the quantised values as f16 (their exact integer values)
// instead of int8, for the prefill engine's tensor-map loads.
template <bool kGain, bool kF16>
__global__ void __launch_bounds__(kThreads)
    quant_act_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ gain, int64_t M,
                     int64_t K, float eps, void *__restrict__ qout, float *__restrict__ tok_scale,
                     int wpt) {
    pdl_launch_dependents();
    __shared__ float s_mx[kThreads / 32];
    __shared__ float s_hi[kThreads / 32], s_lo[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tpc = (kThreads / 32) / wpt;               // tokens per CTA
    const int64_t m = static_cast<int64_t>(blockIdx.x) * tpc + warp / wpt;
    const int sub = warp % wpt;
    const int nthr = wpt * 32, tid = sub * 32 + lane;
    const int64_t chunks = K / 8;                        // 8 bf16 per 16-byte chunk
    const bool active = m < M;
    pdl_wait();

    float mx = 0.0f;
    FF2 ss;
    if (active) {
        const uint4 *xr = x + m * chunks;
#pragma unroll 4
        for (int64_t i = tid; i < chunks; i += nthr) {
            if (!dbg_ok(fits(m * K + 8 * i, 8, M * K) && fits(8 * i, 8, K), 0)) continue;
            float v[8];
            bf16x8_to_f32(xr[i], v);
            if (kGain) {
                float gv[8];
                bf16x8_to_f32(gain[i], gv);
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], gv[j]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                mx = fmaxf(mx, fabsf(v[j]));
                ss.add_sq(v[j]);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        FF2 o;
        o.hi = __shfl_xor_sync(0xffffffffu, ss.hi, off);
        o.lo = __shfl_xor_sync(0xffffffffu, ss.lo, off);
        ss.add(o);
    }
    if (lane == 0) {
        s_mx[warp] = mx;
        s_hi[warp] = ss.hi;
        s_lo[warp] = ss.lo;
    }
    __syncthreads();
    if (wpt > 1) {
        const int base = (warp / wpt) * wpt;
        mx = 0.0f;
        ss = FF2();
        for (int w = 0; w < wpt; ++w) {
            mx = fmaxf(mx, s_mx[base + w]);
            FF2 o;
            o.hi = s_hi[base + w];
            o.lo = s_lo[base + w];
            ss.add(o);
        }
    }
    if (!active) return;
    if (!(mx >= 1e-5f)) mx = 1e-5f;
    const float c = __fdiv_rn(127.0f, mx);
    const uint4 *xr = x + m * chunks;
    uint2 *qr = reinterpret_cast<uint2 *>(static_cast<int8_t *>(qout) + m * K);
    uint4 *qh = reinterpret_cast<uint4 *>(static_cast<__half *>(qout) + m * K);
#pragma unroll 4
    for (int64_t i = tid; i < chunks; i += nthr) {
        if (!dbg_ok(fits(m * K + 8 * i, 8, M * K) && fits(8 * i, 8, K), 1)) continue;
        float v[8];
        bf16x8_to_f32(xr[i], v);
        if (kGain) {
            float gv[8];
            bf16x8_to_f32(gain[i], gv);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], gv[j]);
        }
        uint32_t b[2] = {0u, 0u};
        uint32_t h[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int iv = __float2int_rn(__fmul_rn(v[j], c));
            iv = iv > 127 ? 127 : (iv < -128 ? -128 : iv);
            b[j >> 2] |= (static_cast<uint32_t>(iv) & 0xffu) << (8 * (j & 3));
            h[j >> 1] |= static_cast<uint32_t>(__half_as_ushort(__int2half_rn(iv))) << (16 * (j & 1));
        }
        if (kF16)
            qh[i] = make_uint4(h[0], h[1], h[2], h[3]);
        else
            qr[i] = make_uint2(b[0], b[1]);
    }
    if (tid == 0 && dbg_ok(fits(m, 1, M), 2)) {
        const float ms = __fadd_rn(__fdiv_rn(ss.value(), static_cast<float>(K)), eps);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(ms));
        tok_scale[m] = __fdiv_rn(__fmul_rn(r, mx), 127.0f);
    }
}

}  // namespace
}  // namespace bl

namespace bl {
namespace {
bitlinear_status_t quant_entry(const void *x_bf16, const void *gain_bf16, int64_t M, int64_t K, float eps,
                               void *q, float *tok_scale, void *stream, bool f16) {
    if (M < 0 || K < 16 || (K % 16) != 0 || K > (1ll << 30)) return BITLINEAR_ERR_INVALID_ARG;
    if (M == 0) return BITLINEAR_OK;
    if (!x_bf16 || !q || !tok_scale) return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(q) || !aligned4(tok_scale) ||
        (gain_bf16 && !aligned16(gain_bf16)))
        return BITLINEAR_ERR_INVALID_ARG;
    // Few tokens: spread each token over more warps to cut latency.
    int wpt = M <= 16 ? 8 : (M <= 64 ? 4 : (M <= 512 ? 2 : 1));
    const int tpc = (kThreads / 32) / wpt;
    const int64_t blocks = (M + tpc - 1) / tpc;
    if (blocks > 0x7fffffffll) return BITLINEAR_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint4 *xv = static_cast<const uint4 *>(x_bf16);
    const uint4 *gv = static_cast<const uint4 *>(gain_bf16);
    const dim3 grid(static_cast<unsigned>(blocks)), block(kThreads);
    cudaError_t e;
    if (gain_bf16)
        e = f16 ? launch_pdl(quant_act_kernel<true, true>, grid, block, 0, st, 1, xv, gv, M, K, eps, q, tok_scale, wpt)
                : launch_pdl(quant_act_kernel<true, false>, grid, block, 0, st, 1, xv, gv, M, K, eps, q, tok_scale, wpt);
    else
        e = f16 ? launch_pdl(quant_act_kernel<false, true>, grid, block, 0, st, 1, xv, gv, M, K, eps, q, tok_scale, wpt)
                : launch_pdl(quant_act_kernel<false, false>, grid, block, 0, st, 1, xv, gv, M, K, eps, q, tok_scale, wpt);
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}
}  // namespace
}  // namespace bl

extern "C" bitlinear_status_t bitlinear_quant_act(const void *x_bf16, const void *gain_bf16,
                                                  int64_t M, int64_t K, float eps, int8_t *q,
                                                  float *tok_scale, void *stream) {
    return bl::quant_entry(x_bf16, gain_bf16, M, K, eps, q, tok_scale, stream, false);
}

extern "C" bitlinear_status_t bitlinear_quant_act_f16(const void *x_bf16, const void *gain_bf16,
                                                      int64_t M, int64_t K, float eps, void *q_f16,
                                                      float *tok_scale, void *stream) {
    return bl::quant_entry(x_bf16, gain_bf16, M, K, eps, q_f16, tok_scale, stream, true);
}
