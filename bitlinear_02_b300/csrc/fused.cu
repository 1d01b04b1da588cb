// Decode BitLinear with the quantiser folded into the matmul (M <= 16).
//
// The BitLinear layer (cheatsheet.md, "BitNet b1.58とは？") quantises every
// projection's input per token by its absolute maximum and rescales with the
// RMS.  Run as separate kernels, a decode layer is a chain of eleven
// dependent launches (four quantisers, seven GEMVs), each bound by launch
// latency.  Here the quantiser disappears into the GEMVs:
//   - the producer of an activation (a fused GEMV, or bitlinear_act_stats
//     for the layer input) leaves, next to it, the per-token quantisation
//     factors c = 127/max|v| and tok_scale = rms^-1 * max / 127;
//   - a fused GEMV reads its bf16 input and those factors, quantises its
//     K-slice in registers while loading it (q = rint(v * c), exactly as
//     bitlinear_quant_act), and runs the decode GEMV arithmetic
//     (decode_math.cuh) on up to four projections that share the input in
//     one launch (q/k/v, gate/up);
//   - its epilogue folds the outputs' per-token max |v| (atomicMax on the bit
//     pattern: exact) and sum v^2 (fp32 atomics: order varies, so the token
//     scale may vary in its last bits, well inside 1e-6) into a small
//     accumulator; the last CTA of the projection (fence + counter) turns it
//     into the next factors and clears it.
// A decode layer becomes four launches, chained with programmatic dependent
// launch.  q and the int32 accumulators are bit-identical to the unfused
// path; the token scale agrees to about 1e-7.
#include "decode_math.cuh"

namespace bl {
namespace {

constexpr int kWarps = 4;
constexpr int kGroups = 4;  // 16-row groups per CTA
constexpr int kRows = 16 * kGroups;
constexpr int kMaxFused = 4;

// Factor buffer (floats / words): c[16] | tok_scale[16] | counter (u32) |
// pad | acc_max[kCopies][16] (u32) | acc_sum[kCopies][16].  The accumulator
// has kCopies copies (a CTA uses copy rowblock % kCopies), so the atomics of
// many CTAs do not all meet on the same words.
constexpr int kCopies = 16;
constexpr int kOffC = 0, kOffTs = 16, kOffCount = 32, kOffMax = 64, kOffSum = 64 + 16 * kCopies;
constexpr size_t kStatsBytes = (64 + 32 * kCopies) * 4;

struct FProj {
    const uint8_t *packed;
    const float *gamma;
    __nv_bfloat16 *out;
    int32_t *acc_out;
    float *stats;  // factor buffer of this output, or NULL
    int N, RGN, rb0, rb1;  // row groups; row blocks [rb0, rb1) of the launch
};

struct FArgs {
    const __nv_bfloat16 *x;
    const float *xs;  // factor buffer of the input
    FProj p[kMaxFused];
    int nproj, M, K, KT, tiles_per_cta;
    float eps;
};

template <int NT>
struct Stage {
    uint4 w[kGroups];
    uint4 q[NT][2];
};

__device__ __forceinline__ uint32_t quant_byte(float v, float c) {
    int iv = __float2int_rn(__fmul_rn(v, c));
    iv = iv > 127 ? 127 : (iv < -128 ? -128 : iv);
    return static_cast<uint32_t>(iv) & 0xffu;
}
// 16 bf16 -> 16 int8 (one uint4)
__device__ __forceinline__ uint4 quant16(const uint4 &a, const uint4 &b, float c) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
        o[i] = quant_byte(__uint_as_float(w0 << 16), c) | (quant_byte(__uint_as_float(w0 & 0xffff0000u), c) << 8) |
               (quant_byte(__uint_as_float(w1 << 16), c) << 16) |
               (quant_byte(__uint_as_float(w1 & 0xffff0000u), c) << 24);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int NT>
__global__ void __launch_bounds__(kWarps * 32, 3) fused_gemv_kernel(const FArgs A) {
    __shared__ int32_t part[kWarps][NT * 8][kRows];
    __shared__ int32_t total[NT * 8 * kRows];
    __shared__ float s_max[16], s_sum[16];
    __shared__ int s_last;

    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rb = blockIdx.y;
    int j = 0;
#pragma unroll
    for (int i = 1; i < kMaxFused; ++i)
        if (i < A.nproj && rb >= A.p[i].rb0) j = i;
    const FProj &P = A.p[j];
    const int rbl = rb - P.rb0;  // row block within the projection
    const int S = gridDim.x, s = blockIdx.x;
    const int KT = A.KT, M = A.M, K = A.K;
    const int c_begin = s * A.tiles_per_cta;
    const int c_end = min(KT, c_begin + A.tiles_per_cta);

    auto load_w = [&](Stage<NT> &st, int c) {
        if (c >= c_end) return;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int rg = rbl * kGroups + i;
            if (rg < P.RGN)
                st.w[i] = ld_stream16(P.packed + (static_cast<int64_t>(rg) * KT + c) * 512 + lane * 16);
            else
                st.w[i] = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
        }
    };
    float cq[NT];  // 127 / max|x| of this lane's tokens
    auto load_q = [&](Stage<NT> &st, int c) {
        if (c >= c_end) return;
        const int k0 = c * 128 + t * 32;
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) {
            const int tok = 8 * jj + g;
            const __nv_bfloat16 *src = A.x + static_cast<int64_t>(tok) * K + k0;
            uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0, v2 = v0, v3 = v0;
            if (tok < M && k0 < K) {
                v0 = ld_ro16(src);
                v1 = ld_ro16(src + 8);
            }
            if (tok < M && k0 + 16 < K) {
                v2 = ld_ro16(src + 16);
                v3 = ld_ro16(src + 24);
            }
            st.q[jj][0] = quant16(v0, v1, cq[jj]);
            st.q[jj][1] = quant16(v2, v3, cq[jj]);
        }
    };

    float d[kGroups][NT][4];
#pragma unroll
    for (int i = 0; i < kGroups; ++i)
#pragma unroll
        for (int jj = 0; jj < NT; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[i][jj][e] = 0.0f;
    int corr[NT];
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) corr[jj] = 0;
    auto compute = [&](const Stage<NT> &st) {
        uint32_t b[NT][8][2];
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) dm::build_b(st.q[jj][0], st.q[jj][1], b[jj], corr[jj]);
        dm::mma_tile<NT>(st.w, b, d);
    };

    Stage<NT> SA, SB;
    int c = c_begin + warp;
    load_w(SA, c);
    load_w(SB, c + kWarps);
    pdl_wait();  // the input and its factors come from earlier kernels
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
        const int tok = 8 * jj + g;
        cq[jj] = tok < M ? A.xs[kOffC + tok] : 0.0f;
    }
    load_q(SA, c);
    load_q(SB, c + kWarps);
    for (; c < c_end; c += 2 * kWarps) {
        compute(SA);
        load_w(SA, c + 2 * kWarps);
        load_q(SA, c + 2 * kWarps);
        if (c + kWarps < c_end) {
            compute(SB);
            load_w(SB, c + 3 * kWarps);
            load_q(SB, c + 3 * kWarps);
        }
    }

    // sum(q) per token over this warp's k (the four t lanes), then the
    // partial sums of this thread's output tokens 8j+2t and 8j+2t+1.
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
        corr[jj] += __shfl_xor_sync(0xffffffffu, corr[jj], 1);
        corr[jj] += __shfl_xor_sync(0xffffffffu, corr[jj], 2);
    }
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
        const int ce = __shfl_sync(0xffffffffu, corr[jj], 4 * (2 * t));
        const int co = __shfl_sync(0xffffffffu, corr[jj], 4 * (2 * t + 1));
        const int t0 = 8 * jj + 2 * t;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int r0 = 16 * i + g;
            part[warp][t0][r0] = __float2int_rn(d[i][jj][0] * 16777216.0f) - ce;
            part[warp][t0 + 1][r0] = __float2int_rn(d[i][jj][1] * 16777216.0f) - co;
            part[warp][t0][r0 + 8] = __float2int_rn(d[i][jj][2] * 16777216.0f) - ce;
            part[warp][t0 + 1][r0 + 8] = __float2int_rn(d[i][jj][3] * 16777216.0f) - co;
        }
    }
    __syncthreads();
    constexpr int E = NT * 8 * kRows;
    for (int e = threadIdx.x; e < E; e += kWarps * 32) {
        const int tk = e / kRows, rr = e % kRows;
        int v = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += part[w][tk][rr];
        total[e] = v;
    }
    int e0 = 0, e1 = E;
    if (S > 1) {
        cluster_sync();
        const int per = (E + S - 1) / S;
        e0 = s * per;
        e1 = min(E, e0 + per);
    } else {
        __syncthreads();
    }
    if (threadIdx.x < 16) {
        s_max[threadIdx.x] = 0.0f;
        s_sum[threadIdx.x] = 0.0f;
    }
    __syncthreads();
    const float gam = *P.gamma;
    float *vals = reinterpret_cast<float *>(&part[0][0][0]);  // bf16 outputs as floats, by entry
    for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += kWarps * 32) {
        int v;
        if (S > 1) {
            v = 0;
            const uint32_t la = smem_addr(&total[e]);
            for (int r = 0; r < S; ++r) v += ld_cluster_s32(cluster_map(la, r));
        } else {
            v = total[e];
        }
        const int tk = e / kRows, rr = e % kRows;
        const int n = rbl * kRows + rr;
        float vf = 0.0f;
        if (tk < M && n < P.N) {
            const float f = __fmul_rn(gam, A.xs[kOffTs + tk]);
            const __nv_bfloat16 o = __float2bfloat16_rn(__fmul_rn(static_cast<float>(v), f));
            P.out[static_cast<int64_t>(tk) * P.N + n] = o;
            if (P.acc_out) P.acc_out[static_cast<int64_t>(tk) * P.N + n] = v;
            vf = __bfloat162float(o);
        }
        vals[e] = vf;
    }
    if (S > 1) cluster_sync();  // peers have read this CTA's totals
    else __syncthreads();
    if (P.stats == nullptr) return;

    // Fold this CTA's outputs into the per-token accumulator of the projection.
    if (threadIdx.x < M) {
        const int tk = threadIdx.x;
        float mx = 0.0f, hi = 0.0f, lo = 0.0f;
        const int lo_e = max(e0, tk * kRows), hi_e = min(e1, (tk + 1) * kRows);
        for (int e = lo_e; e < hi_e; ++e) {
            const float v = vals[e];
            mx = fmaxf(mx, fabsf(v));
            const float p = __fmul_rn(v, v);  // exact: v is a bf16 value
            const float sm = __fadd_rn(hi, p), bp = __fsub_rn(sm, hi);
            lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(sm, bp)), __fsub_rn(p, bp)));
            hi = sm;
        }
        if (hi_e > lo_e) {
            const int cp = (rbl % kCopies) * 16 + tk;
            atomicMax(reinterpret_cast<unsigned int *>(P.stats + kOffMax) + cp, __float_as_uint(mx));
            atomicAdd(P.stats + kOffSum + cp, __fadd_rn(hi, lo));
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned nblk = static_cast<unsigned>((P.rb1 - P.rb0) * S);
        const unsigned old = atomicAdd(reinterpret_cast<unsigned int *>(P.stats + kOffCount), 1u);
        s_last = old == nblk - 1u;
    }
    __syncthreads();
    if (!s_last) return;
    // Last CTA of the projection: the next input's factors, then a clean
    // accumulator for the next use of this buffer.
    __threadfence();
    if (threadIdx.x < M) {
        const int tk = threadIdx.x;
        volatile float *vs = P.stats;
        float mx = 0.0f, hi = 0.0f, lo = 0.0f;
        for (int cpy = 0; cpy < kCopies; ++cpy) {  // fixed order
            mx = fmaxf(mx, __uint_as_float(reinterpret_cast<volatile unsigned int *>(vs)[kOffMax + cpy * 16 + tk]));
            const float p = vs[kOffSum + cpy * 16 + tk];
            const float sm = __fadd_rn(hi, p), bp = __fsub_rn(sm, hi);
            lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(sm, bp)), __fsub_rn(p, bp)));
            hi = sm;
        }
        const float ss = __fadd_rn(hi, lo);
        if (!(mx >= 1e-5f)) mx = 1e-5f;
        const float ms = __fadd_rn(__fdiv_rn(ss, static_cast<float>(P.N)), A.eps);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(ms));
        P.stats[kOffC + tk] = __fdiv_rn(127.0f, mx);
        P.stats[kOffTs + tk] = __fdiv_rn(__fmul_rn(r, mx), 127.0f);
        for (int cpy = 0; cpy < kCopies; ++cpy) {
            reinterpret_cast<unsigned int *>(P.stats)[kOffMax + cpy * 16 + tk] = 0u;
            P.stats[kOffSum + cpy * 16 + tk] = 0.0f;
        }
    }
    if (threadIdx.x == 0) reinterpret_cast<unsigned int *>(P.stats)[kOffCount] = 0u;
}

// Factors of an external input x [M, K]: one CTA per token.
__global__ void __launch_bounds__(256) act_stats_kernel(const uint4 *__restrict__ x, int M, int K, float eps,
                                                        float *__restrict__ stats) {
    pdl_launch_dependents();
    __shared__ float s_mx[8], s_hi[8], s_lo[8];
    const int m = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    float mx = 0.0f, hi = 0.0f, lo = 0.0f;
    auto add = [&](float p) {
        const float sm = __fadd_rn(hi, p), bp = __fsub_rn(sm, hi);
        lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(sm, bp)), __fsub_rn(p, bp)));
        hi = sm;
    };
    const uint4 *xr = x + static_cast<int64_t>(m) * (K / 8);
    for (int i = threadIdx.x; i < K / 8; i += 256) {
        const uint4 v = xr[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float a = __uint_as_float(w[q] << 16), b = __uint_as_float(w[q] & 0xffff0000u);
            mx = fmaxf(mx, fmaxf(fabsf(a), fabsf(b)));
            add(__fmul_rn(a, a));
            add(__fmul_rn(b, b));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float oh = __shfl_xor_sync(0xffffffffu, hi, off), ol = __shfl_xor_sync(0xffffffffu, lo, off);
        add(oh);
        lo = __fadd_rn(lo, ol);
    }
    if (lane == 0) {
        s_mx[warp] = mx;
        s_hi[warp] = hi;
        s_lo[warp] = lo;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mx = 0.0f;
        hi = 0.0f;
        lo = 0.0f;
        for (int w = 0; w < 8; ++w) {
            mx = fmaxf(mx, s_mx[w]);
            add(s_hi[w]);
            lo = __fadd_rn(lo, s_lo[w]);
        }
        if (!(mx >= 1e-5f)) mx = 1e-5f;
        const float ms = __fadd_rn(__fdiv_rn(__fadd_rn(hi, lo), static_cast<float>(K)), eps);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(ms));
        stats[kOffC + m] = __fdiv_rn(127.0f, mx);
        stats[kOffTs + m] = __fdiv_rn(__fmul_rn(r, mx), 127.0f);
    }
}

}  // namespace
}  // namespace bl

extern "C" size_t bitlinear_fused_stats_bytes(void) { return bl::kStatsBytes; }

extern "C" bitlinear_status_t bitlinear_act_stats(const void *x_bf16, int64_t M, int64_t K, float eps,
                                                  void *stats, void *stream) {
    using namespace bl;
    if (M < 1 || M > 16 || K < 16 || (K % 16) != 0 || K > 65536) return BITLINEAR_ERR_INVALID_ARG;
    if (!x_bf16 || !stats || !aligned16(x_bf16) || !aligned16(stats)) return BITLINEAR_ERR_INVALID_ARG;
    const cudaError_t e = launch_pdl(act_stats_kernel, dim3(static_cast<unsigned>(M)), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), 1, static_cast<const uint4 *>(x_bf16),
                                     static_cast<int>(M), static_cast<int>(K), eps, static_cast<float *>(stats));
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" bitlinear_status_t bitlinear_forward_fused(const void *x_bf16, const void *x_stats, int64_t M,
                                                      int64_t K, int32_t nproj,
                                                      const bitlinear_fused_proj_t *projs, float eps,
                                                      void *stream) {
    using namespace bl;
    if (M < 1 || M > 16 || K < 16 || (K % 16) != 0 || K > 65536) return BITLINEAR_ERR_INVALID_ARG;
    if (!x_bf16 || !x_stats || !aligned16(x_bf16) || !aligned16(x_stats)) return BITLINEAR_ERR_INVALID_ARG;
    if (nproj < 1 || nproj > kMaxFused || !projs) return BITLINEAR_ERR_INVALID_ARG;
    FArgs A{};
    A.x = static_cast<const __nv_bfloat16 *>(x_bf16);
    A.xs = static_cast<const float *>(x_stats);
    A.nproj = nproj;
    A.M = static_cast<int>(M);
    A.K = static_cast<int>(K);
    A.KT = static_cast<int>((K + 127) / 128);
    A.eps = eps;
    int rbs = 0;
    for (int j = 0; j < nproj; ++j) {
        const bitlinear_fused_proj_t &q = projs[j];
        if (!q.packed || !q.gamma || !q.out_bf16 || q.N < 1 || q.N > (1 << 24)) return BITLINEAR_ERR_INVALID_ARG;
        if (!aligned16(q.packed) || !aligned4(q.gamma) || !aligned16(q.out_bf16) ||
            (q.acc_out && !aligned16(q.acc_out)) || (q.stats && !aligned16(q.stats)))
            return BITLINEAR_ERR_INVALID_ARG;
        FProj &P = A.p[j];
        P.packed = q.packed;
        P.gamma = q.gamma;
        P.out = static_cast<__nv_bfloat16 *>(q.out_bf16);
        P.acc_out = q.acc_out;
        P.stats = static_cast<float *>(q.stats);
        P.N = static_cast<int>(q.N);
        P.RGN = (P.N + 15) / 16;
        P.rb0 = rbs;
        P.rb1 = rbs + (P.RGN + kGroups - 1) / kGroups;
        rbs = P.rb1;
    }
    if (rbs > 65535) return BITLINEAR_ERR_UNSUPPORTED;
    // K split over a cluster of S CTAs (combined in distributed shared memory)
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int S = (2 * sms + rbs - 1) / rbs;
    const int smax = A.KT / kWarps > 1 ? A.KT / kWarps : 1;
    if (S > smax) S = smax;
    if (S > 8) S = 8;
    if (S < 1) S = 1;
    int tpc = (A.KT + S - 1) / S;
    S = (A.KT + tpc - 1) / tpc;
    A.tiles_per_cta = tpc;
    for (int j = 0; j < nproj; ++j)
        if (static_cast<int64_t>(A.p[j].rb1 - A.p[j].rb0) * S > (1 << 30)) return BITLINEAR_ERR_UNSUPPORTED;
    const dim3 grid(S, rbs), block(kWarps * 32);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = M <= 8 ? launch_pdl(fused_gemv_kernel<1>, grid, block, 0, st, S, A)
                                 : launch_pdl(fused_gemv_kernel<2>, grid, block, 0, st, S, A);
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}
