// Decode BitLinear with the quantiser folded into the matmul (M <= 16).
//
// The BitLinear layer (cheatsheet.md, "BitNet b1.58とは？") quantises every
// projection's input per token by its absolute maximum and rescales with the
// RMS.  Run as separate kernels, a decode layer is a chain of eleven
// dependent launches (four quantisers, seven GEMVs), each bound by launch
// latency.  Here the quantiser disappears into the GEMVs:
//   - the producer of an activation (a fused GEMV, or bitlinear_act_stats
//     for the layer input) leaves, next to it, what its consumer needs to
//     quantise it: a fused GEMV folds its outputs' per-token max |v|
//     (atomicMax on the bit pattern: exact) and sum v^2 (fp32 atomics) into
//     a small accumulator of 16 copies and marks it pending; nothing else
//     waits at the end of the producer;
//   - a fused GEMV, right after its dependency wait, reduces the input's 16
//     accumulator copies in a fixed shuffle tree (every CTA computes the
//     same bits) to c = 127/max|x| and tok_scale = rms^-1 * max / 127,
//     reads its bf16 input, quantises its K-slice in registers (q =
//     rint(x * c), exactly as bitlinear_quant_act) and runs the decode GEMV
//     arithmetic (decode_math.cuh) for up to four projections that share the
//     input (q/k/v, gate/up);
//   - each consuming CTA takes a ticket once it has read the accumulator;
//     the last one writes the factors into the buffer and clears the
//     accumulator for the next production.  Later launches reading the same
//     buffer use those factors.
// A decode layer becomes four launches, chained with programmatic dependent
// launch.  Launches with many weight bytes (at least 16 MiB by default)
// quantise their input once instead, in fused_quant_kernel, which consumes
// the factor buffer the same way, and the GEMV reads int8 (every row block
// quantising the whole input again costs more there than it saves).  q and
// the int32 accumulators are bit-identical to the unfused path; the token
// scale agrees to about 1e-7.
#include "decode_math.cuh"

#include <atomic>

namespace bl {
cudaError_t status_word(unsigned int **dev_ptr);  // gemm.cu: the library's device status word
cudaError_t scratch_alloc(void **p, size_t bytes, cudaStream_t st);  // gemm.cu: stream-ordered scratch

// Launches of at least this many packed weight bytes quantise their input
// in a pre-pass (bitlinear_set_fused_prepass; -1: this default).  Measured
// on the stacks: the 70B one at one token 8.28 ms without the pre-pass,
// 7.48 with it from 32 MiB (gate+up 117 MB, down 58.7 MB), 7.32 from 16 MiB
// (also q+k+v 21 MB and o 16.8 MB), 7.32 on every launch; the 3B one (all
// launches under 14 MB) 0.865 ms without it and 0.920 with it everywhere.
constexpr int64_t kPrepassDefault = 16ll << 20;
std::atomic<int64_t> g_prepass_min{-1};
namespace {

constexpr int kWarps = 4;
constexpr int kGroups = 4;  // 16-row groups per CTA
constexpr int kRows = 16 * kGroups;
constexpr int kMaxFused = 4;
static_assert(kWarps == 4, "cta_factors covers 16 tokens with 4 warps");

// Factor buffer (floats / words): c[16] | tok_scale[16] | state (u32) |
// ticket counter (u32) | pad | acc_max[kCopies][16] (u32) |
// acc_sum[kCopies][16].  A CTA of a producer folds into copy
// (row block * S + slice) % kCopies, so the atomics spread over many words.
constexpr int kCopies = 16;
constexpr int kOffC = 0, kOffTs = 16, kOffState = 32, kOffTicket = 33, kOffMax = 64, kOffSum = 64 + 16 * kCopies;
constexpr size_t kStatsBytes = (64 + 32 * kCopies) * 4;
constexpr int64_t kStatsFloats = static_cast<int64_t>(kStatsBytes / 4);
constexpr unsigned kPending = 1u;     // state: the accumulator holds an unconsumed production
constexpr unsigned kStateError = 2u;  // status bit: a factor buffer was produced twice unconsumed

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
    const int8_t *q;  // the input quantised by fused_quant_kernel (large launches), else unused
    float *xs;  // factor buffer of the input (consumed)
    unsigned int *status;
    FProj p[kMaxFused];
    int nproj, M, K, KT, tiles_per_cta;
    int prefetch;  // bulk L2 prefetch of the weights past the register stages
    float eps;
};

// Register stage of a warp: one 128-k tile of packed weights for its 4 row
// groups, and the raw bf16 input of that tile for the lane's tokens (32
// values of token 8j+g at k = 128c + 32t, quantised just before the MMAs).
template <int NT>
struct Stage {
    uint4 w[kGroups];
    uint4 x[NT][4];
};

// q = rint(v * c) (ties to even) in the low byte of the result: adding
// 1.5 * 2^23 to fl(v * c) rounds it to an integer, as rint does.  No clamp:
// c = 127 / max|x| comes from these very values, so |v * c| <= 127 (the
// clamp of the definition never acts), and |v * c| < 2^22 keeps the trick
// exact.
__device__ __forceinline__ uint32_t qbits(float v, float c) {
    return __float_as_uint(__fadd_rn(__fmul_rn(v, c), 12582912.0f));
}
// 16 bf16 -> 16 int8 (one uint4)
__device__ __forceinline__ uint4 quant16(const uint4 &a, const uint4 &b, float c) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
        const uint32_t lo = prmt(qbits(__uint_as_float(w0 << 16), c), qbits(__uint_as_float(w0 & 0xffff0000u), c),
                                 0x0040u);
        const uint32_t hi = prmt(qbits(__uint_as_float(w1 << 16), c), qbits(__uint_as_float(w1 & 0xffff0000u), c),
                                 0x0040u);
        o[i] = prmt(lo, hi, 0x5410u);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// (hi, lo) += (bh, bl): compensated fp32 sum (two-sum of the high parts).
// Symmetric in its operands, so both lanes of a shuffle pair get the same bits.
__device__ __forceinline__ void ff_add(float &hi, float &lo, float bh, float bl_) {
    const float s = __fadd_rn(hi, bh), bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(bh, bp));
    lo = __fadd_rn(__fadd_rn(lo, bl_), err);
    hi = s;
}

// c and tok_scale of one token from max |v| and sum v^2 over K values.
__device__ __forceinline__ void token_factors(float mx, float ss, int K, float eps, float &c, float &ts) {
    if (!(mx >= 1e-5f)) mx = 1e-5f;
    const float ms = __fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), eps);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(ms));
    c = __fdiv_rn(127.0f, mx);
    ts = __fdiv_rn(__fmul_rn(r, mx), 127.0f);
}

// Factors of tokens [0, M) of a factor buffer, by a CTA of 4 warps, into
// c_out / ts_out (shared memory).  Every load is issued at once, whether the
// buffer is pending or published (one round trip): the state word, the
// published factors, and the 16 copies of each token's accumulator.  Warp w
// takes token pairs w and w + 4: lanes 0-15 hold the copies of token 2p,
// lanes 16-31 those of token 2p+1; max and the compensated sum are reduced in
// a fixed butterfly, so every CTA and every caller gets the same bits.
// Returns whether the buffer was pending.
__device__ __forceinline__ bool cta_factors(const float *xs, int M, int K, float eps, float *c_out,
                                            float *ts_out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cp = lane & 15;
    float mx[2], hi[2], lo[2] = {0.0f, 0.0f};
    int tk[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        tk[r] = 2 * (warp + 4 * r) + (lane >> 4);
        const bool ok = tk[r] < M;
        mx[r] = ok ? ld_cg_f32(xs + kOffMax + cp * 16 + tk[r]) : 0.0f;
        hi[r] = ok ? ld_cg_f32(xs + kOffSum + cp * 16 + tk[r]) : 0.0f;
    }
    const bool pend = ld_cg_u32(xs + kOffState) == kPending;
    const float pub_c = lane < 16 ? ld_cg_f32(xs + kOffC + lane) : 0.0f;
    const float pub_ts = lane < 16 ? ld_cg_f32(xs + kOffTs + lane) : 0.0f;
    if (pend) {
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], off));
                const float oh = __shfl_xor_sync(0xffffffffu, hi[r], off);
                const float ol = __shfl_xor_sync(0xffffffffu, lo[r], off);
                ff_add(hi[r], lo[r], oh, ol);
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (cp == 0 && tk[r] < M) token_factors(mx[r], __fadd_rn(hi[r], lo[r]), K, eps, c_out[tk[r]], ts_out[tk[r]]);
    } else if (warp == 0 && lane < 16) {
        c_out[lane] = pub_c;
        ts_out[lane] = pub_ts;
    }
    return pend;
}

// kQ: the input comes quantised (A.q, int8) from fused_quant_kernel instead
// of as bf16 to quantise here.
template <int NT, bool kQ>
__global__ void __launch_bounds__(kWarps * 32, NT == 1 ? 4 : 3) fused_gemv_kernel(const FArgs A) {
    __shared__ int32_t part[kWarps][NT * 8][kRows];
    __shared__ int32_t total[NT * 8 * kRows];
    __shared__ float s_c[16], s_ts[16];

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

    // Weight loads are clamped to the last row group instead of predicated
    // (its outputs are not stored); the input loads stay predicated
    // (clamping them measured 4 % slower at 16 tokens).
    auto load_w = [&](Stage<NT> &st, int c) {
        if (c >= c_end) return;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int rg = min(rbl * kGroups + i, P.RGN - 1);
            const int64_t off = (static_cast<int64_t>(rg) * KT + c) * 512 + lane * 16;
            if (dbg_ok(fits(off, 16, static_cast<int64_t>(P.RGN) * KT * 512), 0)) st.w[i] = ld_stream16(P.packed + off);
        }
    };
    auto load_x = [&](Stage<NT> &st, int c) {
        if (c >= c_end) return;
        const int k0 = c * 128 + t * 32;
        if constexpr (kQ) {
            // 32 int8 values per lane, clamped like the decode GEMV's large
            // matrices: a token past M reads token M-1 (not stored), k past K
            // rereads the row's last 16 values against padding codes c = 1,
            // which add 1*q to the MMA sum and q to sum(q): nothing.
            const int ka = min(k0, K - 16), kb = min(k0 + 16, K - 16);
#pragma unroll
            for (int jj = 0; jj < NT; ++jj) {
                const int64_t o = static_cast<int64_t>(min(8 * jj + g, M - 1)) * K;
                if (dbg_ok(fits(o + ka, 16, static_cast<int64_t>(M) * K) && fits(o + kb, 16, static_cast<int64_t>(M) * K), 1)) {
                    st.x[jj][0] = ld_ro16(A.q + o + ka);
                    st.x[jj][1] = ld_ro16(A.q + o + kb);
                }
            }
        } else {
#pragma unroll
            for (int jj = 0; jj < NT; ++jj) {
                const int tok = 8 * jj + g;
                const __nv_bfloat16 *src = A.x + static_cast<int64_t>(tok) * K + k0;
                const uint4 z = make_uint4(0, 0, 0, 0);
                const int64_t o = static_cast<int64_t>(tok) * K + k0, xe = static_cast<int64_t>(M) * K;
                const bool lo_ok = tok < M && k0 < K && dbg_ok(fits(o, 16, xe), 2);
                const bool hi_ok = tok < M && k0 + 16 < K && dbg_ok(fits(o + 16, 16, xe), 2);
                st.x[jj][0] = lo_ok ? ld_ro16(src) : z;
                st.x[jj][1] = lo_ok ? ld_ro16(src + 8) : z;
                st.x[jj][2] = hi_ok ? ld_ro16(src + 16) : z;
                st.x[jj][3] = hi_ok ? ld_ro16(src + 24) : z;
            }
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
    float cq[NT];  // 127 / max|x| of this lane's tokens
    auto compute = [&](const Stage<NT> &st) {
        uint32_t b[NT][8][2];
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) {
            if constexpr (kQ)
                dm::build_b(st.x[jj][0], st.x[jj][1], b[jj], corr[jj]);
            else
                dm::build_b(quant16(st.x[jj][0], st.x[jj][1], cq[jj]), quant16(st.x[jj][2], st.x[jj][3], cq[jj]),
                            b[jj], corr[jj]);
        }
        dm::mma_tile<NT>(st.w, b, d);
    };

    Stage<NT> SA, SB;
    int c = c_begin + warp;
    load_w(SA, c);
    load_w(SB, c + kWarps);
    // tiles past the two register stages: into L2 now, one bulk prefetch per
    // row group - for launches of under 16 MB of weights, which it speeds up;
    // it slows larger ones (70B down at 16 tokens: 49.4 -> 46.9 us without)
    if (A.prefetch && threadIdx.x < kGroups && c_end > c_begin + 2 * kWarps) {
        const int rg = rbl * kGroups + static_cast<int>(threadIdx.x);
        if (rg < P.RGN)
            bulk_prefetch_l2(P.packed + (static_cast<int64_t>(rg) * KT + c_begin + 2 * kWarps) * 512,
                             static_cast<uint32_t>(c_end - c_begin - 2 * kWarps) * 512u);
    }
    const float gam = *P.gamma;  // static, like the weights
    pdl_wait();  // the input and its factors come from earlier kernels
    load_x(SA, c);
    load_x(SB, c + kWarps);

    // The input's factors: from its pending accumulator, or as published.
    unsigned *const xs_u = reinterpret_cast<unsigned *>(A.xs);
    const bool pend = cta_factors(A.xs, M, K, A.eps, s_c, s_ts);
    // This launch produces into P.stats: mark it pending (once per buffer).
    if (P.stats != nullptr && rbl == 0 && s == 0 && threadIdx.x == 0) {
        unsigned *const st = reinterpret_cast<unsigned *>(P.stats) + kOffState;
        if (ld_cg_u32(st) == kPending) atomicOr(A.status, kStateError);
        *st = kPending;
    }
    __syncthreads();
    // Ticket: taken after the barrier, so after every thread of this CTA has
    // consumed the values it loaded from the accumulator.  The last CTA's
    // clearing stores are issued only after its own atomic has returned the
    // final count, which includes this increment.  By then no CTA's load of
    // the accumulator is still pending.  The atomic is relaxed and its result
    // is needed only at the CTA's end, so it stays off the critical path.
    // (A release here would first wait for this thread's weight loads still in
    // flight.)
    unsigned ticket = 0u;
    if (pend && threadIdx.x == 0) ticket = atomicAdd(xs_u + kOffTicket, 1u);
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
        const int tok = 8 * jj + g;
        cq[jj] = tok < M ? s_c[tok] : 0.0f;
    }

    for (; c < c_end; c += 2 * kWarps) {
        compute(SA);
        load_w(SA, c + 2 * kWarps);
        load_x(SA, c + 2 * kWarps);
        if (c + kWarps < c_end) {
            compute(SB);
            load_w(SB, c + 3 * kWarps);
            load_x(SB, c + 3 * kWarps);
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
    const int E = M * kRows;  // entries e = token * kRows + row of the real tokens
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
        e0 = min(E, s * per);
        e1 = min(E, e0 + per);
    } else {
        __syncthreads();
    }
    float *vals = reinterpret_cast<float *>(&part[0][0][0]);  // bf16 outputs as floats, by entry
    for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += kWarps * 32) {
        int v = total[e];
        if (S > 1) {
            // every slice's total (this CTA's own included), all loads in flight at once
            const uint32_t la = smem_addr(&total[e]);
            int pv[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) pv[r] = r < S ? ld_cluster_s32(cluster_map(la, r)) : 0;
            v = 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) v += pv[r];
        }
        const int tk = e / kRows, rr = e % kRows;
        const int n = rbl * kRows + rr;
        float vf = 0.0f;
        const int64_t oi = static_cast<int64_t>(tk) * P.N + n;
        if (n < P.N && dbg_ok(fits(oi, 1, static_cast<int64_t>(M) * P.N), 3)) {
            const float f = __fmul_rn(gam, s_ts[tk]);
            const __nv_bfloat16 o = __float2bfloat16_rn(__fmul_rn(static_cast<float>(v), f));
            P.out[oi] = o;
            if (P.acc_out) P.acc_out[oi] = v;
            vf = __bfloat162float(o);
        }
        vals[e] = vf;
    }
    if (S > 1) cluster_sync();  // peers have read this CTA's totals; vals complete
    else __syncthreads();

    // Fold this CTA's outputs into the per-token accumulator of the output:
    // one warp per token, two entries per lane, a compensated butterfly.
    if (P.stats != nullptr) {
        const int cp = (rbl * S + s) % kCopies;
        for (int tk = warp; tk < M; tk += kWarps) {
            const int b0 = tk * kRows;
            if (min(e1, b0 + kRows) <= max(e0, b0)) continue;  // no entry of this token here
            const int ea = b0 + lane, eb = b0 + lane + 32;
            const float va = (ea >= e0 && ea < e1) ? vals[ea] : 0.0f;
            const float vb = (eb >= e0 && eb < e1) ? vals[eb] : 0.0f;
            float mx = fmaxf(fabsf(va), fabsf(vb));
            float hi = __fmul_rn(va, va), lo = 0.0f;  // exact: va is a bf16 value
            ff_add(hi, lo, __fmul_rn(vb, vb), 0.0f);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float oh = __shfl_xor_sync(0xffffffffu, hi, off), ol = __shfl_xor_sync(0xffffffffu, lo, off);
                ff_add(hi, lo, oh, ol);
            }
            if (lane == 0 && dbg_ok(fits(kOffSum + cp * 16 + tk, 1, kStatsFloats) && tk < 16, 4)) {
                atomicMax(reinterpret_cast<unsigned int *>(P.stats + kOffMax) + cp * 16 + tk, __float_as_uint(mx));
                atomicAdd(P.stats + kOffSum + cp * 16 + tk, __fadd_rn(hi, lo));
            }
        }
    }

    // The last CTA to take a ticket publishes the input's factors and
    // clears its accumulator (every CTA has read it by then).
    if (pend && warp == 0) {
        const unsigned tk0 = __shfl_sync(0xffffffffu, ticket, 0);
        if (tk0 == gridDim.x * gridDim.y - 1u) {
            if (lane < M) {
                A.xs[kOffC + lane] = s_c[lane];
                A.xs[kOffTs + lane] = s_ts[lane];
            }
            for (int i = lane; i < 2 * 16 * kCopies; i += 32) xs_u[kOffMax + i] = 0u;
            if (lane == 0) {
                xs_u[kOffTicket] = 0u;
                xs_u[kOffState] = 0u;
            }
        }
    }
    // Only now may the next launch's CTAs start: they then find the SMs
    // empty and spread evenly (started earlier, they land wherever this
    // launch left room, several to an SM), and their weight loads overlap
    // this launch's completion.
    pdl_launch_dependents();
}

// The input of a large launch, quantised once (q = rint(x * c), the same
// bits as the GEMV CTAs' own quantisation) into q [M, K] for
// fused_gemv_kernel<NT, true>: quantising in every row block's CTAs costs
// more integer work than the weights' decoding there (70B gate/up at one
// token: 29.9 against 22 us for the GEMV on int8 input).  Consumes the input's
// factor buffer like the GEMV CTAs do (ticket; the last CTA publishes the
// factors and clears the accumulator), so the GEMV finds them published.
// Its dependents may launch at once: their weight loads overlap this pass.
__global__ void __launch_bounds__(kWarps * 32) fused_quant_kernel(const __nv_bfloat16 *__restrict__ x, float *xs,
                                                                  int M, int K, float eps, int8_t *__restrict__ q) {
    __shared__ float s_c[16], s_ts[16];
    pdl_launch_dependents();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned *const xs_u = reinterpret_cast<unsigned *>(xs);
    const bool pend = cta_factors(xs, M, K, eps, s_c, s_ts);
    __syncthreads();
    unsigned ticket = 0u;
    if (pend && threadIdx.x == 0) ticket = atomicAdd(xs_u + kOffTicket, 1u);
    const int64_t n16 = static_cast<int64_t>(M) * K / 16;  // K % 16 == 0: a chunk is one token's
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int tok = static_cast<int>(i * 16 / K);
        const uint4 *src = reinterpret_cast<const uint4 *>(x) + 2 * i;
        if (dbg_ok(fits(16 * i, 16, static_cast<int64_t>(M) * K) && tok < M, 5))
            reinterpret_cast<uint4 *>(q)[i] = quant16(__ldg(src), __ldg(src + 1), s_c[tok]);
    }
    if (pend && warp == 0) {
        const unsigned tk0 = __shfl_sync(0xffffffffu, ticket, 0);
        if (tk0 == gridDim.x - 1u) {
            if (lane < M) {
                xs[kOffC + lane] = s_c[lane];
                xs[kOffTs + lane] = s_ts[lane];
            }
            for (int i = lane; i < 2 * 16 * kCopies; i += 32) xs_u[kOffMax + i] = 0u;
            if (lane == 0) {
                xs_u[kOffTicket] = 0u;
                xs_u[kOffState] = 0u;
            }
        }
    }
}

// Factors of an external input x [M, K]: one CTA per token.
__global__ void __launch_bounds__(256) act_stats_kernel(const uint4 *__restrict__ x, int M, int K, float eps,
                                                        float *__restrict__ stats) {
    pdl_launch_dependents();
    __shared__ float s_mx[8], s_hi[8], s_lo[8];
    const int m = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    if (m == 0) {  // a fresh buffer: clear the accumulator and any pending state
        unsigned *const su = reinterpret_cast<unsigned *>(stats);
        for (int i = threadIdx.x; i < 2 * 16 * kCopies; i += 256) su[kOffMax + i] = 0u;
        if (threadIdx.x == 0) {
            su[kOffTicket] = 0u;
            su[kOffState] = 0u;
        }
    }
    float mx = 0.0f, hi = 0.0f, lo = 0.0f;
    auto add = [&](float p) {
        const float sm = __fadd_rn(hi, p), bp = __fsub_rn(sm, hi);
        lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(sm, bp)), __fsub_rn(p, bp)));
        hi = sm;
    };
    const uint4 *xr = x + static_cast<int64_t>(m) * (K / 8);
    for (int i = threadIdx.x; i < K / 8; i += 256) {
        if (!dbg_ok(fits(static_cast<int64_t>(m) * K + 8 * i, 8, static_cast<int64_t>(M) * K), 6)) continue;
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
        token_factors(mx, __fadd_rn(hi, lo), K, eps, stats[kOffC + m], stats[kOffTs + m]);
    }
}

// Reads (and, if `consume`, publishes and clears) a factor buffer's factors.
__global__ void __launch_bounds__(128) read_factors_kernel(float *stats, int M, int K, float eps, int consume,
                                                           float *c_out, float *ts_out) {
    __shared__ float s_c[16], s_ts[16];
    pdl_launch_dependents();
    pdl_wait();
    unsigned *const su = reinterpret_cast<unsigned *>(stats);
    const bool pend = cta_factors(stats, M, K, eps, s_c, s_ts);
    __syncthreads();
    if (threadIdx.x < M) {
        if (c_out) c_out[threadIdx.x] = s_c[threadIdx.x];
        if (ts_out) ts_out[threadIdx.x] = s_ts[threadIdx.x];
    }
    if (pend && consume) {
        if (threadIdx.x < M) {
            stats[kOffC + threadIdx.x] = s_c[threadIdx.x];
            stats[kOffTs + threadIdx.x] = s_ts[threadIdx.x];
        }
        for (int i = threadIdx.x; i < 2 * 16 * kCopies; i += 128) su[kOffMax + i] = 0u;
        if (threadIdx.x == 0) {
            su[kOffTicket] = 0u;
            su[kOffState] = 0u;
        }
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

extern "C" bitlinear_status_t bitlinear_fused_factors(void *stats, int64_t M, int64_t K, float eps,
                                                      int32_t consume, float *c_out, float *ts_out,
                                                      void *stream) {
    using namespace bl;
    if (M < 1 || M > 16 || K < 1 || !stats || !aligned16(stats)) return BITLINEAR_ERR_INVALID_ARG;
    if ((c_out && !aligned4(c_out)) || (ts_out && !aligned4(ts_out))) return BITLINEAR_ERR_INVALID_ARG;
    const cudaError_t e = launch_pdl(read_factors_kernel, dim3(1), dim3(128), 0, static_cast<cudaStream_t>(stream),
                                     1, static_cast<float *>(stats), static_cast<int>(M), static_cast<int>(K), eps,
                                     consume ? 1 : 0, c_out, ts_out);
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" bitlinear_status_t bitlinear_forward_fused(const void *x_bf16, void *x_stats, int64_t M,
                                                      int64_t K, int32_t nproj,
                                                      const bitlinear_fused_proj_t *projs, float eps,
                                                      void *stream) {
    using namespace bl;
    if (M < 1 || M > 16 || K < 16 || (K % 16) != 0 || K > 65536) return BITLINEAR_ERR_INVALID_ARG;
    if (!x_bf16 || !x_stats || !aligned16(x_bf16) || !aligned16(x_stats)) return BITLINEAR_ERR_INVALID_ARG;
    if (nproj < 1 || nproj > kMaxFused || !projs) return BITLINEAR_ERR_INVALID_ARG;
    FArgs A{};
    A.x = static_cast<const __nv_bfloat16 *>(x_bf16);
    A.xs = static_cast<float *>(x_stats);
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
        if (q.stats && q.stats == x_stats) return BITLINEAR_ERR_INVALID_ARG;  // reads and writes one buffer
        for (int i = 0; i < j; ++i)
            if (q.stats && projs[i].stats == q.stats) return BITLINEAR_ERR_INVALID_ARG;
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
    A.prefetch = static_cast<int64_t>(rbs) * A.KT * 2048 < (16ll << 20);
    // every argument is checked: only now the first CUDA call
    if (status_word(&A.status) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    // K split over a cluster of S CTAs (combined in distributed shared
    // memory).  Launches that quantise in the loop: sized for about two
    // CTAs per SM up to 8 tokens and one above
    // (the 16-token kernel holds 168 registers a thread; measured on the 2B
    // step: 12.16 -> 11.68 us per launch at M = 16, while M <= 8 is 3 %
    // slower with one CTA per SM and 14 % slower with three)
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int per_sm = M <= 8 ? 2 : 1;
    int S = (per_sm * sms + rbs - 1) / rbs;
    const int64_t wbytes = static_cast<int64_t>(rbs) * A.KT * 2048;
    const int64_t pre_min = g_prepass_min.load();
    const bool prepass = wbytes >= (pre_min >= 0 ? pre_min : kPrepassDefault);
    if (prepass) {
        // Large launches split K until their CTAs fill every resident slot
        // (4 per SM for the 8-token kernel, 3 for the 16-token one), as the
        // decode GEMV does: the 70B stack 8.00 -> 7.60 ms at 4 tokens, 8.46
        // -> 7.75 at 8 and 12.91 -> 11.81 at 16 (unchanged at one token).
        const int cap = ((M <= 8 ? 4 : 3) * sms) / rbs;
        if (cap > S) S = cap;
    }
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
    if (!prepass) {
        const cudaError_t e = M <= 8 ? launch_pdl(fused_gemv_kernel<1, false>, grid, block, 0, st, S, A)
                                     : launch_pdl(fused_gemv_kernel<2, false>, grid, block, 0, st, S, A);
        return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
    }
    // Large launch: quantise the input once, then the GEMV on int8 input.
    void *qs = nullptr;
    cudaError_t e = scratch_alloc(&qs, static_cast<size_t>(M) * K, st);
    if (e != cudaSuccess) {
        cudaGetLastError();  // a failed allocation is this call's error, not the caller's next one
        return BITLINEAR_ERR_CUDA;
    }
    const int64_t n16 = M * K / 16;
    int64_t blocks = (n16 + kWarps * 32 - 1) / (kWarps * 32);
    if (blocks > 2 * sms) blocks = 2 * sms;
    e = launch_pdl(fused_quant_kernel, dim3(static_cast<unsigned>(blocks)), block, 0, st, 1, A.x, A.xs, A.M, A.K,
                   A.eps, static_cast<int8_t *>(qs));
    if (e == cudaSuccess) {
        A.q = static_cast<const int8_t *>(qs);
        e = M <= 8 ? launch_pdl(fused_gemv_kernel<1, true>, grid, block, 0, st, S, A)
                   : launch_pdl(fused_gemv_kernel<2, true>, grid, block, 0, st, S, A);
    }
    const cudaError_t ef = cudaFreeAsync(qs, st);
    return (e == cudaSuccess && ef == cudaSuccess) ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" bitlinear_status_t bitlinear_set_fused_prepass(int64_t min_weight_bytes) {
    if (min_weight_bytes < -1) return BITLINEAR_ERR_INVALID_ARG;
    bl::g_prepass_min.store(min_weight_bytes);
    return BITLINEAR_OK;
}
