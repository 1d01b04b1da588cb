// Decode engine (bitlinear_forward up to 64 tokens: 16-token chunks as
// blockIdx.z): HBM-bound stream of packed ternary weights.
//
// asi.tokyo, "マイクロソフトが偶然に作った史上最も効率的なAI" (2025-04-27), the paragraph on
// running the model on a GPU: the weights travel packed four per byte and are
// unpacked right next to the math units, then multiplied with 8-bit
// activations.  Here every 16-byte lane chunk of the packed layout is
// loaded once (128-bit, streaming), unpacked in registers and fed to the
// legacy tensor-core MMA (m16n8k16, f16 inputs, fp32 accumulate) - on B300
// its f16 rate is four times its int8 rate and far above dp4a.
//
// Unpacking costs one AND per two weights: a 2-bit code c = Wq + 1 kept in
// place at bit pair p of each 16-bit half reads, as an f16, c * 2^(E(p)-24)
// (a subnormal or the smallest normals; E = 0,2,4,6,8,10 for p = 0..5, and
// pairs 6,7 are shifted down by 8 bits to E = 4,6).  The matching
// activation operand is q * 2^-E(p), exact in f16, so every product is
// c*q*2^-24 and the fp32 sums are exact multiples of 2^-24 below 1.  The
// accumulator times 2^24 is the integer sum of c*q; subtracting sum(q)
// (from dp4a) gives sum((c-1)*q) = sum(Wq*q) exactly.
//
// Work split: a CTA of 4 warps owns 64 output rows (4 row groups) and a
// range of 128-k tiles; warp w takes every 4th tile of that range and all
// 4 row groups, reusing each activation fragment 4 times.  A thread-block
// cluster of S CTAs splits K; partial int32 sums are combined through
// distributed shared memory, and each CTA of the cluster finishes a slice
// of the outputs.  Weight loads for the first tiles are issued before the
// programmatic-dependent-launch wait, so they overlap the previous kernel.
#include "decode_math.cuh"

namespace bl {

namespace {

constexpr int kWarps = 4;
constexpr int kGroups = 4;  // 16-row groups per CTA
constexpr int kRows = 16 * kGroups;

template <int NT>
struct Stage {
    uint4 w[kGroups];  // one 16-byte chunk per row group
    uint4 q[NT][2];    // 32 activation bytes per 8-token tile
};

template <int NT, bool kClamp>
__global__ void __launch_bounds__(kWarps * 32, NT == 1 ? 4 : 3)
    gemv_kernel(const int8_t *__restrict__ q, const float *__restrict__ tok_scale,
                const uint8_t *__restrict__ packed, const float *__restrict__ gamma, int M, int N,
                int K, int KT, int RGN, int tiles_per_cta, __nv_bfloat16 *__restrict__ out,
                int32_t *__restrict__ acc_out) {
    __shared__ int32_t part[kWarps][NT * 8][kRows];
    __shared__ int32_t total[NT * 8 * kRows];

    // Extents of the buffers, for the debug build's bounds checks (offsets
    // from the unshifted pointers: q_base, o_base).
    const int64_t w_ext = static_cast<int64_t>(RGN) * KT * 512, q_ext = static_cast<int64_t>(M) * K,
                  o_ext = static_cast<int64_t>(M) * N, s_ext = M;
    const int64_t q_base = static_cast<int64_t>(blockIdx.z) * 16 * K, o_base = static_cast<int64_t>(blockIdx.z) * 16 * N,
                  s_base = 16 * static_cast<int64_t>(blockIdx.z);
    // Batches of up to 64 tokens: blockIdx.z picks a 16-token chunk (its rows
    // of q, scales and outputs); the chunks share the weights through L2.
    {
        const int z = static_cast<int>(blockIdx.z);
        q += static_cast<int64_t>(z) * 16 * K;
        tok_scale += 16 * z;
        out += static_cast<int64_t>(z) * 16 * N;
        if (acc_out) acc_out += static_cast<int64_t>(z) * 16 * N;
        M = min(16, M - 16 * z);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rb = blockIdx.y;
    const int S = gridDim.x, s = blockIdx.x;
    const int c_begin = s * tiles_per_cta;
    const int c_end = min(KT, c_begin + tiles_per_cta);

    // Large matrices (kClamp): loads are clamped into the buffers instead
    // of predicated, from row pointers set once (no fill values or address
    // arithmetic per stage; 70B gate/up and down at one token: 23.6 -> 21.9
    // and 23.8 -> 21.5 us).  What they read at the edges cannot change a
    // stored result: a row group past the matrix reads the last one, a token
    // past M reads token M-1, and neither is stored; k past K (in the last
    // 128-k tile) rereads the row's last 16 bytes, and since the weight codes
    // there are padding (c = 1, weight 0) those bytes add 1*q to the MMA sum
    // and the same q to sum(q): nothing to the result.  Small matrices keep
    // the predicated loads, which start a few cycles sooner (the 512 x 256
    // layer: 4.05 against 4.14 us).
    const uint8_t *wrow[kGroups];
    const int8_t *qrow[NT];
    if (kClamp) {
#pragma unroll
        for (int i = 0; i < kGroups; ++i)
            wrow[i] = packed + static_cast<int64_t>(min(rb * kGroups + i, RGN - 1)) * KT * 512 + lane * 16;
#pragma unroll
        for (int j = 0; j < NT; ++j) qrow[j] = q + static_cast<int64_t>(min(8 * j + g, M - 1)) * K;
    }
    auto load_w = [&](Stage<NT> &st, int c) {
        if (c >= c_end) return;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            if (kClamp) {
                if (dbg_ok(fits(wrow[i] + c * 512 - packed, 16, w_ext), 0)) st.w[i] = ld_stream16(wrow[i] + c * 512);
            } else {
                const int rg = rb * kGroups + i;
                const int64_t off = (static_cast<int64_t>(rg) * KT + c) * 512 + lane * 16;
                if (rg < RGN && dbg_ok(fits(off, 16, w_ext), 1))
                    st.w[i] = ld_stream16(packed + off);
                else
                    st.w[i] = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
            }
        }
    };
    auto load_q = [&](Stage<NT> &st, int c) {
        if (c >= c_end) return;
        const int k0 = c * 128 + t * 32;
        if (kClamp) {
            const int ka = min(k0, K - 16), kb = min(k0 + 16, K - 16);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int64_t o = q_base + (qrow[j] - q);
                if (dbg_ok(fits(o + ka, 16, q_ext) && fits(o + kb, 16, q_ext), 2)) {
                    st.q[j][0] = ld_ro16(qrow[j] + ka);
                    st.q[j][1] = ld_ro16(qrow[j] + kb);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int tok = 8 * j + g;
                const int64_t o = static_cast<int64_t>(tok) * K + k0;
                const int8_t *src = q + o;
                const bool lo = tok < M && k0 < K && dbg_ok(fits(q_base + o, 16, q_ext), 3);
                const bool hi = tok < M && k0 + 16 < K && dbg_ok(fits(q_base + o + 16, 16, q_ext), 3);
                st.q[j][0] = lo ? ld_ro16(src) : make_uint4(0, 0, 0, 0);
                st.q[j][1] = hi ? ld_ro16(src + 16) : make_uint4(0, 0, 0, 0);
            }
        }
    };

    float d[kGroups][NT][4];
#pragma unroll
    for (int i = 0; i < kGroups; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[i][j][e] = 0.0f;
    int corr[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) corr[j] = 0;

    auto compute = [&](const Stage<NT> &st) {
        uint32_t b[NT][8][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) dm::build_b(st.q[j][0], st.q[j][1], b[j], corr[j]);
        dm::mma_tile<NT>(st.w, b, d);
    };

    // Two-deep software pipeline over this warp's tiles c, c+4, c+8, ...
    Stage<NT> A, B;
    int c = c_begin + warp;
    load_w(A, c);
    load_w(B, c + kWarps);
    pdl_wait();  // activations, scales and gamma come from earlier kernels
    load_q(A, c);
    load_q(B, c + kWarps);
    for (; c < c_end; c += 2 * kWarps) {
        compute(A);
        load_w(A, c + 2 * kWarps);
        load_q(A, c + 2 * kWarps);
        if (c + kWarps < c_end) {
            compute(B);
            load_w(B, c + 3 * kWarps);
            load_q(B, c + 3 * kWarps);
        }
    }

    // sum(q) over this warp's k for token 8j+g (reduce over the 4 t lanes),
    // then fetch the sums of this thread's output tokens 8j+2t and 8j+2t+1.
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        corr[j] += __shfl_xor_sync(0xffffffffu, corr[j], 1);
        corr[j] += __shfl_xor_sync(0xffffffffu, corr[j], 2);
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int ce = __shfl_sync(0xffffffffu, corr[j], 4 * (2 * t));
        const int co = __shfl_sync(0xffffffffu, corr[j], 4 * (2 * t + 1));
        const int t0 = 8 * j + 2 * t;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int r0 = 16 * i + g;
            part[warp][t0][r0] = __float2int_rn(d[i][j][0] * 16777216.0f) - ce;
            part[warp][t0 + 1][r0] = __float2int_rn(d[i][j][1] * 16777216.0f) - co;
            part[warp][t0][r0 + 8] = __float2int_rn(d[i][j][2] * 16777216.0f) - ce;
            part[warp][t0 + 1][r0 + 8] = __float2int_rn(d[i][j][3] * 16777216.0f) - co;
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

    // Combine the cluster's partial sums; CTA s finishes entries [e0, e1).
    int e0 = 0, e1 = E;
    if (S > 1) {
        cluster_sync();
        const int per = (E + S - 1) / S;
        e0 = s * per;
        e1 = min(E, e0 + per);
    } else {
        __syncthreads();
    }
    const float gam = *gamma;
    for (int e = e0 + threadIdx.x; e < e1; e += kWarps * 32) {
        int v;
        if (S > 1) {
            v = 0;
            const uint32_t la = smem_addr(&total[e]);
            for (int r = 0; r < S; ++r) v += ld_cluster_s32(cluster_map(la, r));
        } else {
            v = total[e];
        }
        const int tk = e / kRows, rr = e % kRows;
        const int n = rb * kRows + rr;
        const int64_t o = static_cast<int64_t>(tk) * N + n;
        if (tk < M && n < N && dbg_ok(fits(s_base + tk, 1, s_ext) && fits(o_base + o, 1, o_ext), 4)) {
            const float f = __fmul_rn(gam, tok_scale[tk]);
            out[o] = __float2bfloat16_rn(__fmul_rn(static_cast<float>(v), f));
            if (acc_out) acc_out[o] = v;
        }
    }
    if (S > 1) cluster_sync();  // keep this CTA's shared memory alive for its peers
    // The next launch's CTAs start only now, on SMs this launch is leaving:
    // they spread evenly instead of piling into the room left beside it.
    pdl_launch_dependents();
}

}  // namespace

// Host launcher (called by bitlinear_forward for M <= 64, in 16-token chunks).
cudaError_t launch_gemv(const int8_t *q, const float *tok_scale, const uint8_t *packed,
                        const float *gamma, int M, int N, int K, __nv_bfloat16 *out,
                        int32_t *acc_out, cudaStream_t st, int num_sms) {
    const int KT = (K + 127) / 128;
    const int RGN = (N + 15) / 16;
    const int RB = (RGN + kGroups - 1) / kGroups;
    const int Z = (M + 15) / 16;  // 16-token chunks (M <= 64)
    // about two CTAs per SM, but never more than fit at once (4 per SM for
    // the 8-token kernel, 3 for the 16-token one at 168 registers): a second
    // wave cost up to 1.6x (3B gate/up at 32 tokens: 16.9 -> 10.3 us).  Up
    // to 8 tokens the split fills every resident slot (70B down and q/o at
    // one token: 22.5 -> 21.3 and 9.7 -> 9.3 us; 3B gate/up 6.6 -> 6.3).
    const int cap = ((M <= 8 ? 4 : 3) * num_sms) / (RB * Z);
    int S = M <= 8 ? cap : (2 * num_sms + RB * Z - 1) / (RB * Z);
    if (S > cap) S = cap;
    const int smax = KT / kWarps > 1 ? KT / kWarps : 1;
    if (S > smax) S = smax;
    if (S > 8) S = 8;
    if (S < 1) S = 1;
    int tpc = (KT + S - 1) / S;
    S = (KT + tpc - 1) / tpc;
    const dim3 grid(S, RB, Z), block(kWarps * 32);
    auto go = [&](auto kernel) {
        return launch_pdl(kernel, grid, block, 0, st, S, q, tok_scale, packed, gamma, M, N, K, KT, RGN, tpc,
                          out, acc_out);
    };
    const bool large = static_cast<int64_t>(N) * K >= (1ll << 20);
    if (M <= 8) return large ? go(gemv_kernel<1, true>) : go(gemv_kernel<1, false>);
    return large ? go(gemv_kernel<2, true>) : go(gemv_kernel<2, false>);
}

}  // namespace bl
