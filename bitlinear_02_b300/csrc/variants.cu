// Decode engines for two variant weight formats (up to 64 tokens, 16-token
// chunks as blockIdx.z), with the structure of the 2-bit decode GEMV: a CTA
// of 4 warps owns 64 output rows (4 row groups) and a range of k tiles, a
// cluster of CTAs splits K and combines int32 partial sums through
// distributed shared memory, weight loads for the first tiles go out before
// the programmatic-dependent-launch wait.
//
// Five ternary digits per byte (vi.news.hada.io topic 20406, the comments on
// ternary packing: 3^5 = 243 <= 256, 1.6 bits per weight).  A byte holds
// b = ceil(256 v / 243), v the five digits e = Wq + 1 in base 3, most
// significant first; multiplying by 3 moves the next digit above the low 8
// bits.  Two bytes sit in the two 16-bit halves of a register, so one
// multiply, one byte permute and one mask give a register whose halves hold
// two digits in their lowest bits: read as f16 that is c * 2^-24, the
// operand the legacy tensor-core MMA (m16n8k16) multiplies by q.  A tile is
// 16 rows x 160 k in 512 bytes; lane 4g+t's 16 bytes hold rows g, g+8 at
// k in [40t, 40t+40), byte j of a row holding k = 40t + 5j .. 40t + 5j + 4.
// The accumulator times 2^24 is sum(c q); subtracting sum(q) gives
// sum(Wq q).
//
// The original binary BitNet (lumen-it.ai BitNet article: weights binarised
// by the signum function, absmax activations, group quantisation): one bit
// per weight (1 for +1, 0 for -1); a tile is 16 rows x 256 k, lane 4g+t
// holding rows g, g+8 at k in [64t, 64t+64), one 32-bit word per (row,
// 32-k half); the bit of k-offset j = 4s + 2sb + h of the word sits at
// 16h + 2s + sb.  Bit p of a half reads as 2^(p-24) (p <= 11; bits 12-15 are
// shifted down 8 first), the activation operand is q * 2^-p, and
// acc = 2 sum(c q) - sum(q), c the bit.  Each group of N/G consecutive rows
// has its own scale beta.
#include "decode_math.cuh"

namespace bl {

namespace {

constexpr int kWarps = 4;
constexpr int kGroups = 4;  // 16-row groups per CTA
constexpr int kRows = 16 * kGroups;

enum class Fmt { kTrits5, kBinary };

template <Fmt F>
struct FmtInfo;
template <>
struct FmtInfo<Fmt::kTrits5> {
    static constexpr int kTileK = 160;
    static constexpr int kLaneK = 40;  // k per lane and row in a tile
    static constexpr int kQWords = 10;
};
template <>
struct FmtInfo<Fmt::kBinary> {
    static constexpr int kTileK = 256;
    static constexpr int kLaneK = 64;
    static constexpr int kQWords = 16;
};

template <Fmt F, int NT>
struct VStage {
    uint4 w[kGroups];                         // one 16-byte chunk per row group
    uint32_t q[NT][FmtInfo<F>::kQWords];      // the lane's activation bytes per 8-token tile
};

// Two activation bytes (positions ka, kb of the lane's bytes, already offset
// by 128 as unsigned) -> f16 pair (q_a, q_b) * 2^-e.
template <int KA, int KB>
__device__ __forceinline__ uint32_t bpair(const uint32_t *x, uint32_t scale, uint32_t offset) {
    constexpr uint32_t sel = static_cast<uint32_t>(KA % 4) | (static_cast<uint32_t>(4 + KB % 4) << 8);
    const uint32_t gth = prmt(x[KA / 4], x[KB / 4], sel);
    return hfma2(prmt(gth, 0x64646464u, 0x4240u), scale, offset);
}

// f16x2 2^-e and -1152 * 2^-e (e = 0..11).
__device__ __forceinline__ uint32_t pscale(int e) {
    const uint32_t h = static_cast<uint32_t>(15 - e) << 10;
    return h | (h << 16);
}
__device__ __forceinline__ uint32_t poffset(int e) {
    // -1152 = -1.125 * 2^10: sign 1, exponent 25 - e, mantissa 0x080
    const uint32_t h = 0x8000u | (static_cast<uint32_t>(25 - e) << 10) | 0x080u;
    return h | (h << 16);
}

// ---- five digits per byte ----
// The ten A registers of one row and one 4-byte word (bytes j0..j0+3):
// r = 5s + i holds digit i of bytes j0 + s (low half) and j0 + s + 2 (high).
__device__ __forceinline__ void trits_regs(uint32_t w, uint32_t (&r)[10]) {
    uint32_t x0 = w & 0x00ff00ffu, x1 = (w >> 8) & 0x00ff00ffu;
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        x0 *= 3u;
        x1 *= 3u;
        r[i] = prmt(x0, 0u, 0x4341u);
        r[5 + i] = prmt(x1, 0u, 0x4341u);
        x0 &= 0x00ff00ffu;
        x1 &= 0x00ff00ffu;
    }
}

// B registers of one 8-token tile: for word W (bytes 4W..4W+3 of a row),
// MMA m (0..4) and pair pr: register index r = 2m + pr, s = r / 5, i = r % 5,
// k = 5(4W + s) + i (low half) and k + 10 (high half).
template <int W, int M5>
__device__ __forceinline__ void trits_b(const uint32_t *x, uint32_t &b0, uint32_t &b1) {
    constexpr int r0 = 2 * M5, r1 = 2 * M5 + 1;
    constexpr int k0 = 5 * (4 * W + r0 / 5) + r0 % 5, k1 = 5 * (4 * W + r1 / 5) + r1 % 5;
    b0 = bpair<k0, k0 + 10>(x, 0x3C003C00u, 0xE480E480u);
    b1 = bpair<k1, k1 + 10>(x, 0x3C003C00u, 0xE480E480u);
}

template <int NT, int W>
__device__ __forceinline__ void trits_word(const VStage<Fmt::kTrits5, NT> &st, const uint32_t (&x)[NT][10],
                                           float (&d)[kGroups][NT][4]) {
    uint32_t b[NT][5][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        trits_b<W, 0>(x[j], b[j][0][0], b[j][0][1]);
        trits_b<W, 1>(x[j], b[j][1][0], b[j][1][1]);
        trits_b<W, 2>(x[j], b[j][2][0], b[j][2][1]);
        trits_b<W, 3>(x[j], b[j][3][0], b[j][3][1]);
        trits_b<W, 4>(x[j], b[j][4][0], b[j][4][1]);
    }
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
        uint32_t ra[10], rb[10];
        trits_regs(W ? st.w[gi].y : st.w[gi].x, ra);  // row g
        trits_regs(W ? st.w[gi].w : st.w[gi].z, rb);  // row g + 8
#pragma unroll
        for (int m = 0; m < 5; ++m)
#pragma unroll
            for (int j = 0; j < NT; ++j)
                dm::mma16816(d[gi][j], ra[2 * m], rb[2 * m], ra[2 * m + 1], rb[2 * m + 1], b[j][m][0], b[j][m][1]);
    }
}

// ---- binary ----
template <int P>
__device__ __forceinline__ uint32_t bit_reg(uint32_t w) {
    if constexpr (P < 12)
        return w & (0x00010001u << P);
    else
        return (w >> 8) & (0x00010001u << (P - 8));
}
template <int P>
constexpr int bit_exp() {
    return P < 12 ? P : P - 8;
}

// MMA step s (0..7) of word half P2 (0/1): pairs at bit positions 2s, 2s+1,
// k = 32 P2 + 4s + 2sb + h.
template <int NT, int P2, int S>
__device__ __forceinline__ void binary_step(const VStage<Fmt::kBinary, NT> &st, const uint32_t (&x)[NT][16],
                                            float (&d)[kGroups][NT][4]) {
    constexpr int p0 = 2 * S, p1 = 2 * S + 1;
    constexpr int k0 = 32 * P2 + 4 * S, k1 = k0 + 2;
    uint32_t b[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        b[j][0] = bpair<k0, k0 + 1>(x[j], pscale(bit_exp<p0>()), poffset(bit_exp<p0>()));
        b[j][1] = bpair<k1, k1 + 1>(x[j], pscale(bit_exp<p1>()), poffset(bit_exp<p1>()));
    }
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
        const uint32_t X = P2 ? st.w[gi].z : st.w[gi].x, Y = P2 ? st.w[gi].w : st.w[gi].y;
#pragma unroll
        for (int j = 0; j < NT; ++j)
            dm::mma16816(d[gi][j], bit_reg<p0>(X), bit_reg<p0>(Y), bit_reg<p1>(X), bit_reg<p1>(Y), b[j][0],
                         b[j][1]);
    }
}

template <int NT, int P2>
__device__ __forceinline__ void binary_half(const VStage<Fmt::kBinary, NT> &st, const uint32_t (&x)[NT][16],
                                            float (&d)[kGroups][NT][4]) {
    binary_step<NT, P2, 0>(st, x, d);
    binary_step<NT, P2, 1>(st, x, d);
    binary_step<NT, P2, 2>(st, x, d);
    binary_step<NT, P2, 3>(st, x, d);
    binary_step<NT, P2, 4>(st, x, d);
    binary_step<NT, P2, 5>(st, x, d);
    binary_step<NT, P2, 6>(st, x, d);
    binary_step<NT, P2, 7>(st, x, d);
}

template <Fmt F, int NT>
__global__ void __launch_bounds__(kWarps * 32, 3)
    variant_gemv_kernel(const int8_t *__restrict__ q, const float *__restrict__ tok_scale,
                        const uint8_t *__restrict__ packed, const float *__restrict__ scales, int group_rows,
                        int M, int N, int K, int KT, int RGN, int tiles_per_cta, __nv_bfloat16 *__restrict__ out,
                        int32_t *__restrict__ acc_out) {
    using I = FmtInfo<F>;
    __shared__ int32_t part[kWarps][NT * 8][kRows];
    __shared__ int32_t total[NT * 8 * kRows];

    // extents and chunk offsets, for the debug build's bounds checks
    const int64_t w_ext = static_cast<int64_t>(RGN) * KT * 512, q_ext = static_cast<int64_t>(M) * K,
                  o_ext = static_cast<int64_t>(M) * N, s_ext = M;
    const int64_t q_base = static_cast<int64_t>(blockIdx.z) * 16 * K, o_base = static_cast<int64_t>(blockIdx.z) * 16 * N,
                  s_base = 16 * static_cast<int64_t>(blockIdx.z);
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

    auto load_w = [&](VStage<F, NT> &st, int c) {
        if (c >= c_end) return;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int rg = rb * kGroups + i;
            const int64_t off = (static_cast<int64_t>(rg) * KT + c) * 512 + lane * 16;
            if (rg < RGN && dbg_ok(fits(off, 16, w_ext), 0))
                st.w[i] = ld_stream16(packed + off);
            else
                st.w[i] = make_uint4(0u, 0u, 0u, 0u);  // never stored (rows past N)
        }
    };
    auto load_q = [&](VStage<F, NT> &st, int c) {
        if (c >= c_end) return;
        const int k0 = c * I::kTileK + t * I::kLaneK;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int tok = 8 * j + g;
            const int8_t *src = q + static_cast<int64_t>(tok) * K + k0;
            if constexpr (F == Fmt::kTrits5) {
#pragma unroll
                for (int p = 0; p < 5; ++p) {  // 8-byte pieces: k0 is a multiple of 8, K of 16
                    const bool ok = tok < M && k0 + 8 * p < K &&
                                    dbg_ok(fits(q_base + static_cast<int64_t>(tok) * K + k0 + 8 * p, 8, q_ext), 1);
                    const uint2 v = ok ? __ldg(reinterpret_cast<const uint2 *>(src + 8 * p)) : make_uint2(0u, 0u);
                    st.q[j][2 * p] = v.x;
                    st.q[j][2 * p + 1] = v.y;
                }
            } else {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const bool ok = tok < M && k0 + 16 * p < K &&
                                    dbg_ok(fits(q_base + static_cast<int64_t>(tok) * K + k0 + 16 * p, 16, q_ext), 1);
                    const uint4 v = ok ? ld_ro16(src + 16 * p) : make_uint4(0u, 0u, 0u, 0u);
                    st.q[j][4 * p] = v.x;
                    st.q[j][4 * p + 1] = v.y;
                    st.q[j][4 * p + 2] = v.z;
                    st.q[j][4 * p + 3] = v.w;
                }
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

    auto compute = [&](const VStage<F, NT> &st) {
        uint32_t x[NT][I::kQWords];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int i = 0; i < I::kQWords; ++i) {
                x[j][i] = st.q[j][i] ^ 0x80808080u;  // q + 128 per byte
                corr[j] = __dp4a(static_cast<int>(st.q[j][i]), 0x01010101, corr[j]);
            }
        if constexpr (F == Fmt::kTrits5) {
            trits_word<NT, 0>(st, x, d);
            trits_word<NT, 1>(st, x, d);
        } else {
            binary_half<NT, 0>(st, x, d);
            binary_half<NT, 1>(st, x, d);
        }
    };

    VStage<F, NT> A, B;
    int c = c_begin + warp;
    load_w(A, c);
    load_w(B, c + kWarps);
    pdl_wait();  // activations, scales and the weight scale come from earlier kernels
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

    // sum(q) of token 8j+g over this warp's k (the four t lanes), then the
    // sums of this thread's output tokens 8j+2t and 8j+2t+1.
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        corr[j] += __shfl_xor_sync(0xffffffffu, corr[j], 1);
        corr[j] += __shfl_xor_sync(0xffffffffu, corr[j], 2);
    }
    constexpr int kMul = F == Fmt::kBinary ? 2 : 1;  // binary: sum(Wb q) = 2 sum(c q) - sum(q)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int ce = __shfl_sync(0xffffffffu, corr[j], 4 * (2 * t));
        const int co = __shfl_sync(0xffffffffu, corr[j], 4 * (2 * t + 1));
        const int t0 = 8 * j + 2 * t;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int r0 = 16 * i + g;
            part[warp][t0][r0] = kMul * __float2int_rn(d[i][j][0] * 16777216.0f) - ce;
            part[warp][t0 + 1][r0] = kMul * __float2int_rn(d[i][j][1] * 16777216.0f) - co;
            part[warp][t0][r0 + 8] = kMul * __float2int_rn(d[i][j][2] * 16777216.0f) - ce;
            part[warp][t0 + 1][r0 + 8] = kMul * __float2int_rn(d[i][j][3] * 16777216.0f) - co;
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
        if (tk < M && n < N &&
            dbg_ok(fits(o_base + o, 1, o_ext) && fits(s_base + tk, 1, s_ext) && fits(n / group_rows, 1, N / group_rows),
                   2)) {
            const float f = __fmul_rn(scales[n / group_rows], tok_scale[tk]);
            out[o] = __float2bfloat16_rn(__fmul_rn(static_cast<float>(v), f));
            if (acc_out) acc_out[o] = v;
        }
    }
    if (S > 1) cluster_sync();  // keep this CTA's shared memory alive for its peers
    pdl_launch_dependents();
}

// 2-bit layout -> five digits per byte, one thread per output byte.  The
// 2-bit code of (n, k), from the layout of bitlinear_packed_bytes: tile
// (n/16, k/128); g = n%8, u = (n%16)/8, t = (k%128)/32, j = k%32;
// P = j/16, m = (j%16)/4, sb = (j%4)/2, h = j%2, p = 2m + sb;
// byte 16(4g+t) + 4(2P+u) + (16h+2p)/8 of the tile, shift (16h+2p)%8.
__global__ void __launch_bounds__(256) repack5_kernel(const uint8_t *__restrict__ src, int64_t N, int64_t K,
                                                      int64_t KT, int64_t KT5, int64_t nbytes,
                                                      uint8_t *__restrict__ dst) {
    const int64_t ob = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (ob >= nbytes) return;
    const int64_t tile = ob / 512;
    const int o = static_cast<int>(ob % 512);
    const int64_t r = tile / KT5, c = tile % KT5;
    const int lane = o / 16, u = (o % 16) / 8, j = o % 8;
    const int g = lane / 4, t = lane % 4;
    const int64_t n = 16 * r + 8 * u + g;
    const int64_t k0 = 160 * c + 40 * t + 5 * j;
    int v = 0;
#pragma unroll
    for (int dd = 0; dd < 5; ++dd) {
        const int64_t k = k0 + dd;
        int e = 1;
        if (n < N && k < K) {
            const int kk = static_cast<int>(k % 128);
            const int t2 = kk / 32, j2 = kk % 32;
            const int P = j2 / 16, m = (j2 % 16) / 4, sb = (j2 % 4) / 2, h = j2 % 2;
            const int bit = 16 * h + 2 * (2 * m + sb);
            const int64_t byte = 512 * (r * KT + k / 128) + 16 * (4 * g + t2) + 4 * (2 * P + u) + bit / 8;
            if (dbg_ok(fits(byte, 1, (N + 15) / 16 * KT * 512), 3)) e = (src[byte] >> (bit % 8)) & 3;
        }
        v = 3 * v + e;
    }
    if (dbg_ok(fits(ob, 1, (N + 15) / 16 * KT5 * 512), 4)) dst[ob] = static_cast<uint8_t>((256 * v + 242) / 243);
}

template <Fmt F>
cudaError_t launch_variant(const int8_t *q, const float *tok_scale, const uint8_t *packed, const float *scales,
                           int group_rows, int M, int N, int K, __nv_bfloat16 *out, int32_t *acc_out,
                           cudaStream_t st, int num_sms) {
    const int KT = (K + FmtInfo<F>::kTileK - 1) / FmtInfo<F>::kTileK;
    const int RGN = (N + 15) / 16;
    const int RB = (RGN + kGroups - 1) / kGroups;
    const int Z = (M + 15) / 16;
    // about two CTAs per SM, never more than fit at once (these kernels hold
    // 127-168 registers a thread: 3 CTAs per SM)
    const int cap = (3 * num_sms) / (RB * Z);
    int S = (2 * num_sms + RB * Z - 1) / (RB * Z);
    if (S > cap) S = cap;
    const int smax = KT / kWarps > 1 ? KT / kWarps : 1;
    if (S > smax) S = smax;
    if (S > 8) S = 8;
    if (S < 1) S = 1;
    int tpc = (KT + S - 1) / S;
    S = (KT + tpc - 1) / tpc;
    const dim3 grid(S, RB, Z), block(kWarps * 32);
    if (M <= 8)
        return launch_pdl(variant_gemv_kernel<F, 1>, grid, block, 0, st, S, q, tok_scale, packed, scales, group_rows,
                          M, N, K, KT, RGN, tpc, out, acc_out);
    return launch_pdl(variant_gemv_kernel<F, 2>, grid, block, 0, st, S, q, tok_scale, packed, scales, group_rows, M,
                      N, K, KT, RGN, tpc, out, acc_out);
}

int sms_of_device() {
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        sms[dev] = v;
    }
    return sms[dev];
}

bool forward_args_ok(const int8_t *q, const float *tok_scale, const uint8_t *packed, const float *scales, int64_t M,
                     int64_t N, int64_t K, void *out) {
    if (M < 0 || N < 1 || K < 16 || (K % 16) != 0 || K > 65536 || N > (1ll << 30)) return false;
    if (M == 0) return true;
    if (!q || !tok_scale || !packed || !scales || !out) return false;
    return aligned16(q) && aligned4(tok_scale) && aligned16(packed) && aligned4(scales) && aligned16(out);
}

}  // namespace
}  // namespace bl

extern "C" size_t bitlinear_packed5_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 1) return 0;
    return static_cast<size_t>((N + 15) / 16 * 16 * ((K + 159) / 160 * 160) / 5);
}

extern "C" bitlinear_status_t bitlinear_repack5(const uint8_t *packed, int64_t N, int64_t K, uint8_t *packed5,
                                                void *stream) {
    using namespace bl;
    if (!packed || !packed5 || N < 1 || K < 16 || (K % 16) != 0 || N > (1ll << 31) || K > (1ll << 31))
        return BITLINEAR_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(packed5)) return BITLINEAR_ERR_INVALID_ARG;
    const int64_t nbytes = static_cast<int64_t>(bitlinear_packed5_bytes(N, K));
    const int64_t KT = (K + 127) / 128, KT5 = (K + 159) / 160;
    const int64_t blocks = (nbytes + 255) / 256;
    if (blocks > 0x7fffffffll) return BITLINEAR_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    repack5_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(packed, N, K, KT, KT5, nbytes, packed5);
    return cudaGetLastError() == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" bitlinear_status_t bitlinear_forward5(const int8_t *q, const float *tok_scale, const uint8_t *packed5,
                                                 const float *gamma, int64_t M, int64_t N, int64_t K,
                                                 void *out_bf16, int32_t *acc_out, void *stream) {
    using namespace bl;
    if (!forward_args_ok(q, tok_scale, packed5, gamma, M, N, K, out_bf16) || (acc_out && !aligned16(acc_out)))
        return BITLINEAR_ERR_INVALID_ARG;
    if (M == 0) return BITLINEAR_OK;
    if (M > 64 || (N + 15) / 16 > 65535 * 4) return BITLINEAR_ERR_UNSUPPORTED;
    const cudaError_t e = launch_variant<Fmt::kTrits5>(
        q, tok_scale, packed5, gamma, static_cast<int>(N), static_cast<int>(M), static_cast<int>(N),
        static_cast<int>(K), static_cast<__nv_bfloat16 *>(out_bf16), acc_out, static_cast<cudaStream_t>(stream),
        sms_of_device());
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" bitlinear_status_t bitlinear_forward_binary(const int8_t *q, const float *tok_scale,
                                                       const uint8_t *packed1, const float *beta, int64_t groups,
                                                       int64_t M, int64_t N, int64_t K, void *out_bf16,
                                                       int32_t *acc_out, void *stream) {
    using namespace bl;
    if (!forward_args_ok(q, tok_scale, packed1, beta, M, N, K, out_bf16) || (acc_out && !aligned16(acc_out)))
        return BITLINEAR_ERR_INVALID_ARG;
    if (groups < 1 || N % groups != 0) return BITLINEAR_ERR_INVALID_ARG;
    if (M == 0) return BITLINEAR_OK;
    if (M > 64 || (N + 15) / 16 > 65535 * 4) return BITLINEAR_ERR_UNSUPPORTED;
    const cudaError_t e = launch_variant<Fmt::kBinary>(
        q, tok_scale, packed1, beta, static_cast<int>(N / groups), static_cast<int>(M), static_cast<int>(N),
        static_cast<int>(K), static_cast<__nv_bfloat16 *>(out_bf16), acc_out, static_cast<cudaStream_t>(stream),
        sms_of_device());
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}
