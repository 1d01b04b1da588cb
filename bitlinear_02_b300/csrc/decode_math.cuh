// Register-level arithmetic of the decode engines (M <= 16 tokens), shared by
// the per-projection GEMV and the fused decode GEMV.
//
// The packed 2-bit code c = Wq + 1 of a weight is fed to the legacy
// tensor-core MMA (m16n8k16, f16 inputs, fp32 accumulate) without being
// unpacked: kept in place at bit pair p of each 16-bit half, it reads as the
// f16 number c * 2^(E(p)-24) (E = 0,2,4,6,8,10 for p = 0..5; pairs 6 and 7
// are first shifted down by 8 bits, to E = 4, 6).  The matching activation
// operand is q * 2^-E(p), exact in f16, so every product is c*q*2^-24 and
// the fp32 sums are exact multiples of 2^-24 below 1.  The accumulator
// times 2^24 is the integer sum of c*q; subtracting sum(q) (from dp4a on the
// same activation bytes) gives sum((c-1)*q) = sum(Wq*q) exactly.
#pragma once

#include "bl_device.cuh"

namespace bl {
namespace dm {

// f16x2 constants: 2^-E(p) and -1152 * 2^-E(p) in both halves.
__device__ __forceinline__ uint32_t scale_c(int p) {
    constexpr uint32_t s[8] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u,
                               0x1C001C00u, 0x14001400u, 0x2C002C00u, 0x24002400u};
    return s[p];
}
__device__ __forceinline__ uint32_t offset_c(int p) {
    constexpr uint32_t o[8] = {0xE480E480u, 0xDC80DC80u, 0xD480D480u, 0xCC80CC80u,
                               0xC480C480u, 0xBC80BC80u, 0xD480D480u, 0xCC80CC80u};
    return o[p];
}
// A operand register for bit pair p of a packed word.
__device__ __forceinline__ uint32_t code_reg(uint32_t w, int p) {
    if (p < 6) return w & (0x00030003u << (2 * p));
    return (w >> 8) & (0x00030003u << (2 * (p - 4)));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// B operand registers for one 8-token tile and one 128-k tile: from the 32
// activation bytes this lane holds (token g of the tile, k = 32t .. 32t+31),
// build the scaled f16 fragments for the 8 sixteen-k steps, and add the
// bytes' sum to `corr`.
__device__ __forceinline__ void build_b(const uint4 &q0, const uint4 &q1, uint32_t (&b)[8][2],
                                        int &corr) {
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int mu = 0; mu < 8; ++mu) {
        const int m = mu & 3;
        const uint32_t x = qw[mu] ^ 0x80808080u;  // q + 128 per byte
        const uint32_t lo = prmt(x, 0x64646464u, 0x4140u);  // f16 (1024 + u0, 1024 + u1)
        const uint32_t hi = prmt(x, 0x64646464u, 0x4342u);
        b[mu][0] = hfma2(lo, scale_c(2 * m), offset_c(2 * m));
        b[mu][1] = hfma2(hi, scale_c(2 * m + 1), offset_c(2 * m + 1));
        corr = __dp4a(static_cast<int>(qw[mu]), 0x01010101, corr);
    }
}

// d[i][j] += (16 weight rows of row group i: one packed 16-byte lane chunk)
// x (B fragments of token tile j), for all four row groups (a caller with
// fewer passes a copy and discards the result: no branches in the loop).
// The loop order puts independent accumulators next to each other so the
// MMAs overlap.
template <int NT>
__device__ __forceinline__ void mma_tile(const uint4 (&w)[4], const uint32_t (&b)[NT][8][2],
                                         float (&d)[4][NT][4]) {
#pragma unroll
    for (int P = 0; P < 2; ++P) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int mu = 4 * P + m;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t X = P ? w[i].z : w[i].x, Y = P ? w[i].w : w[i].y;
                const uint32_t a0 = code_reg(X, 2 * m), a1 = code_reg(Y, 2 * m);
                const uint32_t a2 = code_reg(X, 2 * m + 1), a3 = code_reg(Y, 2 * m + 1);
#pragma unroll
                for (int j = 0; j < NT; ++j) mma16816(d[i][j], a0, a1, a2, a3, b[j][mu][0], b[j][mu][1]);
            }
        }
    }
}

// d += (16 weight rows of one packed 16-byte lane chunk) x (B fragments).
__device__ __forceinline__ void mma_chunk(const uint4 &w, const uint32_t (&b)[8][2], float (&d)[4]) {
    const uint32_t wr[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int P = 0; P < 2; ++P) {
        const uint32_t X = wr[2 * P], Y = wr[2 * P + 1];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int mu = 4 * P + m;
            mma16816(d, code_reg(X, 2 * m), code_reg(Y, 2 * m), code_reg(X, 2 * m + 1),
                     code_reg(Y, 2 * m + 1), b[mu][0], b[mu][1]);
        }
    }
}

}  // namespace dm
}  // namespace bl
