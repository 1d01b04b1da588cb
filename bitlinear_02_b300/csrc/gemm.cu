// Prefill and mid-M engine (bitlinear_forward above 48-64 tokens,
// bitlinear_forward_f16 at any M): a dense contraction on the 5th-generation
// tensor cores.
//
// asi.tokyo, "マイクロソフトが偶然に作った史上最も効率的なAI" (2025-04-27), the paragraph on
// running the model on a GPU: a custom kernel packs four weights per byte,
// unpacks them next to the math units and multiplies them with 8-bit
// activations.  B300 (sm_103a) has no int8 tcgen05 MMA, so both operands are fed as f16: ternary codes become
// -1/0/+1 and int8 activations their exact f16 values.  Every product is an
// integer of magnitude <= 128 and every partial sum an integer below 2^24
// for K <= 65536, so the fp32 TMEM accumulator holds the exact int32 result.
//
// CTA tile: 128 weight rows (MMA M, TMEM lanes) x BN tokens (MMA N, TMEM
// columns); k advances 64 per pipeline stage.  Roles:
//   - loader (warp 9, one thread): per stage, a 2-D tensor-map copy of the
//     activation tile (BN tokens x 64 k) and one 5-D tensor-map copy of the
//     stage's half of the eight packed weight tiles, into the stage's buffers;
//   - converters (warps 0-7): the weight operand A lives in tensor memory:
//     warps 0-3 / 4-7 each own 32 rows (their TMEM lane quarter), expand the
//     row's 2-bit codes to f16 in registers and store them with tcgen05.st;
//     with int8 activations all eight warps also expand the int8 tile to f16
//     into the 128-byte-swizzled K-major B tile in shared memory;
//   - MMA issuer (warp 8): the whole warp waits, one elected lane issues
//     tcgen05.mma kind::f16 (A from TMEM, B from shared memory), 4 x K16 per
//     stage, committed to the stage's "empty" mbarrier.  (Issue from an
//     elected lane of a converged warp costs a fraction of issue from one
//     lane of a diverged warp.)
// After the last stage warps 0-7 read the accumulator with tcgen05.ld and
// apply the rescale epilogue.
//
// Split K (a cluster of S CTAs per output tile): where the output tiles
// alone would leave most SMs idle (a few dozen row tiles at 65-256 tokens),
// the S CTAs of a cluster take consecutive k ranges of the same tile; each
// moves its partial accumulator into its own shared memory as int32, and
// after a cluster barrier CTA r sums the S partials (read through
// distributed shared memory) over its share of the token columns and
// writes those outputs.  Integer partials make the sum exact in any order.
//
// Every mbarrier wait is bounded.  A wait that expires raises a flag in
// shared memory that ends every other role's waits at their next poll; the
// CTA then drains the copies and MMAs it issued, frees its tensor memory and
// sets the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "bl_device.cuh"

namespace bl {

__device__ unsigned int g_gemm_status = 0u;

namespace {

constexpr int kConverters = 256;                // warps 0-7
constexpr int kThreads = kConverters + 64;      // + MMA warp 8 + loader warp 9
constexpr uint32_t kDrainLimit = 1u << 30;
constexpr uint32_t kRawA = 8 * 256;             // packed codes of 8 row groups, one 64-k stage
constexpr int kMaxSplit = 16;                   // CTAs of a cluster sharing one tile's k range
constexpr int kMinSplitStages = 4;              // 64-k stages per CTA of a split, at least

// Behind the stages: the mbarriers, then the control words, and at +512 the
// epilogue's per-token factors gamma * s_tok (up to 256 floats).
constexpr uint32_t kFactorOff = 512;
constexpr uint32_t kCtlBytes = kFactorOff + 256 * 4;

// Control words behind the mbarriers.
struct Ctl {
    uint32_t tmem;  // TMEM base address from tcgen05.alloc
    int issued;     // stages whose copies the loader issued
    int abort;      // raised by the first wait that expires
};

// int8 activations: kRaw raw stages (packed weights + int8 tile, landed by
// TMA) feed kOps operand stages (f16 B tile in shared memory + 32 weight
// columns in TMEM).  A converted operand stage waits on a proxy fence and two
// barrier hand-offs before its MMAs can run, so the operand ring is made as
// deep as shared memory (227 KB) and TMEM (512 columns, the accumulator
// first) allow for the token tile.
template <int BN>
struct Smem {
    static constexpr int kOps = BN <= 64 ? 8 : BN <= 128 ? 6 : BN <= 192 ? 5 : 4;
    static constexpr int kRaw = BN <= 64 ? 16 : BN <= 128 ? 7 : 5;
    static constexpr uint32_t kTileB = BN * 128;        // f16 tile, BN tokens x 64 k, swizzled
    static constexpr uint32_t kRawB = BN * 64;              // int8 tile, BN tokens x 64 k
    static constexpr uint32_t kRawStage = kRawA + kRawB;    // packed codes | int8 tile
    static constexpr uint32_t kRawBase = kOps * kTileB;     // operand tiles first: 1024-aligned
    static constexpr uint32_t kBarOff = kRawBase + kRaw * kRawStage;
    static constexpr uint32_t kBytes = kBarOff + 1024 /*align*/ + kCtlBytes;
    // TMEM: accumulator in columns [0, BN), weight stages after it (32 columns each)
    static constexpr uint32_t kACol = BN;
    static constexpr uint32_t kCols = BN + 32 * kOps <= 256 ? 256 : 512;
    static_assert(BN + 32 * kOps <= 512, "accumulator and weight stages fit in TMEM");
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
    static_assert(8 * (2 * kRaw + 2 * kOps + 1) + sizeof(int) * 3 <= kFactorOff, "barriers and control words");
    static_assert(128u * BN * 4u <= kBarOff, "a split's int32 partial tile fits below the barriers");
    static_assert(128u * BN * 6u <= kBarOff, "the staged bf16 and int32 output tiles fit below the barriers");
};

// f16 activations: NSTG stages of swizzled f16 tile | packed codes (as deep
// as shared memory and TMEM allow for the token tile).
template <int BN, int NSTG>
struct Smem16 {
    static constexpr uint32_t kTileB = BN * 128;
    static constexpr uint32_t kStage = kTileB + kRawA;  // multiple of 1024
    static constexpr uint32_t kBarOff = NSTG * kStage;
    static constexpr uint32_t kBytes = kBarOff + 1024 /*align*/ + kCtlBytes;
    static constexpr uint32_t kACol = BN;
    static constexpr uint32_t kCols = BN + 32 * NSTG <= 128 ? 128 : (BN + 32 * NSTG <= 256 ? 256 : 512);
    static_assert(BN + 32 * NSTG <= 512, "accumulator and weight stages fit in TMEM");
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
    static_assert(8 * (3 * NSTG + 1) + sizeof(int) * 3 <= kFactorOff, "barriers and control words");
    static_assert(128u * BN * 4u <= kBarOff, "a split's int32 partial tile fits below the barriers");
    static_assert(128u * BN * 6u <= kBarOff, "the staged bf16 and int32 output tiles fit below the barriers");
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Shared -> global tensor-map store (bulk group), and its completion.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_addr(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group 0;" ::: "memory");
}

// Packed weights of 8 row groups for one 64-k stage (half of a 128-k tile),
// by one tensor-map copy.  A tile's lane chunk (g, t), 16 bytes at 64g + 16t,
// holds rows g and g+8 at k 32t..32t+31 as words x y z w = (g, P0) (g+8, P0)
// (g, P1) (g+8, P1).  The map lists the dimensions word, g, t, k-tile, row
// group (g before t), so the box 4 x 8 x 2 x 1 x 8 over the stage's two t
// lands as [row group][t'][g][word], 256 bytes per row group: a
// converter lane reading word (hi + 2P) of (g, t') at 16g + 4(hi + 2P)
// hits a bank of its own among the 16 rows of a row group.
__device__ __forceinline__ void tma_load_w8(void *dst, const CUtensorMap *map, int half, int c, int rg0,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(2 * half), "r"(c), "r"(rg0), "r"(smem_addr(bar))
        : "memory");
}

// The two code words (P = 0, 1) of one weight row at one 64-k stage, from the
// stage's packed codes: row `ri` (0..15) of row group `rgl`, k-half t2 (32 k).
// Odd row groups read P = 1 first, so the 32 lanes of a warp (two row groups)
// touch 32 distinct banks in each of the two loads.
__device__ __forceinline__ void load_codes(const uint8_t *codes, int rgl, int ri, int t2, bool row_ok, uint32_t &w0,
                                           uint32_t &w1) {
    if (!row_ok) {
        w0 = w1 = 0x55555555u;  // code 1: weight 0
        return;
    }
    const uint32_t *base = reinterpret_cast<const uint32_t *>(codes + 256 * rgl + 128 * t2 + 16 * (ri & 7)) + (ri >> 3);
    const int sw = rgl & 1;
    const uint32_t a = base[2 * sw], b = base[2 * (sw ^ 1)];
    w0 = sw ? b : a;
    w1 = sw ? a : b;
}

// The 2-bit codes of one weight row at 32 k (two 16-k words of the row's
// lane in the packed tile) -> 16 registers of f16 pairs (Wq = code - 1),
// i.e. 16 TMEM columns.  `w0`, `w1`: the row's 32-bit code words.
__device__ __forceinline__ void expand_codes(uint32_t w0, uint32_t w1, uint32_t (&f)[16]) {
    // Pair p <= 4 stays in place: (bits | 0x6400) reads as 1024 + c*4^p
    // (mantissa bits 0-9), and one f16x2 FMA by 4^-p with offset
    // -(1024*4^-p + 1) gives c - 1 exactly (a power-of-two scaling and an
    // exactly representable result).  Pairs 5-7 come down to 0-2 with one
    // shift shared by the three.  9 integer operations per 16 weights
    // instead of 15 (shift, mask and OR per pair), the rest on the FMA pipe
    // (measured: 28672x8192 at 64 tokens 81.6 -> 78.0 us, 2560x2560 at 4096
    // 48.1 -> 46.9; the other prefill and mid-M shapes within 1 %).
    constexpr uint32_t kScale[5] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u, 0x1C001C00u};
    constexpr uint32_t kOffset[5] = {0xE401E401u, 0xDC04DC04u, 0xD410D410u, 0xCC40CC40u, 0xC500C500u};
    const uint32_t v0 = w0 >> 10, v1 = w1 >> 10;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int s = p < 5 ? p : p - 5;
        const uint32_t m = 0x00030003u << (2 * s);
        f[p] = hfma2(((p < 5 ? w0 : v0) & m) | 0x64006400u, kScale[s], kOffset[s]);
        f[8 + p] = hfma2(((p < 5 ? w1 : v1) & m) | 0x64006400u, kScale[s], kOffset[s]);
    }
}

// Outputs from accumulator values: bf16(acc * f), f = gamma * s_tok rounded
// to nearest in fp32 (once per token, into shared memory), the product
// rounded likewise.  The fp32 accumulator holds the exact integer acc, so it
// is multiplied as it is: float(int(v)) == v, and the conversions to and
// from int32 (slow-pipe instructions, three per output with the bf16
// rounding) reduce to one packed bf16 rounding per two outputs.
__device__ __forceinline__ __nv_bfloat162 rescale2(float v0, float f0, float v1, float f1) {
    return __floats2bfloat162_rn(__fmul_rn(v0, f0), __fmul_rn(v1, f1));
}

// The accumulator tile (TMEM lanes = 128 weight rows, columns = BN tokens)
// to the outputs, by warps 0-7 (warp w: lane quarter w % 4, column half w / 4),
// two 16-column loads in flight at a time.
template <int BN>
__device__ __forceinline__ void store_tile(uint32_t tmem, int warp, int lane, int tile, int tok0, int M, int N,
                                           const float *s_f, __nv_bfloat16 *__restrict__ out,
                                           int32_t *__restrict__ acc_out) {
    static_assert((BN / 2) % 32 == 0, "column halves in steps of 32");
    const int lq = warp & 3, ch = warp >> 2;
    const int n = tile * 128 + 32 * lq + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * lq) << 16);
#pragma unroll 1
    for (int col = ch * (BN / 2); col < (ch + 1) * (BN / 2); col += 32) {
        uint32_t v[32];
        tc_ld16(lane_base + col, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
        tc_ld16(lane_base + col + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const int c = col + i, tk = tok0 + c;
            const __nv_bfloat162 o = rescale2(__uint_as_float(v[i]), s_f[c], __uint_as_float(v[i + 1]), s_f[c + 1]);
            const int64_t oe = static_cast<int64_t>(M) * N;
            if (n < N) {
                if (tk < M && dbg_ok(fits(static_cast<int64_t>(tk) * N + n, 1, oe), 0)) {
                    out[static_cast<int64_t>(tk) * N + n] = o.x;
                    if (acc_out) acc_out[static_cast<int64_t>(tk) * N + n] = __float2int_rn(__uint_as_float(v[i]));
                }
                if (tk + 1 < M && dbg_ok(fits(static_cast<int64_t>(tk + 1) * N + n, 1, oe), 0)) {
                    out[static_cast<int64_t>(tk + 1) * N + n] = o.y;
                    if (acc_out)
                        acc_out[static_cast<int64_t>(tk + 1) * N + n] = __float2int_rn(__uint_as_float(v[i + 1]));
                }
            }
        }
    }
}

// The same through shared memory: warps 0-7 write the bf16 tile (and the
// int32 tile if wanted) as [token][row], 256 (512) bytes per token, then one
// thread stores each with a tensor-map copy, which also drops the rows and
// tokens past N and M.  (Per-thread 2-byte stores of a thread's row across
// tokens kept the store path busy for a third of a tile's time.)  The stage
// buffers are free: every copy landed and every MMA that read them retired.
template <int BN>
__device__ __forceinline__ void store_tile_staged(uint32_t tmem, int warp, int lane, int tile, int tok0,
                                                  const float *s_f, uint8_t *smem, const CUtensorMap *omap,
                                                  const CUtensorMap *amap) {
    const int lq = warp & 3, ch = warp >> 2, r = 32 * lq + lane;
    __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(smem);
    int32_t *oa = reinterpret_cast<int32_t *>(smem + BN * 256);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * lq) << 16);
#pragma unroll 1
    for (int col = ch * (BN / 2); col < (ch + 1) * (BN / 2); col += 32) {
        uint32_t v[32];
        tc_ld16(lane_base + col, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
        tc_ld16(lane_base + col + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const int c = col + i;
            const __nv_bfloat162 o = rescale2(__uint_as_float(v[i]), s_f[c], __uint_as_float(v[i + 1]), s_f[c + 1]);
            ob[c * 128 + r] = o.x;
            ob[(c + 1) * 128 + r] = o.y;
            if (amap) {
                oa[c * 128 + r] = __float2int_rn(__uint_as_float(v[i]));
                oa[(c + 1) * 128 + r] = __float2int_rn(__uint_as_float(v[i + 1]));
            }
        }
    }
    fence_proxy_async_smem();
    asm volatile("bar.sync 1, %0;" ::"r"(kConverters) : "memory");
    if (warp == 0 && lane == 0) {
        tma_store_2d(omap, ob, tile * 128, tok0);
        if (amap) tma_store_2d(amap, oa, tile * 128, tok0);
        bulk_commit_and_wait();
    }
}

// Split K, step 1: this CTA's partial accumulator tile into its own shared
// memory as fp32 [BN tokens][128 rows] (exact integers below 2^24, so any
// sum of them below 2^24 - every partial and total of a K <= 65536 dot
// product of ternary and int8 values - is exact in fp32, in any order).
template <int BN>
__device__ __forceinline__ void stage_partial(uint32_t tmem, int warp, int lane, uint32_t *red) {
    const int lq = warp & 3, ch = warp >> 2, row = 32 * lq + lane;
#pragma unroll 1
    for (int col = ch * (BN / 2); col < (ch + 1) * (BN / 2); col += 16) {
        uint32_t v[16];
        tc_ld16(tmem + (static_cast<uint32_t>(32 * lq) << 16) + col, v);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) red[(col + i) * 128 + row] = v[i];
    }
}

// Split K, step 2 (after a cluster barrier): CTA `split` of the S sums the S
// partial tiles over its share of the token columns, reading the peers'
// shared memory, and writes those outputs.  Each item is four consecutive
// rows of one token column (a 16-byte read from every peer).
template <int BN>
__device__ __forceinline__ void reduce_partials(const uint32_t *red, int split, int S, int tid, int tile, int tok0,
                                                int M, int N, const float *s_f, __nv_bfloat16 *__restrict__ out,
                                                int32_t *__restrict__ acc_out) {
    const int per = (BN + S - 1) / S;
    const int c0 = split * per, c1 = c0 + per < BN ? c0 + per : BN;
    const uint32_t base = smem_addr(red);
    const bool vec = (N & 3) == 0;  // then a 4-row group is all in range and 8/16-byte aligned
    for (int item = tid; item < (c1 - c0) * 32; item += kConverters) {
        const int col = c0 + (item >> 5), r4 = (item & 31) * 4;
        const int tk = tok0 + col, n0 = tile * 128 + r4;
        if (tk >= M || n0 >= N) continue;
        const uint32_t off = base + static_cast<uint32_t>((col * 128 + r4) * 4);
        float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int p0 = 0; p0 < S; p0 += 8) {
            int4 part[8];
#pragma unroll
            for (int p = 0; p < 8; ++p)
                part[p] = p0 + p < S ? ld_cluster_v4(cluster_map(off, static_cast<uint32_t>(p0 + p)))
                                     : make_int4(0, 0, 0, 0);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                a[0] = __fadd_rn(a[0], __int_as_float(part[p].x));
                a[1] = __fadd_rn(a[1], __int_as_float(part[p].y));
                a[2] = __fadd_rn(a[2], __int_as_float(part[p].z));
                a[3] = __fadd_rn(a[3], __int_as_float(part[p].w));
            }
        }
        const float f = s_f[col];
        const int64_t o = static_cast<int64_t>(tk) * N + n0;
        if (!dbg_ok(fits(o, vec ? 4 : 1, static_cast<int64_t>(M) * N), 1)) continue;
        const __nv_bfloat162 lo = rescale2(a[0], f, a[1], f), hi = rescale2(a[2], f, a[3], f);
        if (vec) {
            uint2 pk;
            pk.x = *reinterpret_cast<const uint32_t *>(&lo);
            pk.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(out + o) = pk;
            if (acc_out)
                *reinterpret_cast<int4 *>(acc_out + o) =
                    make_int4(__float2int_rn(a[0]), __float2int_rn(a[1]), __float2int_rn(a[2]), __float2int_rn(a[3]));
        } else {
            const __nv_bfloat16 ob[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (n0 + j < N) {
                    out[o + j] = ob[j];
                    if (acc_out) acc_out[o + j] = __float2int_rn(a[j]);
                }
        }
    }
}

// Named barrier `id` over the first `threads` threads, returning the AND of
// `pred` over them (the same value in every participant).
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{.reg .pred p, q; setp.ne.u32 p, %3, 0;\n\t"
        "barrier.red.and.pred q, %1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;}"
        : "=r"(r)
        : "r"(id), "r"(threads), "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// The part every kernel ends with: the outputs (directly, or through the
// cluster's split-K reduction), the status word, and the teardown (drain the
// issued copies and MMAs, free the tensor memory).  All threads call it.
template <int BN, bool SPLIT>
__device__ __forceinline__ void finish_tile(uint8_t *smem, uint32_t tmem, uint32_t cols, uint64_t *accum,
                                            uint64_t *full, int nfull, const Ctl *ctl, float *s_f, volatile int *abort,
                                            bool timed_out, int split, int S, int tile, int M, int N,
                                            const float *__restrict__ tok_scale, const float *__restrict__ gamma,
                                            __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ acc_out,
                                            const CUtensorMap *omap, const CUtensorMap *amap, uint32_t wait_limit) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tok0 = blockIdx.y * BN;
    if (warp < 8) {
        // The tile's token factors, while the last MMAs run (the scales come
        // from an earlier kernel: wait for it, which has long completed).
        pdl_wait();
        const float gam = *gamma;
        for (int c = tid; c < BN; c += kConverters)
            s_f[c] = tok0 + c < M && dbg_ok(fits(tok0 + c, 1, M), 2) ? __fmul_rn(gam, tok_scale[tok0 + c]) : 0.0f;
        asm volatile("bar.sync 1, %0;" ::"r"(kConverters) : "memory");  // warps 0-7
        // The same outcome in all eight warps (the staged store below has a
        // barrier of its own that all of them, or none, must reach).
        bool have = mbar_wait_abortable_warp(accum, 0, wait_limit, abort);
        have = bar_and(1, kConverters, have);
        if (!have) timed_out = true;
        tc_fence_after();
        if (have) {
            if constexpr (SPLIT)
                stage_partial<BN>(tmem, warp, lane, reinterpret_cast<uint32_t *>(smem));
            else if (omap)
                store_tile_staged<BN>(tmem, warp, lane, tile, tok0, s_f, smem, omap, acc_out ? amap : nullptr);
            else
                store_tile<BN>(tmem, warp, lane, tile, tok0, M, N, s_f, out, acc_out);
        }
    }
    if constexpr (SPLIT) {
        __syncwarp();
        cluster_sync();  // every CTA's partial tile is in its shared memory
        if (warp < 8)
            reduce_partials<BN>(reinterpret_cast<const uint32_t *>(smem), split, S, tid, tile, tok0, M, N, s_f, out,
                                acc_out);
        __syncwarp();
        cluster_sync();  // the peers have read this CTA's partials
    }
    if (timed_out) atomicOr(&g_gemm_status, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        // All MMAs must have retired, and every copy landed, before the
        // accumulator and shared memory are released.
        if (lane == 0) {
            mbar_wait_bounded(accum, 0, kDrainLimit);
            const int n = ctl->issued;  // only copies that were issued can be in flight
            for (int j = n > nfull ? n - nfull : 0; j < n; ++j)
                mbar_wait_bounded(&full[j % nfull], (j / nfull) & 1, kDrainLimit);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, cols);
    }
}

// The k range (in 64-k stages) of CTA `split` of S.
__device__ __forceinline__ void split_range(int NS, int split, int S, int &st0, int &ns) {
    st0 = static_cast<int>(static_cast<int64_t>(NS) * split / S);
    ns = static_cast<int>(static_cast<int64_t>(NS) * (split + 1) / S) - st0;
}

// ---------------------------------------------------------------------------
// int8 activations (bitlinear_quant_act).
// ---------------------------------------------------------------------------
template <int BN, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap amap, int staged,
                const float *__restrict__ tok_scale, const float *__restrict__ gamma, int M, int N, int KT,
                int RGN, __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ acc_out, uint32_t wait_limit) {
    using L = Smem<BN>;
    constexpr int kRaw = L::kRaw, kOps = L::kOps;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *raw_full = bars, *raw_empty = bars + kRaw;
    uint64_t *mma_full = bars + 2 * kRaw, *op_empty = bars + 2 * kRaw + kOps;
    uint64_t *accum = bars + 2 * kRaw + 2 * kOps;
    Ctl *ctl = reinterpret_cast<Ctl *>(accum + 1);
    volatile int *abort = &ctl->abort;

    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = SPLIT ? static_cast<int>(cluster_size()) : 1;
    const int split = SPLIT ? static_cast<int>(cluster_rank()) : 0;
    const int tile = blockIdx.x / S;
    int st0, ns;
    split_range(2 * KT, split, S, st0, ns);
    bool timed_out = false;

    if (tid == 0) {
        ctl->issued = 0;
        ctl->abort = 0;
        for (int i = 0; i < kRaw; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kConverters);
        }
        for (int i = 0; i < kOps; ++i) {
            mbar_init(&mma_full[i], kConverters);
            mbar_init(&op_empty[i], 1);
        }
        mbar_init(accum, 1);
        mbar_fence_init();
    }
    if (warp == 8) {
        tmem_alloc(&ctl->tmem, L::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    const int rg0 = tile * 8;
    const int nrg = RGN - rg0 < 8 ? RGN - rg0 : 8;

    if (warp == 9) {
        // ---------------- loader ----------------
        if (lane == 0) {
            const uint32_t bytes = kRawA + L::kRawB;  // a full box: rows past N arrive zero-filled (unread)
            // the packed weights are static: their copies may start before the
            // previous kernel finished; the activations may not
            bool waited = false;
            for (int j = 0; j < ns; ++j) {
                const int st = st0 + j, rs = j % kRaw;
                if (!mbar_wait_abortable(&raw_empty[rs], ((j / kRaw) & 1) ^ 1, wait_limit, abort)) {
                    timed_out = true;
                    break;
                }
                uint8_t *raw = smem + L::kRawBase + rs * L::kRawStage;
                mbar_arrive_expect_tx(&raw_full[rs], bytes);
                tma_load_w8(raw, &wmap, st & 1, st >> 1, rg0, &raw_full[rs]);
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                tma_load_2d(raw + kRawA, &qmap, st * 64, blockIdx.y * BN, &raw_full[rs]);
                ctl->issued = j + 1;
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // Warp w owns TMEM lane quarter w % 4 (weight rows 32(w%4) + lane)
        // and half t' = w / 4 of each stage's 32 weight columns.
        const int row = 32 * (warp & 3) + lane;
        const int ri = row & 15, rgl = row >> 4, t2 = warp >> 2;
        const bool row_ok = rgl < nrg;
        const uint32_t a_lane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        for (int j = 0; j < ns; ++j) {
            const int rs = j % kRaw, slot = j % kOps;
            if (!mbar_wait_abortable_warp(&raw_full[rs], (j / kRaw) & 1, wait_limit, abort) ||
                !mbar_wait_abortable_warp(&op_empty[slot], ((j / kOps) & 1) ^ 1, wait_limit, abort)) {
                timed_out = true;
                break;
            }
            const uint8_t *raw = smem + L::kRawBase + rs * L::kRawStage;
            uint8_t *stage = smem + slot * L::kTileB;
            {
                // column c of the stage holds k = 2c, 2c+1: word (t' = c/16, P = (c%16)/8), pair p = c%8
                uint32_t w0, w1, f[16];
                load_codes(raw, rgl, ri, t2, row_ok, w0, w1);
                expand_codes(w0, w1, f);
                tc_st16(tmem + a_lane + L::kACol + 32 * slot + 16 * t2, f);
            }
            // int8 tile (token-major, 64 bytes per token) -> swizzled f16 tile
            const uint8_t *rb = raw + kRawA;
#pragma unroll
            for (int i = 0; i < BN * 4 / kConverters; ++i) {
                const int e = tid + kConverters * i;
                const int tok = e >> 2, ch = e & 3;
                const uint4 xv = *reinterpret_cast<const uint4 *>(rb + 16 * e);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                uint32_t f[8];
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint32_t x = xw[wi] ^ 0x80808080u;
                    f[2 * wi] = hadd2(prmt(x, 0x64646464u, 0x4140u), 0xE480E480u);  // -1152
                    f[2 * wi + 1] = hadd2(prmt(x, 0x64646464u, 0x4342u), 0xE480E480u);
                }
                *reinterpret_cast<uint4 *>(stage + sw128_off(tok, 2 * ch)) = make_uint4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<uint4 *>(stage + sw128_off(tok, 2 * ch + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
            }
            mbar_arrive(&raw_empty[rs]);  // every read of the raw stage has returned
            tc_wait_st();  // the weight stores above, overlapped with the activation work
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&mma_full[slot]);
        }
    } else {
        // ---------------- MMA issuer (warp 8) ----------------
        constexpr uint32_t idesc = idesc_f16_f32(128, BN);
        const uint32_t base = smem_addr(smem);
        for (int j = 0; j < ns; ++j) {
            const int slot = j % kOps;
            if (!mbar_wait_abortable_warp(&mma_full[slot], (j / kOps) & 1, wait_limit, abort)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            if (elect_one()) {
                const uint64_t bd = sw128_desc(base + slot * L::kTileB);
                const uint32_t at = tmem + L::kACol + 32 * slot;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16_ta(tmem, at + 8 * kk, bd + 2 * kk, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&op_empty[slot]);
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(accum);
        __syncwarp();
    }

    finish_tile<BN, SPLIT>(smem, tmem, L::kCols, accum, raw_full, kRaw, ctl,
                           reinterpret_cast<float *>(smem + L::kBarOff + kFactorOff), abort, timed_out, split, S, tile, M,
                           N, tok_scale, gamma, out, acc_out, staged ? &omap : nullptr, &amap, wait_limit);
}

// ---------------------------------------------------------------------------
// f16 activations (bitlinear_quant_act_f16): the activation tile arrives by
// tensor-map copy already in the 128-byte-swizzled K-major layout the MMA
// reads, so the converter warps only expand the weight codes into tensor
// memory.  NSTG stages of swizzled f16 tile | packed codes.
// ---------------------------------------------------------------------------
template <int BN, int NSTG, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm16_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap amap, int staged,
                  const float *__restrict__ tok_scale, const float *__restrict__ gamma, int M, int N, int KT,
                  int RGN, __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ acc_out, uint32_t wait_limit) {
    using L = Smem16<BN, NSTG>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *full = bars, *a_ready = bars + NSTG, *empty = bars + 2 * NSTG;
    uint64_t *accum = bars + 3 * NSTG;
    Ctl *ctl = reinterpret_cast<Ctl *>(accum + 1);
    volatile int *abort = &ctl->abort;

    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = SPLIT ? static_cast<int>(cluster_size()) : 1;
    const int split = SPLIT ? static_cast<int>(cluster_rank()) : 0;
    const int tile = blockIdx.x / S;
    int st0, ns;
    split_range(2 * KT, split, S, st0, ns);
    bool timed_out = false;
    if (tid == 0) {
        ctl->issued = 0;
        ctl->abort = 0;
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&a_ready[i], kConverters / 2);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accum, 1);
        mbar_fence_init();
    }
    if (warp == 8) {
        tmem_alloc(&ctl->tmem, L::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    const int rg0 = tile * 8;
    const int nrg = RGN - rg0 < 8 ? RGN - rg0 : 8;

    if (warp == 9) {
        // ---------------- loader ----------------
        if (lane == 0) {
            const uint32_t bytes = kRawA + L::kTileB;  // a full box: rows past N arrive zero-filled (unread)
            bool waited = false;
            for (int j = 0; j < ns; ++j) {
                const int st = st0 + j, s = j % NSTG;
                if (!mbar_wait_abortable(&empty[s], ((j / NSTG) & 1) ^ 1, wait_limit, abort)) {
                    timed_out = true;
                    break;
                }
                uint8_t *stage = smem + s * L::kStage;
                mbar_arrive_expect_tx(&full[s], bytes);
                tma_load_w8(stage + L::kTileB, &wmap, st & 1, st >> 1, rg0, &full[s]);
                if (!waited) {  // the weights are static; the activations come from earlier kernels
                    pdl_wait();
                    waited = true;
                }
                tma_load_2d(stage, &qmap, st * 64, blockIdx.y * BN, &full[s]);
                ctl->issued = j + 1;
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ---------------- converters: weight codes -> f16 in TMEM ----------------
        // Warp w owns TMEM lane quarter w % 4 (weight rows 32(w%4) + lane) and
        // the stages of parity w / 4, so two stages are converted at once.
        const int row = 32 * (warp & 3) + lane;
        const int ri = row & 15, rgl = row >> 4;
        const bool row_ok = rgl < nrg;
        const uint32_t a_lane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        for (int j = warp >> 2; j < ns; j += 2) {
            const int s = j % NSTG;
            if (!mbar_wait_abortable_warp(&full[s], (j / NSTG) & 1, wait_limit, abort)) {
                timed_out = true;
                break;
            }
            const uint8_t *codes = smem + s * L::kStage + L::kTileB;
#pragma unroll
            for (int t2 = 0; t2 < 2; ++t2) {  // two 16-column halves (fewer live registers)
                uint32_t w0, w1, f[16];
                load_codes(codes, rgl, ri, t2, row_ok, w0, w1);
                expand_codes(w0, w1, f);
                tc_st16(tmem + a_lane + L::kACol + 32 * s + 16 * t2, f);
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&a_ready[s]);
        }
    } else {
        // ---------------- MMA issuer (warp 8) ----------------
        constexpr uint32_t idesc = idesc_f16_f32(128, BN);
        const uint32_t base = smem_addr(smem);
        for (int j = 0; j < ns; ++j) {
            const int s = j % NSTG;
            if (!mbar_wait_abortable_warp(&full[s], (j / NSTG) & 1, wait_limit, abort) ||
                !mbar_wait_abortable_warp(&a_ready[s], (j / NSTG) & 1, wait_limit, abort)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            if (elect_one()) {
                const uint64_t bd = sw128_desc(base + s * L::kStage);
                const uint32_t at = tmem + L::kACol + 32 * s;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16_ta(tmem, at + 8 * kk, bd + 2 * kk, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&empty[s]);
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(accum);
        __syncwarp();
    }

    finish_tile<BN, SPLIT>(smem, tmem, L::kCols, accum, full, NSTG, ctl,
                           reinterpret_cast<float *>(smem + L::kBarOff + kFactorOff), abort, timed_out, split, S, tile, M, N,
                           tok_scale, gamma, out, acc_out, staged ? &omap : nullptr, &amap, wait_limit);
}

// ---------------------------------------------------------------------------
// Persistent variant of the f16-operand GEMM, for grids of more tiles than
// SMs: one CTA per SM walks the tiles t = blockIdx.x, + gridDim.x, ... with
// two TMEM accumulators, so the epilogue of one tile (4 warps of their own)
// runs under the next tile's MMAs instead of after them.  Tensor memory:
// accumulators in columns [0, BN) and [BN, 2BN), then a ring of NA 32-column
// weight slots (2 BN + 32 NA <= 512); the weight slots have their own
// empty/ready barriers, decoupled from the NSTG shared-memory stages.  Warps:
// 0-7 converters (parity w / 4 takes alternate stages), 8 MMA issuer, 9
// loader, 10-13 epilogue (each drains its TMEM lane quarter, warp % 4).  The
// output tile goes through one shared-memory buffer by tensor-map store.
// ---------------------------------------------------------------------------
constexpr int kThreadsP = kThreads + 128;

template <int BN, int NSTG, int NA>
struct SmemP {
    static constexpr uint32_t kTileB = BN * 128;
    static constexpr uint32_t kStage = kTileB + kRawA;  // multiple of 1024
    static constexpr uint32_t kOutOff = NSTG * kStage;
    static constexpr uint32_t kBarOff = kOutOff + BN * 256;
    static constexpr uint32_t kFactOff = kBarOff + 512;          // s_f[2][256]
    static constexpr uint32_t kBytes = kFactOff + 2048 + 1024 /*align*/;
    static constexpr uint32_t kACol = 2 * BN;
    static_assert(2 * BN + 32 * NA <= 512, "two accumulators and the weight ring fit in TMEM");
    // the second accumulator (and every weight slot) starts on a 32-column
    // boundary: with BN = 176 (second accumulator at column 176) the kernel
    // faulted the GPU, BN = 128 and 160 ran exact
    static_assert(BN % 32 == 0, "TMEM operands start on 32-column boundaries");
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
    static_assert(8 * (2 * NSTG + 2 * NA + 5) + sizeof(int) * 3 <= 512, "barriers and control words");
};

template <int BN, int NSTG, int NA>
__global__ void __launch_bounds__(kThreadsP, 1)
    gemm16p_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                   const __grid_constant__ CUtensorMap omap, const float *__restrict__ tok_scale,
                   const float *__restrict__ gamma, int M, int N, int KT, int RGN, int row_tiles, int tiles,
                   uint32_t wait_limit) {
    using L = SmemP<BN, NSTG, NA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
    uint64_t *full = bars, *empty = bars + NSTG, *a_ready = bars + 2 * NSTG, *a_empty = bars + 2 * NSTG + NA;
    uint64_t *acc_full = bars + 2 * NSTG + 2 * NA, *acc_empty = acc_full + 2, *mma_done = acc_full + 4;
    Ctl *ctl = reinterpret_cast<Ctl *>(mma_done + 1);
    volatile int *abort = &ctl->abort;
    float *s_f = reinterpret_cast<float *>(smem + L::kFactOff);  // [2][256]

    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NS = 2 * KT;
    bool timed_out = false;
    if (tid == 0) {
        ctl->issued = 0;
        ctl->abort = 0;
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(&a_ready[i], kConverters / 2);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 128);
        }
        mbar_init(mma_done, 1);
        mbar_fence_init();
    }
    if (warp == 8) {
        tmem_alloc(&ctl->tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    if (warp == 9) {
        // ---------------- loader ----------------
        if (lane == 0) {
            bool waited = false, stop = false;
            int g = 0;
            for (int t = blockIdx.x; t < tiles && !stop; t += gridDim.x) {
                const int rg0 = (t % row_tiles) * 8, tok0 = (t / row_tiles) * BN;
                for (int j = 0; j < NS; ++j, ++g) {
                    const int s = g % NSTG;
                    if (!mbar_wait_abortable(&empty[s], ((g / NSTG) & 1) ^ 1, wait_limit, abort)) {
                        timed_out = stop = true;
                        break;
                    }
                    uint8_t *stage = smem + s * L::kStage;
                    mbar_arrive_expect_tx(&full[s], L::kStage);
                    tma_load_w8(stage + L::kTileB, &wmap, j & 1, j >> 1, rg0, &full[s]);
                    if (!waited) {
                        pdl_wait();
                        waited = true;
                    }
                    tma_load_2d(stage, &qmap, j * 64, tok0, &full[s]);
                    ctl->issued = g + 1;
                }
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ---------------- converters ----------------
        const int row = 32 * (warp & 3) + lane;
        const int ri = row & 15, rgl = row >> 4, par = warp >> 2;
        const uint32_t a_lane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        bool stop = false;
        int g = 0;
        for (int t = blockIdx.x; t < tiles && !stop; t += gridDim.x) {
            const int rg0 = (t % row_tiles) * 8;
            const bool row_ok = rgl < RGN - rg0;
            for (int j = 0; j < NS; ++j, ++g) {
                if ((g & 1) != par) continue;
                const int s = g % NSTG, a = g % NA;
                if (!mbar_wait_abortable_warp(&full[s], (g / NSTG) & 1, wait_limit, abort) ||
                    !mbar_wait_abortable_warp(&a_empty[a], ((g / NA) & 1) ^ 1, wait_limit, abort)) {
                    timed_out = stop = true;
                    break;
                }
                tc_fence_after();
                const uint8_t *codes = smem + s * L::kStage + L::kTileB;
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2) {
                    uint32_t w0, w1, f[16];
                    load_codes(codes, rgl, ri, t2, row_ok, w0, w1);
                    expand_codes(w0, w1, f);
                    tc_st16(tmem + a_lane + L::kACol + 32 * a + 16 * t2, f);
                }
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(&a_ready[a]);
            }
        }
    } else if (warp == 8) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t idesc = idesc_f16_f32(128, BN);
        const uint32_t base = smem_addr(smem);
        bool stop = false;
        int g = 0, i = 0;
        for (int t = blockIdx.x; t < tiles && !stop; t += gridDim.x, ++i) {
            const int b = i & 1;
            if (!mbar_wait_abortable_warp(&acc_empty[b], ((i >> 1) & 1) ^ 1, wait_limit, abort)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            for (int j = 0; j < NS; ++j, ++g) {
                const int s = g % NSTG, a = g % NA;
                if (!mbar_wait_abortable_warp(&full[s], (g / NSTG) & 1, wait_limit, abort) ||
                    !mbar_wait_abortable_warp(&a_ready[a], (g / NA) & 1, wait_limit, abort)) {
                    timed_out = stop = true;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint64_t bd = sw128_desc(base + s * L::kStage);
                    const uint32_t at = tmem + L::kACol + 32 * a;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_f16_ta(tmem + b * BN, at + 8 * kk, bd + 2 * kk, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[s]);
                    tc_commit(&a_empty[a]);
                }
                __syncwarp();
            }
            if (stop) break;
            if (elect_one()) tc_commit(&acc_full[b]);
            __syncwarp();
        }
        if (elect_one()) tc_commit(mma_done);
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 10-13) ----------------
        // a warp reaches only the TMEM lane quarter warp % 4 (warps 10-13:
        // quarters 2, 3, 0, 1)
        const int ew = warp & 3, etid = tid - 10 * 32, r = 32 * ew + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * ew) << 16);
        __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(smem + L::kOutOff);
        pdl_wait();  // the token scales come from an earlier kernel
        const float gam = *gamma;
        int i = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
            const int b = i & 1, rt = t % row_tiles, tok0 = (t / row_tiles) * BN;
            float *f = s_f + 256 * b;
            for (int c = etid; c < BN; c += 128)
                f[c] = tok0 + c < M && dbg_ok(fits(tok0 + c, 1, M), 3) ? __fmul_rn(gam, tok_scale[tok0 + c]) : 0.0f;
            bool have = mbar_wait_abortable_warp(&acc_full[b], (i >> 1) & 1, wait_limit, abort);
            if (etid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the buffer is free
            have = bar_and(2, 128, have);  // also publishes f[] and the free buffer to all four warps
            if (!have) {
                timed_out = true;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int col = 0; col < BN; col += 32) {
                uint32_t v[32];
                tc_ld16(lane_base + b * BN + col, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                tc_ld16(lane_base + b * BN + col + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                tc_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const int c = col + k;
                    const __nv_bfloat162 o = rescale2(__uint_as_float(v[k]), f[c], __uint_as_float(v[k + 1]), f[c + 1]);
                    ob[c * 128 + r] = o.x;
                    ob[(c + 1) * 128 + r] = o.y;
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);  // the accumulator is read: the MMA may refill it
            fence_proxy_async_smem();
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (etid == 0) {
                tma_store_2d(&omap, ob, rt * 128, tok0);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
        if (etid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }

    if (timed_out) atomicOr(&g_gemm_status, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        if (lane == 0) {
            mbar_wait_bounded(mma_done, 0, kDrainLimit);
            const int n = ctl->issued;
            for (int g = n > NSTG ? n - NSTG : 0; g < n; ++g)
                mbar_wait_bounded(&full[g % NSTG], (g / NSTG) & 1, kDrainLimit);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host ---

std::mutex g_encode_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Tensor maps already encoded, keyed by address and shape: a map holds
// nothing but those, so a cached one is valid for any buffer at that
// address with that shape.
struct MapKey {
    const void *ptr;
    int kind;      // 0 activations, 1 weights, 2 outputs
    int variant;   // activations: f16; outputs: int32
    int box;       // token tile
    int64_t a, b;  // the tensor's two extents
    bool operator==(const MapKey &o) const {
        return ptr == o.ptr && kind == o.kind && variant == o.variant && box == o.box && a == o.a && b == o.b;
    }
};
struct MapEntry {
    MapKey key;
    bool used;
    CUtensorMap map;
};
constexpr int kMapCache = 64;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

// Encode a tiled tensor map through the driver (its entry point looked up
// once), or copy it from the cache.  Caller holds g_encode_mutex.
cudaError_t encode_locked(CUtensorMap *map, const MapKey &key, CUtensorMapDataType type, uint32_t rank,
                          const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                          CUtensorMapSwizzle swz) {
    const void *ptr = key.ptr;
    for (int i = 0; i < kMapCache; ++i)
        if (g_maps[i].used && g_maps[i].key == key) {
            *map = g_maps[i].map;
            return cudaSuccess;
        }
    if (!g_encode) {
        cudaDriverEntryPointQueryResult qr;
        void *fn = nullptr;
        // the ABI version of the function the PFN type below describes
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
        if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    const CUresult r = g_encode(map, type, rank, const_cast<void *>(ptr), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    MapEntry &slot = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    slot.key = key;
    slot.map = *map;
    slot.used = true;
    return cudaSuccess;
}

// Activations [M, K] row-major (int8, or f16 landing in the MMA's 128-byte
// swizzle): boxes of 64 k x BN tokens.
cudaError_t make_qmap(CUtensorMap *map, const void *q, int M, int K, int BN, bool f16) {
    std::lock_guard<std::mutex> lock(g_encode_mutex);
    const MapKey key{q, 0, f16 ? 1 : 0, BN, M, K};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * (f16 ? 2u : 1u)};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(BN)};
    return encode_locked(map, key, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dims,
                         strides, box, f16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Packed weights (layout of bitlinear_packed_bytes: in a tile, lane chunk
// (g, t) at 64g + 16t) with the dimensions listed as word (4 B), g (64 B),
// t (16 B), k-tile, row group: boxes of 4 x 8 x 2 x 1 x 8 (one 64-k stage of
// 8 row groups) land as [row group][t'][g][word].
cudaError_t make_wmap(CUtensorMap *map, const uint8_t *packed, int RGN, int KT) {
    std::lock_guard<std::mutex> lock(g_encode_mutex);
    const MapKey key{packed, 1, 0, 0, RGN, KT};
    const cuuint64_t dims[5] = {4u, 8u, 4u, static_cast<cuuint64_t>(KT), static_cast<cuuint64_t>(RGN)};
    const cuuint64_t strides[4] = {64u, 16u, 512u, static_cast<cuuint64_t>(KT) * 512u};
    const cuuint32_t box[5] = {4u, 8u, 2u, 1u, 8u};
    return encode_locked(map, key, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Outputs [M, N] row-major (bf16 or int32): boxes of 128 rows (n) x BN
// tokens, for the staged epilogue's tensor-map stores.
cudaError_t make_omap(CUtensorMap *map, const void *o, int M, int N, int BN, bool i32) {
    std::lock_guard<std::mutex> lock(g_encode_mutex);
    const MapKey key{o, 2, i32 ? 1 : 0, BN, M, N};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * (i32 ? 4u : 2u)};
    const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(BN)};
    return encode_locked(map, key, i32 ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims,
                         strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

int device_sms(int dev) {
    static int sms[64] = {0};
    if (!sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        sms[dev] = v;
    }
    return sms[dev];
}

// One kernel family (a token tile, int8 or f16 activations): the plain
// kernel, its split-K twin, their attributes (set once per device) and the
// number of S-CTA clusters of the twin that fit on the GPU at once.
template <typename Kern>
struct Family {
    Kern plain, split;
    uint32_t smem;
    bool configured[64] = {false};
    int clusters[64][kMaxSplit + 1] = {};  // 0: not asked yet, -1: none fit

    cudaError_t configure(int dev) {
        if (configured[dev]) return cudaSuccess;
        cudaError_t e = cudaFuncSetAttribute(plain, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e == cudaSuccess) e = cudaFuncSetAttribute(split, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
        return cudaSuccess;
    }
    int max_clusters(int dev, int S) {
        if (!clusters[dev][S]) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(S, 1, 1);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = S;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, split, &cfg) != cudaSuccess || n <= 0) {
                cudaGetLastError();  // a size that cannot be placed is not an error of the call
                n = -1;
            }
            clusters[dev][S] = n;
        }
        return clusters[dev][S];
    }
    // CTAs per cluster along K: 1 where the tiles already occupy half the
    // SMs, else the largest S whose clusters all fit in one wave with at
    // least kMinSplitStages stages each.
    int choose_split(int dev, int tiles, int NS) {
        if (2 * tiles > device_sms(dev)) return 1;
        int best = 1;
        for (int S = 2; S <= kMaxSplit && NS >= S * kMinSplitStages; ++S)
            if (max_clusters(dev, S) >= tiles) best = S;
        return best;
    }
};

template <int BN>
Family<decltype(&gemm_kernel<BN, false>)> &family8() {
    static Family<decltype(&gemm_kernel<BN, false>)> f{gemm_kernel<BN, false>, gemm_kernel<BN, true>,
                                                        Smem<BN>::kBytes};
    return f;
}
template <int BN, int NSTG>
Family<decltype(&gemm16_kernel<BN, NSTG, false>)> &family16() {
    static Family<decltype(&gemm16_kernel<BN, NSTG, false>)> f{gemm16_kernel<BN, NSTG, false>,
                                                                gemm16_kernel<BN, NSTG, true>, Smem16<BN, NSTG>::kBytes};
    return f;
}

std::mutex g_family_mutex;

// Plan and launch one GEMM of a family: grid (row tiles x S, token tiles),
// clusters of S along x.
template <typename Fam>
cudaError_t launch_family(Fam &fam, int BN, const void *q, bool f16, const float *tok_scale, const uint8_t *packed,
                          const float *gamma, int M, int N, int K, __nv_bfloat16 *out, int32_t *acc_out,
                          cudaStream_t st, uint32_t wait_limit, int force_split) {
    const int KT = (K + 127) / 128;
    const int RGN = (N + 15) / 16;
    const int row_tiles = (RGN + 7) / 8, tok_tiles = (M + BN - 1) / BN;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int S;
    {
        std::lock_guard<std::mutex> lock(g_family_mutex);
        e = fam.configure(dev);
        if (e != cudaSuccess) return e;
        if (force_split > 0) {  // clamped to the stages there are and to a cluster size that fits
            S = force_split < 2 * KT ? force_split : 2 * KT;
            if (S > kMaxSplit) S = kMaxSplit;
            while (S > 1 && fam.max_clusters(dev, S) <= 0) --S;
        } else {
            S = fam.choose_split(dev, row_tiles * tok_tiles, 2 * KT);
        }
    }
    CUtensorMap qmap, wmap;
    e = make_qmap(&qmap, q, M, K, BN, f16);
    if (e != cudaSuccess) return e;
    e = make_wmap(&wmap, packed, RGN, KT);
    if (e != cudaSuccess) return e;
    // Tensor-map stores of the output tiles need rows of a multiple of 16
    // bytes (N % 8 for bf16); otherwise each thread stores its own elements.
    CUtensorMap omap = {}, amap = {};
    const int staged = S == 1 && (N % 8) == 0;
    if (staged) {
        e = make_omap(&omap, out, M, N, BN, false);
        if (e == cudaSuccess && acc_out) e = make_omap(&amap, acc_out, M, N, BN, true);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(row_tiles * S, tok_tiles);
    if (S == 1)
        return launch_pdl(fam.plain, grid, dim3(kThreads), fam.smem, st, 1, qmap, wmap, omap, amap, staged, tok_scale,
                          gamma, M, N, KT, RGN, out, acc_out, wait_limit);
    return launch_pdl(fam.split, grid, dim3(kThreads), fam.smem, st, static_cast<unsigned>(S), qmap, wmap, omap, amap,
                      staged, tok_scale, gamma, M, N, KT, RGN, out, acc_out, wait_limit);
}

// The persistent f16-operand GEMM: one CTA per SM over all tiles.
template <int BN, int NSTG, int NA>
cudaError_t launch_persistent(const void *q16, const float *tok_scale, const uint8_t *packed, const float *gamma,
                              int M, int N, int K, __nv_bfloat16 *out, cudaStream_t st, uint32_t wait_limit) {
    using L = SmemP<BN, NSTG, NA>;
    const int KT = (K + 127) / 128, RGN = (N + 15) / 16;
    const int row_tiles = (RGN + 7) / 8, tiles = row_tiles * ((M + BN - 1) / BN);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        static bool configured[64] = {false};
        std::lock_guard<std::mutex> lock(g_family_mutex);
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(gemm16p_kernel<BN, NSTG, NA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(L::kBytes));
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    CUtensorMap qmap, wmap, omap;
    e = make_qmap(&qmap, q16, M, K, BN, true);
    if (e == cudaSuccess) e = make_wmap(&wmap, packed, RGN, KT);
    if (e == cudaSuccess) e = make_omap(&omap, out, M, N, BN, false);
    if (e != cudaSuccess) return e;
    const int sms = device_sms(dev);
    const int grid = tiles < sms ? tiles : sms;
    return launch_pdl(gemm16p_kernel<BN, NSTG, NA>, dim3(grid), dim3(kThreadsP), L::kBytes, st, 1, qmap, wmap, omap,
                      tok_scale, gamma, M, N, KT, RGN, row_tiles, tiles, wait_limit);
}

// Whether the persistent kernel (token tile 192) runs.  Measured with f16
// operands on the 2B shapes (TFLOP/s, one tile per CTA -> persistent):
// 2560x2560 at 4096 tokens 1048 -> 1121, at 2048 790 -> 790; 2560x6912 at
// 4096 1296 -> 1245; 6912x2560 at 4096 1268 -> 1126 (192) / 926 (128).  It
// pays where the tiles are the one-tile plan's (token tile 192 there too)
// and the main loop is short against the epilogue it hides (K <= 4096);
// elsewhere the one-tile kernel's stage rate wins.
bool use_persistent(int M, int N, int K, int sms, int one_tile_bn) {
    if (one_tile_bn != 192 || K > 4096) return false;
    const int64_t tiles = static_cast<int64_t>((N + 127) / 128) * ((M + 191) / 192);
    return tiles > sms;
}

}  // namespace

// Token tile (MMA N) above 128 tokens, one CTA per SM holding a 128-row x
// BN tile: 256, or 192 where that takes fewer whole waves.  A 64-k stage
// costs about the same down to BN = 192 (its copies and weight conversion
// set a floor), so a narrower tile pays only where the wave count drops:
// e.g. N = 2560 (20 row tiles) at M = 4096 gives 320 tiles with BN = 256
// (2.2 waves, three paid) and 440 with BN = 192 (three full waves).
int token_tile(int M, int N) {
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) sms = device_sms(dev);
    const int64_t row_tiles = (N + 127) / 128;
    auto cost = [&](int bn) {  // whole waves x a per-tile time with a large fixed part
        const int64_t tiles = row_tiles * ((M + bn - 1) / bn);
        return (tiles + sms - 1) / sms * (bn + 64);
    };
    return cost(192) < cost(256) ? 192 : 256;
}

// `split`: CTAs per cluster along K, or 0 to let the planner choose.
cudaError_t launch_gemm16(const void *q16, const float *tok_scale, const uint8_t *packed, const float *gamma, int M,
                          int N, int K, __nv_bfloat16 *out, int32_t *acc_out, cudaStream_t st, uint32_t wait_limit,
                          int split) {
    // More tiles than SMs, bf16 rows of whole 16-byte units, no int32 copy
    // wanted, no forced split: the persistent kernel.
    if (!acc_out && (N % 8) == 0 && split <= 1 && M > 128) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
        if (use_persistent(M, N, K, device_sms(dev), token_tile(M, N)))
            return launch_persistent<192, 6, 4>(q16, tok_scale, packed, gamma, M, N, K, out, st, wait_limit);
    }
    if (M <= 64)
        return launch_family(family16<64, 10>(), 64, q16, true, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                             wait_limit, split);
    if (M <= 128)
        return launch_family(family16<128, 8>(), 128, q16, true, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                             wait_limit, split);
    if (token_tile(M, N) == 192)
        return launch_family(family16<192, 6>(), 192, q16, true, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                             wait_limit, split);
    return launch_family(family16<256, 6>(), 256, q16, true, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                         wait_limit, split);
}

namespace {

// int8 -> f16, exact (16 values per thread and step): q + 128 as the low
// mantissa byte of 1024 + u, minus 1152.
__global__ void __launch_bounds__(256) widen_kernel(const uint4 *__restrict__ q, int64_t n16,
                                                    uint4 *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();  // q comes from the previous kernel
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16; i += stride) {
        if (!dbg_ok(fits(i, 1, n16), 4)) continue;
        const uint4 v = q[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t x = w[j] ^ 0x80808080u;
            f[2 * j] = hadd2(prmt(x, 0x64646464u, 0x4140u), 0xE480E480u);
            f[2 * j + 1] = hadd2(prmt(x, 0x64646464u, 0x4342u), 0xE480E480u);
        }
        out[2 * i] = make_uint4(f[0], f[1], f[2], f[3]);
        out[2 * i + 1] = make_uint4(f[4], f[5], f[6], f[7]);
    }
}

// A memory pool per device for the widened activations, which keeps what it
// holds between calls (release threshold: never), so a call's stream-ordered
// allocation is a lookup.  Where it cannot be made (a first call inside a
// stream capture), the device's default pool serves instead.
std::mutex g_pool_mutex;
cudaMemPool_t g_pool[64] = {};
bool g_pool_tried[64] = {false};

cudaError_t widen_alloc(void **p, size_t bytes, cudaStream_t st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_pool_mutex);
        if (!g_pool_tried[dev]) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
                g_pool_tried[dev] = true;
                cudaMemPoolProps props = {};
                props.allocType = cudaMemAllocationTypePinned;
                props.location.type = cudaMemLocationTypeDevice;
                props.location.id = dev;
                if (cudaMemPoolCreate(&g_pool[dev], &props) == cudaSuccess) {
                    uint64_t keep = ~0ull;
                    cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep);
                } else {
                    g_pool[dev] = nullptr;
                    cudaGetLastError();
                }
            }
        }
        pool = g_pool[dev];
    }
    return pool ? cudaMallocFromPoolAsync(p, bytes, pool, st) : cudaMallocAsync(p, bytes, st);
}

}  // namespace

// Stream-ordered scratch memory for the other engines (the fused decode
// path's quantised input).
cudaError_t scratch_alloc(void **p, size_t bytes, cudaStream_t st) { return widen_alloc(p, bytes, st); }

// bitlinear_forward widens the int8 activations to f16 once (one pass over
// M x K) and runs the f16-operand GEMM above 256 tokens, and above 32 for
// matrices of at least 2^24 weights (at 49-64 tokens the f16-operand GEMM
// takes 84 against 104 us on 28672x8192, 72 against 94 on 8192x28672; at
// 33-48 tokens, with the widening pass, 81 against 99 and 68 against 90): in
// the int8 engine every row-tile CTA
// converts the same activation tile again (20-224 times for the 2B-70B
// shapes), which held it at 0.43 of the bf16 peak against 0.67 for f16
// operands at 4096 tokens, and cost 30-55 % at 65-256 tokens on the 2B
// gate/up and down matrices (measured; the 2560x2560 ones gain nothing
// there, the extra launch eats the saving).
bool widen_first(int M, int N, int K) {
    return M > 256 || (M > 32 && static_cast<int64_t>(N) * K >= (1ll << 24));
}

cudaError_t launch_gemm(const int8_t *q, const float *tok_scale, const uint8_t *packed, const float *gamma, int M,
                        int N, int K, __nv_bfloat16 *out, int32_t *acc_out, cudaStream_t st, uint32_t wait_limit,
                        int split) {
    if (widen_first(M, N, K)) {
        const size_t bytes = static_cast<size_t>(M) * K * 2;
        void *q16 = nullptr;
        cudaError_t e = widen_alloc(&q16, bytes, st);
        if (e != cudaSuccess) {
            cudaGetLastError();  // a failed allocation is the call's error, not the caller's next one
            return e;
        }
        const int64_t n16 = static_cast<int64_t>(M) * K / 16;  // K % 16 == 0
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
        int64_t blocks = (n16 + 255) / 256;
        const int64_t cap = static_cast<int64_t>(device_sms(dev)) * 8;
        if (blocks > cap) blocks = cap;
        e = launch_pdl(widen_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1,
                       reinterpret_cast<const uint4 *>(q), n16, static_cast<uint4 *>(q16));
        if (e == cudaSuccess)
            e = launch_gemm16(q16, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit, split);
        const cudaError_t ef = cudaFreeAsync(q16, st);
        return e != cudaSuccess ? e : ef;
    }
    if (M <= 64)
        return launch_family(family8<64>(), 64, q, false, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                             wait_limit, split);
    if (M <= 128)
        return launch_family(family8<128>(), 128, q, false, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                             wait_limit, split);
    if (token_tile(M, N) == 192)
        return launch_family(family8<192>(), 192, q, false, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                             wait_limit, split);
    return launch_family(family8<256>(), 256, q, false, tok_scale, packed, gamma, M, N, K, out, acc_out, st,
                         wait_limit, split);
}

// Device address of the status word, for kernels in other translation units.
cudaError_t status_word(unsigned int **dev_ptr) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_gemm_status);
    if (e != cudaSuccess) return e;
    *dev_ptr = static_cast<unsigned int *>(p);
    return cudaSuccess;
}

cudaError_t gemm_status(unsigned int *out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_gemm_status, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0u;
    e = cudaMemcpyToSymbolAsync(g_gemm_status, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(st);
}

}  // namespace bl
